"""GB300 (sm_103a) latent mixture-of-experts block of Muse Spark Open.

    out = x + RMSNorm_post( F( RMSNorm_pre(x) ) )

F routes on the full-width normalised input (softmax over all experts, top-k,
renormalised weights), pools 8192 -> 4096 and normalises, runs the selected
SwiGLU experts, RMS-normalises each expert output with its own gamma before the
routing weight multiplies it, sums in FP32, and unpools 4096 -> 8192 (LMSYS
"SGLang and Miles Add Day-0 Support for Muse Spark Open", section "MoE with
pooler, unpooler and per-expert normalization"; vLLM "Day 0 support for Muse
Spark Open", sections "Sandwich normalization" and "Latent MoE").

The computation runs in the hand-written CUDA kernels of ``liblatent_moe.so``
behind the C ABI of ``include/latent_moe.h``; this package only marshals
arguments.  Importing it fails if the library has not been built.
"""
from __future__ import annotations

import torch

from ._lib import (Config, LmoeError, lmoe_workspace_size, lmoe_workspace_size_host_io,  # noqa: F401
                   lmoe_get_workspace_layout, latent_moe_forward, latent_moe_forward_ex,
                   latent_moe_forward_host_io, latent_moe_forward_host_io_ex, lmoe_check_status,
                   lmoe_wait_selftest, lmoe_expert_pair, load,
                   LIB_PATH, STAGES, NUM_STAGE_EVENTS, lmoe_kernel_launches, SINGLE_TOKEN_DEFAULT,
                   SINGLE_TOKEN_KERNEL, SINGLE_TOKEN_CHAIN,
                   lmoe_quantize_nvfp4, lmoe_nvfp4_block_scales, SCALES_ROW_MAJOR, SCALES_BLOCKED,
                   GUARD_BYTES, lmoe_workspace_guards, lmoe_validate_routing)

load()


class LatentMoEBlock:
    """Device-resident weights of one block plus a reusable workspace.

    Weights: W_router [E, D]; W_pool [L, D]; W_gate, W_up [E, I, L]; W_down [E, L, I];
    W_unpool [D, L]; gammas g_pre [D], g_pool [L], g_expert [E, L], g_post [D] (fp32).
    NVFP4 weights are (codes, row-major E4M3 scales, tensor scale) triples; their scales are
    converted once into the block layout the kernels read.
    """

    def __init__(self, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert, W_unpool, g_pre,
                 g_post, top_k: int, eps: float = 1e-6, weight_dtype: str = "bf16"):
        if weight_dtype == "nvfp4":   # (codes, row-major scales, s) -> scales in block layout
            def blocked(w, block_rows=128):
                codes, scales, s = w[:3]
                return codes, lmoe_nvfp4_block_scales(scales, codes.shape[-1] * 2, block_rows), s, SCALES_BLOCKED
            W_pool, W_gate, W_up, W_down, W_unpool = map(blocked, (W_pool, W_gate, W_up, W_down, W_unpool))
        self.W = dict(W_router=W_router, W_pool=W_pool, g_pool=g_pool, W_gate=W_gate, W_up=W_up,
                      W_down=W_down, g_expert=g_expert, W_unpool=W_unpool, g_pre=g_pre, g_post=g_post)
        self.top_k, self.eps, self.weight_dtype = top_k, eps, weight_dtype
        self.E, self.D = W_router.shape
        self.L = g_pool.shape[0]
        self.I = (W_gate[0] if isinstance(W_gate, tuple) else W_gate).shape[1]
        self._ws = None

    def config(self, T: int, act_dtype="bf16", out_dtype="f32") -> Config:
        return Config(T, self.D, self.L, self.E, self.I, self.top_k, self.eps, act_dtype,
                      self.weight_dtype, out_dtype)

    def workspace(self, cfg: Config, host_io: bool = False) -> torch.Tensor:
        n = lmoe_workspace_size_host_io(cfg) if host_io else lmoe_workspace_size(cfg)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=self.W["g_pre"].device)
        return self._ws

    def forward(self, x: torch.Tensor, out_dtype="f32", out=None, stream=None, **ex) -> torch.Tensor:
        act = "f32" if x.dtype == torch.float32 else "bf16"
        cfg = self.config(x.shape[0], act, out_dtype)
        if out is None:
            out = torch.empty(x.shape, dtype=torch.float32 if out_dtype == "f32" else torch.bfloat16,
                              device=x.device)
        ws = self.workspace(cfg)
        w = self.W
        fn = latent_moe_forward_ex if ex else latent_moe_forward
        fn(cfg, x, w["W_router"], w["W_pool"], w["g_pool"], w["W_gate"], w["W_up"], w["W_down"],
           w["g_expert"], w["W_unpool"], w["g_pre"], w["g_post"], self.top_k, out, ws, stream, **ex)
        return out
