"""Build oracle parameters (fp64 numpy) from the seeded workload tensors.

TEST INFRASTRUCTURE ONLY.  Dense bf16/fp32 tensors widen exactly to fp64;
packed NVFP4 weights are dequantised by ``oracle.formats``.  For full-size
workloads the expert stacks are regenerated on the host one expert at a time.
"""
from __future__ import annotations

import numpy as np
import torch

import workloads
from .block import BlockParams, ExpertStack
from . import formats


def _np(t: torch.Tensor) -> np.ndarray:
    # widening bf16/fp32 -> fp64 is exact, so it may run where the tensor lives (a device-side
    # widening of a 100 MB expert matrix is much faster than the host's)
    return t.detach().to(torch.float64).to("cpu").numpy()


def _host_u8(t) -> np.ndarray:
    return t.detach().to("cpu").numpy()


def _dense_or_nvfp4(v, per_expert: bool):
    """Tensor, or (codes, scales, s) triple -> fp64 array, or for expert stacks a callable
    that widens one expert on demand (stacks may be tensors or dicts keyed by expert)."""
    if isinstance(v, tuple):
        codes, scales, s = v
        if per_expert:
            return lambda e: formats.nvfp4_dequantize(_host_u8(codes[e]), _host_u8(scales[e]), float(s[e]))
        return formats.nvfp4_dequantize(_host_u8(codes), _host_u8(scales), float(s[0]))
    if per_expert:
        return lambda e: _np(v[e])
    return _np(v)


def params_from_inputs(inp: "workloads.BlockInputs") -> BlockParams:
    """Oracle parameters holding the same values as ``inp`` (any device)."""
    w = inp.w
    return BlockParams(
        W_router=_np(inp.W_router),
        W_pool=_dense_or_nvfp4(inp.W_pool, False),
        g_pool=_np(inp.g_pool),
        W_gate=ExpertStack(_dense_or_nvfp4(inp.W_gate, True), w.E),
        W_up=ExpertStack(_dense_or_nvfp4(inp.W_up, True), w.E),
        W_down=ExpertStack(_dense_or_nvfp4(inp.W_down, True), w.E),
        g_expert=_np(inp.g_expert),
        W_unpool=_dense_or_nvfp4(inp.W_unpool, False),
        g_pre=_np(inp.g_pre), g_post=_np(inp.g_post), eps=w.eps,
        router_bias=None if inp.router_bias is None else _np(inp.router_bias),
        nvfp4=(w.weights == "nvfp4"),
    )


def params_for_workload(w: "workloads.Workload") -> BlockParams:
    """Oracle parameters for workload ``w`` generated on the host; expert weights are
    produced one expert at a time on first use."""
    nv = w.weights == "nvfp4"

    def dense(name):
        if nv:
            c, s, g = workloads.nvfp4_weight(w, name)
            return formats.nvfp4_dequantize(c.numpy(), s.numpy(), float(g[0]))
        return _np(workloads.dense_weight(w, name))

    def expert(name):
        def get(e):
            if nv:
                c, s, g = workloads.nvfp4_weight(w, name, expert=e)
                return formats.nvfp4_dequantize(c.numpy(), s.numpy(), float(g[0]))
            return _np(workloads.dense_weight(w, name, expert=e))
        return ExpertStack(get, w.E)

    g = workloads.gammas(w)
    return BlockParams(
        W_router=_np(workloads.dense_weight(w, "W_router")),
        W_pool=dense("W_pool"), g_pool=_np(g["g_pool"]),
        W_gate=expert("W_gate"), W_up=expert("W_up"), W_down=expert("W_down"),
        g_expert=_np(g["g_expert"]), W_unpool=dense("W_unpool"),
        g_pre=_np(g["g_pre"]), g_post=_np(g["g_post"]), eps=w.eps,
        router_bias=None if w.routing != "zipf" else _np(workloads.zipf_bias(w)),
        nvfp4=nv,
    )
