"""Helpers for the GPU tests: run the block through the C ABI and read the intermediates
back out of the workspace (offsets from lmoe_get_workspace_layout)."""
from __future__ import annotations

import numpy as np
import torch

import workloads


def lib():
    import latent_mixture_experts_router_gb300 as lm
    return lm


def make_block(inp: workloads.BlockInputs):
    lm = lib()
    w = inp.w
    return lm.LatentMoEBlock(inp.W_router, inp.W_pool, inp.g_pool, inp.W_gate, inp.W_up, inp.W_down,
                             inp.g_expert, inp.W_unpool, inp.g_pre, inp.g_post, w.k, w.eps,
                             weight_dtype=w.weights)


def run(inp: workloads.BlockInputs, out_dtype="f32", blk=None, x=None, **ex):
    """One forward; returns (out, topk idx, block, config)."""
    lm = lib()
    blk = blk or make_block(inp)
    x = inp.x if x is None else x
    T, k = x.shape[0], inp.w.k
    idx = torch.full((T, k), -1, dtype=torch.int32, device=x.device)
    kw = dict(topk_idx_out=idx)
    if inp.router_bias is not None:
        kw["router_bias"] = inp.router_bias
    if inp.forced_idx is not None and x is inp.x:
        kw["forced_idx"] = inp.forced_idx
    kw.update(ex)
    out = blk.forward(x, out_dtype=out_dtype, **kw)
    torch.cuda.synchronize()
    cfg = blk.config(T, "f32" if x.dtype == torch.float32 else "bf16", out_dtype)
    st, word = lm.lmoe_check_status(cfg, blk._ws)
    assert st == 0, f"device status {st} word {word:#x}"
    return out, idx, blk, cfg


def views(blk, cfg) -> dict:
    """numpy copies of the workspace intermediates."""
    lm = lib()
    lay = lm.lmoe_get_workspace_layout(cfg)
    ws = blk._ws
    T, D, L, E, I, k = cfg.T, cfg.d_model, cfg.d_latent, cfg.n_experts, cfg.d_ff, cfg.top_k
    R = T * k
    ld_logits = (E + 31) // 32 * 32

    def get(name, n, dtype):
        o = lay[name]
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        return ws[o:o + nbytes].view(dtype)

    bf = torch.bfloat16
    v = {
        "xa": get("xa", T * lay["xa_cols"], bf).view(T, lay["xa_cols"]),
        "logits": get("logits", T * ld_logits, torch.float32).view(T, ld_logits)[:, :E],
        "topk_idx": get("topk_idx", R, torch.int32).view(T, k),
        "topk_w": get("topk_w", R, torch.float32).view(T, k),
        "counts": get("counts", E, torch.int32),
        "offsets": get("offsets", E + 1, torch.int32),
        "row_of": get("row_of", R, torch.int32).view(T, k),
        "tok_of": get("tok_of", R, torch.int32),
        "n_tiles": get("n_tiles", 1, torch.int32),
        "p": get("p", T * L, torch.float32).view(T, L),
        "xe": get("xe", R * L, bf).view(R, L) if cfg.weight_dtype != "nvfp4" else None,
        "h": get("h", R * I, bf).view(R, I) if cfg.weight_dtype != "nvfp4" else None,
        "y": get("y", R * L, bf if cfg.weight_dtype == "nvfp4" else torch.float32).view(R, L),
        "c": get("c", T * L, bf).view(T, L) if cfg.weight_dtype != "nvfp4" else None,
        "u": get("u", T * D, torch.float32).view(T, D),
    }
    if cfg.weight_dtype == "nvfp4":   # xe, h, c hold packed codes there (see the layout)
        for name in ("xe", "h", "c"):
            v.pop(name)
    return {name: t.to(torch.float64 if t.dtype in (bf, torch.float32) else torch.int64).cpu().numpy()
            for name, t in v.items()}


def expected_permutation(idx: np.ndarray, E: int):
    """Stable expert-major order of the (token, slot) pairs, from numpy's stable sort."""
    flat = idx.reshape(-1).astype(np.int64)
    order = np.argsort(flat, kind="stable")          # pair ids in expert-contiguous order
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    row_of = np.empty_like(flat)
    row_of[order] = np.arange(flat.size)
    k = idx.shape[1]
    tok_of = order // k
    return counts, offsets, row_of.reshape(idx.shape), tok_of


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.sqrt(np.mean(b * b)), 1e-30))
