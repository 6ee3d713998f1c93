"""Parity comparison of a GPU block result with the oracle (test infrastructure).

Rules (the tolerances the block is graded on):
  * top-k indices must match exactly, in order, except where the oracle's own fp64
    logits leave the choice open: a token whose k-th and (k+1)-th largest logits
    differ by less than 1e-3 ("near tie") may pick a different set, and two selected
    experts whose logits differ by less than 1e-3 may come in either order.  Such
    tokens are counted and reported; for them the expected output is the oracle
    re-run with the GPU's selection (same math, another legitimate selection).
  * max |out - ref| <= tol * RMS(ref), tol = 2e-2 for BF16 compute, 6e-2 for NVFP4.
  * NVFP4: the activation rule rounds in fp32, and both sides feed it values computed in
    different orders.  Where the oracle's exact value of a quantised activation lies within
    formats.QUANT_BAND (relative) of a rounding boundary, either rounding is a legitimate
    result of the rule.  A token outside the bar is accepted when its output is within the
    bar of the oracle's output with one such decision taken the other way
    (block.forward_token_choices); such tokens are counted and reported.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .block import BlockParams, Trace, forward_batched, forward_per_token, forward_token_choices

TOL_BF16 = 2e-2
TOL_NVFP4 = 6e-2
TIE_BAND = 1e-3


@dataclass
class Report:
    tokens: int
    idx_exact: int
    near_tie_tokens: int
    order_swaps: int
    bad_idx_tokens: list
    max_abs_err: float
    ref_rms: float
    tol: float
    quant_boundary_tokens: int = 0

    @property
    def ok(self) -> bool:
        return not self.bad_idx_tokens and self.max_abs_err <= self.tol * self.ref_rms

    def __str__(self):
        return (f"tokens={self.tokens} idx_exact={self.idx_exact} near_tie={self.near_tie_tokens} "
                f"order_swaps={self.order_swaps} quant_boundary={self.quant_boundary_tokens} "
                f"bad_idx={self.bad_idx_tokens[:8]} "
                f"max|err|={self.max_abs_err:.4e} tol*RMS={self.tol * self.ref_rms:.4e} ok={self.ok}")


def classify_topk(gpu_idx: np.ndarray, tr: Trace, k: int):
    """Split tokens into exact / near-tie (set may differ) / order-swap / bad."""
    gpu_idx = np.asarray(gpu_idx, dtype=np.int64)
    exact = np.all(gpu_idx == tr.idx, axis=1)
    near, swaps, bad = [], [], []
    for t in np.nonzero(~exact)[0]:
        if tr.near_tie[t]:
            near.append(int(t))
            continue
        same_set = set(gpu_idx[t].tolist()) == set(tr.idx[t].tolist())
        if same_set:
            lg = tr.logits[t]
            # every displaced position must hold a logit within the band of the oracle's one
            if np.all(np.abs(lg[gpu_idx[t]] - lg[tr.idx[t]]) < TIE_BAND):
                swaps.append(int(t))
                continue
        bad.append(int(t))
    return exact, near, swaps, bad


def compare_block(gpu_out: np.ndarray, gpu_idx: np.ndarray, x: np.ndarray, P: BlockParams, k: int,
                  tol: float, tr: Trace | None = None, ref: np.ndarray | None = None,
                  forced_idx: np.ndarray | None = None, choices=forward_token_choices) -> Report:
    """Compare a GPU run on rows x with the oracle (batched) under the rules above.
    ``choices`` (NVFP4 only) gives a token's legitimate outputs at near-boundary roundings."""
    x = np.asarray(x, dtype=np.float64)
    gpu_out = np.asarray(gpu_out, dtype=np.float64)
    if tr is None or ref is None:
        tr = Trace()
        ref = forward_batched(x, P, k, forced_idx=forced_idx, trace=tr)
    exact, near, swaps, bad = classify_topk(gpu_idx, tr, k)
    ref = ref.copy()
    for t in near + swaps:   # expected output under the GPU's own (legitimate) selection
        ref[t] = forward_per_token(x[t:t + 1], P, k, forced_idx=np.asarray(gpu_idx)[t:t + 1])[0]
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    boundary = 0
    if P.nvfp4 and ref.size:
        tok_err = np.max(np.abs(gpu_out - ref), axis=1)
        for t in np.nonzero(tok_err > tol * rms)[0]:
            if t in bad:
                continue
            sel = np.asarray(gpu_idx)[t] if (t in near or t in swaps) else \
                (None if forced_idx is None else np.asarray(forced_idx)[t])
            outs = choices(x[t], P, k, sel)
            errs = [float(np.max(np.abs(gpu_out[t] - o))) for o in outs[1:]]
            if errs and min(errs) <= tol * rms:
                ref[t] = outs[1 + int(np.argmin(errs))]
                boundary += 1
    err = np.abs(gpu_out - ref)
    return Report(tokens=x.shape[0], idx_exact=int(exact.sum()), near_tie_tokens=len(near),
                  order_swaps=len(swaps), bad_idx_tokens=bad, max_abs_err=float(err.max()) if err.size else 0.0,
                  ref_rms=rms, tol=tol, quant_boundary_tokens=boundary)
