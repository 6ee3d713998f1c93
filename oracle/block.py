"""Plain fp64 CPU oracle of the Muse Spark Open latent-MoE block.

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU baseline.  It shares no code with the CUDA library and never
imports it; the library never imports this.

What the block computes (per token; the block is token-independent):

  xn  = RMSNorm(x; g_pre)                        sandwich norm, first slice
                                                 (vLLM day-0 post, "Sandwich normalization")
  l   = W_router xn  (+ optional per-expert bias)  router on the FULL-width xn
  P   = softmax(l) over all E experts; S = the k largest logits (ties -> lower
        index); w_j = P[S_j] / sum_{S} P          top-k routing weights
  h0  = RMSNorm(W_pool xn; g_pool)               pooler 8192->4096, pooled input
                                                 normalised before the experts
  z_e = RMSNorm(W_down[e] (silu(W_gate[e] h0) * (W_up[e] h0)); g_expert[e])
                                                 SwiGLU expert, its output RMS-normalised
                                                 BEFORE the routing weight is applied
  c   = sum_j w_j z_{S_j}                        weighted sum (fp32 in the model)
  out = x + RMSNorm(W_unpool c; g_post)          unpooler 4096->8192, post-norm, residual

Sources: LMSYS "SGLang and Miles Add Day-0 Support for Muse Spark Open",
sections "MoE with pooler, unpooler and per-expert normalization" (router on
the full-width input, pooled input normalised before the experts, each
expert output normalised before weighting, then unpool) and "Fused per-expert
post-norm"; "Reinforcement learning" (weighted sum in FP32); vLLM "Day 0
support for Muse Spark Open", sections "Sandwich normalization" and "Latent
MoE" (x + post_norm(F(norm(x))); pooler 8192x4096, unpooler back to 8192).

Readings where the pages are silent (each listed in the design notes):
RMSNorm(v; g) = v / sqrt(mean(v^2) + eps) * g with g stored as is (not 1+g),
eps = 1e-6 inside the square root for all four norms; no gate on the residual;
no shared expert; softmax-over-all then top-k renormalised, lower index on
ties; the slot order is descending logit and the sum runs in slot order.

NVFP4 mode: each GEMM input activation (xn into the pooler, h0 into gate/up,
h into down, c into the unpooler) is replaced by its fake-quantised value
under the activation rule of ``oracle.formats`` (row scale for xn, h0, c;
scale 1 for h); weights are the dequantised packed weights; each expert output
y is rounded to bfloat16 before its norm (the BF16 values the pages' fused
per-expert post-norm squares); the router stays at full precision on xn.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, Optional

import numpy as np

from . import formats

F64 = np.float64


# ------------------------------------------------------------------ primitives
def rms_norm(v: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: v / sqrt(mean(v^2) + eps) * g."""
    v = np.asarray(v, dtype=F64)
    ms = np.mean(v * v, axis=-1, keepdims=True)
    return v / np.sqrt(ms + eps) * np.asarray(g, dtype=F64)


def silu(a: np.ndarray) -> np.ndarray:
    return a / (1.0 + np.exp(-a))


def softmax(l: np.ndarray) -> np.ndarray:
    m = np.max(l, axis=-1, keepdims=True)
    ex = np.exp(l - m)
    return ex / np.sum(ex, axis=-1, keepdims=True)


def top_k(l: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries of each row, largest first; equal values
    are taken in ascending index order (stable sort of -l)."""
    order = np.argsort(-np.asarray(l, dtype=F64), axis=-1, kind="stable")
    return order[..., :k]


def route(logits: np.ndarray, k: int, forced_idx: Optional[np.ndarray] = None):
    """Full softmax over all experts, top-k selection, renormalised weights.

    Returns (idx [T,k] int64, w [T,k] fp64, near_tie [T] bool).  ``forced_idx``
    fixes the selection (weights stay the renormalised softmax at those ids).
    near_tie marks tokens whose k-th and (k+1)-th largest logits differ by < 1e-3.
    """
    logits = np.asarray(logits, dtype=F64)
    P = softmax(logits)
    idx = top_k(logits, k) if forced_idx is None else np.asarray(forced_idx, dtype=np.int64)
    Ps = np.take_along_axis(P, idx, axis=-1)
    w = Ps / np.sum(Ps, axis=-1, keepdims=True)
    E = logits.shape[-1]
    if k < E:
        srt = -np.sort(-logits, axis=-1)
        near_tie = (srt[:, k - 1] - srt[:, k]) < 1e-3
    else:
        near_tie = np.zeros(logits.shape[0], dtype=bool)
    return idx, w, near_tie


# ------------------------------------------------------------------ parameters
class ExpertStack:
    """Per-expert weight access: ``stack[e]`` -> fp64 [rows, cols].  Wraps either a
    dense [E, rows, cols] array or a callable producing one expert on demand
    (full-size expert stacks are 25.8 GB in bf16 and are never expanded whole)."""

    def __init__(self, src, n_experts: int):
        self._src = src
        self.n = n_experts
        self._cache = {}

    def __getitem__(self, e: int) -> np.ndarray:
        e = int(e)
        if callable(self._src):
            if e not in self._cache:
                self._cache = {e: np.asarray(self._src(e), dtype=F64)}  # keep one expert
            return self._cache[e]
        return np.asarray(self._src[e], dtype=F64)


@dataclass
class BlockParams:
    W_router: np.ndarray      # [E, D]
    W_pool: np.ndarray        # [L, D]
    g_pool: np.ndarray        # [L]
    W_gate: ExpertStack       # [E][I, L]
    W_up: ExpertStack         # [E][I, L]
    W_down: ExpertStack       # [E][L, I]
    g_expert: np.ndarray      # [E, L]
    W_unpool: np.ndarray      # [D, L]
    g_pre: np.ndarray         # [D]
    g_post: np.ndarray        # [D]
    eps: float = 1e-6
    router_bias: Optional[np.ndarray] = None   # [E]
    nvfp4: bool = False       # activations fake-quantised at the four GEMM inputs

    @property
    def E(self):
        return self.W_router.shape[0]


@dataclass
class Trace:
    """Intermediates of one forward, for stage-by-stage comparison."""
    xn: np.ndarray = None
    logits: np.ndarray = None
    idx: np.ndarray = None
    w: np.ndarray = None
    near_tie: np.ndarray = None
    p: np.ndarray = None
    h0: np.ndarray = None
    y: dict = field(default_factory=dict)    # (t, j) -> y before its norm
    z: dict = field(default_factory=dict)    # (t, j) -> normalised expert output
    c: np.ndarray = None
    u: np.ndarray = None


def _q(v: np.ndarray, nvfp4: bool, row_scale: bool = True) -> np.ndarray:
    return formats.fake_quantize_activation(v, row_scale) if nvfp4 else v


def expert_ffn(P: BlockParams, e: int, h0: np.ndarray) -> np.ndarray:
    """SwiGLU expert e on rows h0 [n, L] -> y [n, L] (before the per-expert norm).  In NVFP4
    mode y is rounded to bfloat16: the down projection's tiles hold y as BF16 values and the
    per-expert norm squares those values (LMSYS Muse Spark Open post, "Fused per-expert
    post-norm"), and c is quantised again after the weighted sum, so the rounding of y decides
    E2M1 codes downstream."""
    a_in = _q(h0, P.nvfp4)
    a = a_in @ P.W_gate[e].T
    b = a_in @ P.W_up[e].T
    h = silu(a) * b
    y = _q(h, P.nvfp4, row_scale=False) @ P.W_down[e].T
    return formats.bf16_round(y) if P.nvfp4 else y


# ------------------------------------------------------------------ forward
def forward_per_token(x: np.ndarray, P: BlockParams, k: int,
                      forced_idx: Optional[np.ndarray] = None, trace: Optional[Trace] = None):
    """The definition, one token at a time (slow; tiny shapes and sampled tokens)."""
    x = np.asarray(x, dtype=F64)
    T = x.shape[0]
    out = np.empty_like(x)
    tr = trace if trace is not None else Trace()
    tr.xn, tr.logits, tr.p, tr.h0 = [], [], [], []
    tr.idx, tr.w, tr.near_tie, tr.c, tr.u = [], [], [], [], []
    for t in range(T):
        xn = rms_norm(x[t], P.g_pre, P.eps)
        l = P.W_router @ xn
        if P.router_bias is not None:
            l = l + P.router_bias
        fi = None if forced_idx is None else np.asarray(forced_idx)[t:t + 1]
        idx, w, nt = route(l[None, :], k, fi)
        idx, w = idx[0], w[0]
        p = _q(xn[None, :], P.nvfp4)[0] @ P.W_pool.T
        h0 = rms_norm(p, P.g_pool, P.eps)
        c = np.zeros_like(h0)
        for j in range(k):
            e = int(idx[j])
            y = expert_ffn(P, e, h0[None, :])[0]
            z = rms_norm(y, P.g_expert[e], P.eps)
            tr.y[(t, j)], tr.z[(t, j)] = y, z
            c = c + w[j] * z
        u = _q(c[None, :], P.nvfp4)[0] @ P.W_unpool.T
        out[t] = x[t] + rms_norm(u, P.g_post, P.eps)
        for name, v in (("xn", xn), ("logits", l), ("p", p), ("h0", h0), ("idx", idx), ("w", w),
                        ("near_tie", nt[0]), ("c", c), ("u", u)):
            getattr(tr, name).append(v)
    for name in ("xn", "logits", "p", "h0", "idx", "w", "near_tie", "c", "u"):
        setattr(tr, name, np.array(getattr(tr, name)))
    return out


def forward_batched(x: np.ndarray, P: BlockParams, k: int,
                    forced_idx: Optional[np.ndarray] = None, trace: Optional[Trace] = None,
                    progress: Optional[Callable[[int], None]] = None):
    """Same definition, with the rows routed to each expert gathered into one matrix
    product per expert (each expert's weights are touched once)."""
    x = np.asarray(x, dtype=F64)
    T = x.shape[0]
    xn = rms_norm(x, P.g_pre, P.eps)
    logits = xn @ P.W_router.T
    if P.router_bias is not None:
        logits = logits + P.router_bias[None, :]
    idx, w, near_tie = route(logits, k, forced_idx)
    p = _q(xn, P.nvfp4) @ P.W_pool.T
    h0 = rms_norm(p, P.g_pool, P.eps)
    z = np.zeros((T, k, h0.shape[1]), dtype=F64)
    keep_y = trace is not None
    ys = {}
    for e in np.unique(idx):
        t_sel, j_sel = np.nonzero(idx == e)
        y = expert_ffn(P, int(e), h0[t_sel])
        z[t_sel, j_sel] = rms_norm(y, P.g_expert[int(e)], P.eps)
        if keep_y:
            for r, (t, j) in enumerate(zip(t_sel, j_sel)):
                ys[(int(t), int(j))] = y[r]
        if progress:
            progress(int(e))
    c = np.zeros_like(h0)
    for j in range(k):                       # slot order, as the weighted sum is defined
        c = c + w[:, j:j + 1] * z[:, j]
    u = _q(c, P.nvfp4) @ P.W_unpool.T
    out = x + rms_norm(u, P.g_post, P.eps)
    if trace is not None:
        trace.xn, trace.logits, trace.idx, trace.w, trace.near_tie = xn, logits, idx, w, near_tie
        trace.p, trace.h0, trace.c, trace.u, trace.y = p, h0, c, u, ys
        trace.z = {(t, j): z[t, j] for (t, j) in ys}
    return out


def forward_norm_after_sum(x: np.ndarray, P: BlockParams, k: int):
    """The variant the pages warn against: normalise the merged expert output
    instead of each expert output (one RMSNorm with the mean of the selected
    experts' gammas).  Used only to show that it computes something else."""
    x = np.asarray(x, dtype=F64)
    xn = rms_norm(x, P.g_pre, P.eps)
    l = xn @ P.W_router.T
    idx, w, _ = route(l, k)
    h0 = rms_norm(xn @ P.W_pool.T, P.g_pool, P.eps)
    out = np.empty_like(x)
    for t in range(x.shape[0]):
        s = sum(w[t, j] * expert_ffn(P, int(idx[t, j]), h0[t:t + 1])[0] for j in range(k))
        g = np.mean([P.g_expert[int(e)] for e in idx[t]], axis=0)
        c = rms_norm(s, g, P.eps)
        out[t] = x[t] + rms_norm(P.W_unpool @ c, P.g_post, P.eps)
    return out


def forward_token_choices(x_t: np.ndarray, P: BlockParams, k: int, forced_row: Optional[np.ndarray] = None,
                          band: float = formats.QUANT_BAND):
    """NVFP4 mode: the outputs one token may legitimately have when a rounding decision of the
    activation rule is undecided (formats.activation_choices: the exact value within `band` of
    a rounding boundary).  The first entry is the rule's own output (forward_per_token); each
    further entry takes one near-boundary decision of one quantised activation (xn into the
    pooler, h0 into gate/up, the h row of one routed expert into down, c into the unpooler)
    the other way, everything else as the rule decides."""
    assert P.nvfp4
    x_t = np.asarray(x_t, dtype=F64).reshape(-1)
    xn = rms_norm(x_t, P.g_pre, P.eps)
    l = P.W_router @ xn
    if P.router_bias is not None:
        l = l + P.router_bias
    fr = None if forced_row is None else np.asarray(forced_row).reshape(1, -1)
    idx, w, _ = route(l[None, :], k, fr)
    idx, w = idx[0], w[0]

    def quant(v, row_scale=True):
        return formats.activation_choices(v, row_scale, band)

    def expert_h(e, h0q):
        a = h0q @ P.W_gate[int(e)].T
        b = h0q @ P.W_up[int(e)].T
        return silu(a) * b

    def y_of(e, hq):
        return formats.bf16_round(hq @ P.W_down[int(e)].T)

    def c_of(ys):
        c = np.zeros(P.g_pool.shape[0], dtype=F64)
        for j in range(k):
            c = c + w[j] * rms_norm(ys[j], P.g_expert[int(idx[j])], P.eps)
        return c

    def out_of(cq):
        return x_t + rms_norm(cq @ P.W_unpool.T, P.g_post, P.eps)

    def from_ys(ys):
        return out_of(quant(c_of(ys))[0])

    def from_h0q(h0q):
        return from_ys([y_of(idx[j], quant(expert_h(idx[j], h0q), False)[0]) for j in range(k)])

    def from_xnq(xnq):
        return from_h0q(quant(rms_norm(xnq @ P.W_pool.T, P.g_pool, P.eps))[0])

    xn_ch = quant(xn)
    h0_ch = quant(rms_norm(xn_ch[0] @ P.W_pool.T, P.g_pool, P.eps))
    hs = [expert_h(idx[j], h0_ch[0]) for j in range(k)]
    h_ch = [quant(h, False) for h in hs]
    ys = [y_of(idx[j], h_ch[j][0]) for j in range(k)]
    c_ch = quant(c_of(ys))
    outs = [out_of(c_ch[0])]
    outs += [out_of(cq) for cq in c_ch[1:]]
    for j in range(k):
        for hq in h_ch[j][1:]:
            outs.append(from_ys(ys[:j] + [y_of(idx[j], hq)] + ys[j + 1:]))
    outs += [from_h0q(h0q) for h0q in h0_ch[1:]]
    outs += [from_xnq(xnq) for xnq in xn_ch[1:]]
    return outs
