"""Parity at the full Muse shapes (D 8192, L 4096, E 256, I 4096, k 8), in the launch
configuration the benchmark times.

Every token: top-k ids exact against the oracle's fp64 router (near ties and in-band order
swaps counted and printed), and the permutation bit-exact.  At least 64 sampled tokens per
workload (every token below 64): the block output against the oracle, and the stages p
(pooler), y (each routed expert's down projection, before its norm), c (combine, BF16 path)
and u (unpooler) of those tokens against the oracle's own intermediates.  The block is
token-independent, so a token's expected values need only its own row and the weights of the
experts it routes to.  Samples: tokens spread over the batch, every near-tie or swapped token,
tokens routed to the most loaded expert, and tokens routed to experts that fill a single
M tile (the "light" tiles of skewed routing)."""
import gc
import time

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle.compare import TOL_BF16, TOL_NVFP4, classify_topk, compare_block

from gpu_util import expected_permutation, run

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N_SAMPLE = 64


@pytest.fixture(scope="module", autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    yield torch.device("cuda:0")
    gc.collect()
    torch.cuda.empty_cache()


def _full_router(inp, P):
    x = inp.x.double().cpu().numpy()
    xn = oracle.rms_norm(x, P.g_pre, P.eps)
    lg = xn @ P.W_router.T
    if P.router_bias is not None:
        lg = lg + P.router_bias
    idx, w, nt = oracle.route(lg, inp.w.k)
    return x, oracle.Trace(idx=idx, w=w, near_tie=nt, logits=lg)


def _sample(T, gidx, counts, special, seed, n=N_SAMPLE):
    """>= n token ids (all tokens when T <= n): the special ones (near ties, swaps), spread
    rows, tokens on the most loaded expert and on single-tile experts, then seeded fill."""
    if T <= n:
        return list(range(T))
    sel = set(int(t) for t in special)
    sel |= set(int(t) for t in np.linspace(0, T - 1, n // 4).astype(int))
    hot = int(np.argmax(counts))
    on_hot = np.nonzero((gidx == hot).any(axis=1))[0]
    sel |= set(int(t) for t in on_hot[np.linspace(0, len(on_hot) - 1, min(8, len(on_hot))).astype(int)])
    light = [e for e in np.argsort(counts) if 0 < counts[e] <= 128][:8]
    for e in light:
        sel.add(int(np.nonzero((gidx == e).any(axis=1))[0][0]))
    rs = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(T), np.fromiter(sel, dtype=np.int64))
    need = max(0, n - len(sel))
    sel |= set(int(t) for t in rs.choice(rest, size=min(need, len(rest)), replace=False))
    return sorted(sel)


def _rows(blk, cfg, name, n_rows, n_cols, dtype, rows):
    """Rows of a workspace intermediate, gathered on the device (the buffers are GBs)."""
    import latent_mixture_experts_router_gb300 as lm
    o = lm.lmoe_get_workspace_layout(cfg)[name]
    nb = n_rows * n_cols * torch.tensor([], dtype=dtype).element_size()
    buf = blk._ws[o:o + nb].view(dtype).view(n_rows, n_cols)
    idx = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=buf.device)
    return buf[idx].double().cpu().numpy()


def _stage_errs(blk, cfg, w, sample, gidx, tr_s, ok_local):
    """max |err| / RMS(ref) and RMS(err) / RMS(ref) of p, y, c (BF16 path) and u on the
    sampled tokens whose selection equals the oracle's (ok_local: their positions)."""
    import latent_mixture_experts_router_gb300 as lm
    lay = lm.lmoe_get_workspace_layout(cfg)
    R = w.T * w.k
    toks = np.asarray(sample)[ok_local]
    out = {}

    def err(a, b):
        rms = np.sqrt(np.mean(b * b))
        return float(np.max(np.abs(a - b)) / rms), float(np.sqrt(np.mean((a - b) ** 2)) / rms)
    out["p"] = err(_rows(blk, cfg, "p", w.T, w.L, torch.float32, toks), tr_s.p[ok_local])
    out["u"] = err(_rows(blk, cfg, "u", w.T, w.D, torch.float32, toks), tr_s.u[ok_local])
    if w.weights != "nvfp4":
        out["c"] = err(_rows(blk, cfg, "c", w.T, w.L, torch.bfloat16, toks), tr_s.c[ok_local])
    row_of = _rows(blk, cfg, "row_of", w.T, w.k, torch.int32, toks).astype(np.int64)
    y_rows = row_of.reshape(-1)
    y_dt = torch.bfloat16 if w.weights == "nvfp4" else torch.float32   # y is bf16 on the NVFP4 path
    y_gpu = _rows(blk, cfg, "y", R, w.L, y_dt, y_rows).reshape(len(toks), w.k, w.L)
    loc = np.nonzero(ok_local)[0]
    y_ref = np.stack([np.stack([tr_s.y[(int(t), j)] for j in range(w.k)]) for t in loc])
    out["y"] = err(y_gpu, y_ref)
    assert lay["y"] >= 0
    return out


def _grade(name, w, inp, out, idx, blk, cfg, forced=None):
    t0 = time.time()
    P = oracle.params_from_inputs(inp)       # experts widened one at a time on demand
    gidx = idx.cpu().numpy()
    x = inp.x.double().cpu().numpy()
    near, swaps = [], []
    if forced is not None:
        assert np.array_equal(gidx, forced)
    else:
        _, tr = _full_router(inp, P)
        exact, near, swaps, bad = classify_topk(gidx, tr, w.k)
        print(f"{w.name}: top-k exact {int(exact.sum())}/{w.T}, near ties {len(near)}, order swaps {len(swaps)}")
        assert not bad, bad[:10]
    counts, offsets, row_of, tok_of = expected_permutation(gidx, w.E)
    for name_, n_, ref_ in (("counts", w.E, counts), ("offsets", w.E + 1, offsets),
                            ("row_of", w.T * w.k, row_of.reshape(-1)), ("tok_of", w.T * w.k, tok_of)):
        got = _rows(blk, cfg, name_, 1, n_, torch.int32, [0])[0].astype(np.int64)
        assert np.array_equal(got, ref_), name_
    sample = _sample(w.T, gidx, counts, near + swaps, seed=w.T)
    xs = x[sample]
    fs = None if forced is None else forced[sample]
    tr_s = oracle.Trace()
    ref = oracle.forward_batched(xs, P, w.k, forced_idx=fs, trace=tr_s)
    tol = TOL_NVFP4 if w.weights == "nvfp4" else TOL_BF16
    rep = compare_block(out.cpu().numpy()[sample], gidx[sample], xs, P, w.k, tol, tr=tr_s, ref=ref,
                        forced_idx=fs)
    ok_local = np.all(gidx[sample] == tr_s.idx, axis=1)
    st = _stage_errs(blk, cfg, w, sample, gidx, tr_s, ok_local)
    print(f"{w.name}: {len(sample)} sampled tokens, {rep}; stages (max/RMS, rms/RMS): "
          + ", ".join(f"{k} {a:.3e}/{b:.3e}" for k, (a, b) in st.items())
          + f"; oracle {time.time() - t0:.1f} s")
    assert rep.ok, str(rep)
    if w.weights == "nvfp4":
        # each side quantises its own activations (xn, h0, h, c): a value near a rounding
        # boundary may land on the neighbouring E2M1 code on one side, a difference of up to one
        # E2M1 step (1/3 of the block's scale unit) on that element; those flips are rare and
        # spread, so the RMS error stays small while single elements may differ more
        for k_, (mx, rms) in st.items():
            assert rms < 3e-2 and mx < 0.25, (k_, mx, rms)
    else:
        # bf16 operands (xn_hi, h0, h, c) and fp32 accumulation: each bf16 rounding is 2^-9
        # relative (RMS 2^-9/sqrt(3) = 1.1e-3), and a stage inherits those of the stages before
        # it.  Bar: RMS error at most half the block's 2e-2 output bar; the largest of the
        # 10^5-10^6 compared values (about 5 sigma of roughly Gaussian errors) within 5 times that
        for k_, (mx, rms) in st.items():
            assert rms < 1e-2 and mx < 5e-2, (k_, mx, rms)
    return len(sample)


@pytest.mark.parametrize("name", ["decode_bf16", "prefill_bf16_zipf"])
def test_full_size_bf16(cuda, name):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, cuda)
    out, idx, blk, cfg = run(inp)
    n = _grade(name, w, inp, out, idx, blk, cfg)
    assert n >= min(w.T, N_SAMPLE)
    del out, idx, blk, inp


@pytest.mark.parametrize("name,T,path", [("prefill_nvfp4", None, 0), ("decode_nvfp4_hot", 1, 0),
                                         ("decode_nvfp4_hot", 1, 1), ("decode_nvfp4_hot", 1, 2),
                                         ("decode_nvfp4_hot", 8, 0), ("decode_nvfp4_hot", 32, 0),
                                         ("decode_nvfp4_hot", 128, 0), ("decode_nvfp4_hot", 512, 0)])
def test_full_size_nvfp4(cuda, name, T, path):
    # path (lmoe_ex.single_token_path, T = 1 only): 0 pre/post kernels around the expert GEMMs
    # (the default), 1 one kernel, 2 the stage kernels
    w = workloads.WORKLOADS[name]
    if T is not None:
        w = w.with_tokens(T)
    inp = workloads.make_inputs(w, cuda)
    out, idx, blk, cfg = run(inp, single_token_path=path)
    forced = None if inp.forced_idx is None else inp.forced_idx.cpu().numpy()
    n = _grade(w.name, w, inp, out, idx, blk, cfg, forced=forced)
    assert n >= min(w.T, N_SAMPLE)
    del out, idx, blk, inp
