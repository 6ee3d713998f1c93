"""Parity at the full Muse shapes (D 8192, L 4096, E 256, I 4096, k 8), in the launch
configuration the benchmark times.

Every token: top-k ids exact against the oracle's fp64 router (near ties counted), and the
permutation bit-exact.  Sampled tokens: the block output against the oracle (the block is
token-independent, so a token's expected output needs only its own row and the weights of
the experts it routes to)."""
import gc

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle.compare import TOL_BF16, classify_topk, compare_block

from gpu_util import expected_permutation, run, views

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


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


@pytest.mark.parametrize("name,sample", [("decode_bf16", [0, 41, 77, 127]),
                                         ("prefill_bf16_zipf", [0, 5000, 12345, 16383])])
def test_full_size_bf16(cuda, name, sample):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, cuda)
    out, idx, blk, cfg = run(inp)
    P = oracle.params_from_inputs(inp)       # experts widened one at a time on demand
    x, tr = _full_router(inp, P)
    gidx = idx.cpu().numpy()
    exact, near, swaps, bad = classify_topk(gidx, tr, w.k)
    print(f"{name}: top-k exact {int(exact.sum())}/{w.T}, near ties {len(near)}, order swaps {len(swaps)}")
    assert not bad, bad[:10]
    v = views(blk, cfg)
    counts, offsets, row_of, tok_of = expected_permutation(gidx, w.E)
    assert np.array_equal(v["counts"], counts) and np.array_equal(v["offsets"], offsets)
    assert np.array_equal(v["row_of"], row_of) and np.array_equal(v["tok_of"], tok_of)
    # sampled tokens through the oracle
    xs = x[sample]
    tr_s = oracle.Trace()
    ref = oracle.forward_batched(xs, P, w.k, trace=tr_s)
    rep = compare_block(out.cpu().numpy()[sample], gidx[sample], xs, P, w.k, TOL_BF16, tr=tr_s, ref=ref)
    print(name, rep)
    assert rep.ok, str(rep)
    del out, idx, blk, inp, v


@pytest.mark.parametrize("name,T,sample", [("prefill_nvfp4", None, [0, 1234, 4095]),
                                           ("decode_nvfp4_hot", 1, [0]),
                                           ("decode_nvfp4_hot", 8, [0, 7]),
                                           ("decode_nvfp4_hot", 32, [3, 31]),
                                           ("decode_nvfp4_hot", 128, [0, 127]),
                                           ("decode_nvfp4_hot", 512, [5, 300, 511])])
def test_full_size_nvfp4(cuda, name, T, sample):
    from oracle.compare import TOL_NVFP4
    w = workloads.WORKLOADS[name]
    if T is not None:
        w = w.with_tokens(T)
    inp = workloads.make_inputs(w, cuda)
    out, idx, blk, cfg = run(inp)
    gidx = idx.cpu().numpy()
    P = oracle.params_from_inputs(inp)
    x = inp.x.double().cpu().numpy()
    forced = None if inp.forced_idx is None else inp.forced_idx.cpu().numpy()
    if forced is not None:
        assert np.array_equal(gidx, forced)
    else:
        _, tr = _full_router(inp, P)
        exact, near, swaps, bad = classify_topk(gidx, tr, w.k)
        print(f"{w.name}: top-k exact {int(exact.sum())}/{w.T}, near ties {len(near)}, swaps {len(swaps)}")
        assert not bad, bad[:10]
    v = views(blk, cfg)
    counts, offsets, row_of, tok_of = expected_permutation(gidx, w.E)
    assert np.array_equal(v["row_of"], row_of) and np.array_equal(v["tok_of"], tok_of)
    xs = x[sample]
    fs = None if forced is None else forced[sample]
    tr_s = oracle.Trace()
    ref = oracle.forward_batched(xs, P, w.k, forced_idx=fs, trace=tr_s)
    rep = compare_block(out.cpu().numpy()[sample], gidx[sample], xs, P, w.k, TOL_NVFP4, tr=tr_s,
                        ref=ref, forced_idx=fs)
    print(w.name, rep)
    assert rep.ok, str(rep)
    del out, idx, blk, inp, v
