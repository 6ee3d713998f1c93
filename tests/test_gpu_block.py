"""GPU parity of the latent-MoE block against the fp64 oracle, through the C ABI.

Bars: top-k indices exact (near-tie tokens counted, compared against the oracle re-run
with the GPU's selection); permutation bit-exact; every stage and the output within
2e-2 x RMS of the oracle's value (BF16 compute)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle.compare import TOL_BF16, compare_block

from gpu_util import expected_permutation, make_block, rel_err, run, views

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    return torch.device("cuda:0")


def _oracle(inp, rows=None):
    P = oracle.params_from_inputs(inp)
    x = inp.x.double().cpu().numpy()
    forced = None if inp.forced_idx is None else inp.forced_idx.cpu().numpy()
    tr = oracle.Trace()
    ref = oracle.forward_batched(x, P, inp.w.k, forced_idx=forced, trace=tr)
    return P, x, tr, ref


def _check_permutation(v, idx, E):
    counts, offsets, row_of, tok_of = expected_permutation(idx, E)
    assert np.array_equal(v["counts"], counts)
    assert np.array_equal(v["offsets"], offsets)
    assert np.array_equal(v["row_of"], row_of)
    assert np.array_equal(v["tok_of"], tok_of)
    assert int(v["n_tiles"][0]) == int(np.sum((counts + 127) // 128))


def test_tiny_fp32_stage_by_stage(cuda):
    w = workloads.WORKLOADS["tiny_fp32"]
    inp = workloads.make_inputs(w, cuda)
    out, idx, blk, cfg = run(inp)
    P, x, tr, ref = _oracle(inp)
    v = views(blk, cfg)
    D = w.D
    # S1: xn_hi + xn_lo carries xn to 16 significant bits (|lo| <= 2^-8 |xn|, rounded to bf16)
    assert np.all(np.abs(v["xa"][:, :D] + v["xa"][:, D:2 * D] - tr.xn) <= 2.0 ** -16 * np.abs(tr.xn) + 1e-6)
    # S2: router logits to fp32-level accuracy (well inside the 1e-3 tie band)
    assert np.max(np.abs(v["logits"] - tr.logits)) < 2e-4
    # S3: top-k
    rep = compare_block(out.cpu().numpy(), idx.cpu().numpy(), x, P, w.k, TOL_BF16, tr=tr, ref=ref)
    assert not rep.bad_idx_tokens, str(rep)
    ex = np.all(v["topk_idx"] == tr.idx, axis=1)
    assert np.max(np.abs(v["topk_w"][ex] - tr.w[ex])) < 1e-5
    # S4: permutation, bit-exact against numpy's stable sort of the GPU's own ids
    _check_permutation(v, v["topk_idx"], w.E)
    # S5: pooler (from xn_hi, bf16 weights)
    assert rel_err(v["p"], tr.p) < 2e-2
    # S6: h0 rows in expert-contiguous order
    ok_tok = np.all(v["topk_idx"] == tr.idx, axis=1)
    rows = v["row_of"][ok_tok].reshape(-1)
    toks = np.repeat(np.nonzero(ok_tok)[0], w.k)
    assert rel_err(v["xe"][rows], tr.h0[toks]) < 2e-2
    # S8: per-expert outputs before their norm
    for (t, j), y in list(tr.y.items())[:64]:
        if ok_tok[t]:
            assert rel_err(v["y"][v["row_of"][t, j]], y) < 3e-2
    # S9, S10
    assert rel_err(v["c"][ok_tok], tr.c[ok_tok]) < 2e-2
    assert rel_err(v["u"][ok_tok], tr.u[ok_tok]) < 2e-2
    # output
    assert rep.ok, str(rep)


SHAPES = [  # (T, D, L, E, I, k): ragged T, N tails of the 256-wide tiles, k = 1 and k = E
    (1, 256, 128, 4, 128, 1),
    (3, 384, 256, 8, 384, 2),
    (130, 256, 384, 20, 256, 3),
    (257, 512, 256, 6, 128, 6),
    (200, 256, 128, 1, 256, 1),
    (64, 1024, 512, 64, 768, 8),
    (2, 2048, 1024, 16, 512, 4),    # rows split over clusters of 8 CTAs
    (600, 512, 256, 4, 384, 2),     # 256-row tiles, dense and grouped, ragged last tiles
    (2100, 512, 256, 8, 256, 2),    # router in 256-row tiles split along K, ragged last tile
    (2100, 512, 256, 64, 256, 8),   # 16800 pairs: the chunked permutation
    (12, 256, 128, 1024, 128, 16),  # the header's limits: E = 1024, k = 16 (fused top-k/permutation)
    (40, 256, 128, 1024, 128, 16),  # E = 1024, k = 16 through the separate top-k and permutation
    (1100, 256, 128, 1024, 128, 16),  # E = 1024, k = 16, 17600 pairs: the chunked permutation
    (50, 256, 128, 16, 128, 16),    # k = E = 16
]


@pytest.mark.parametrize("T,D,L,E,I,k", SHAPES)
def test_random_shapes_bf16(cuda, T, D, L, E, I, k):
    w = workloads.Workload(f"shape{T}_{D}_{L}_{E}_{I}_{k}", T=T, D=D, L=L, E=E, I=I, k=k, seed=T % 7)
    inp = workloads.make_inputs(w, cuda)
    out, idx, blk, cfg = run(inp)
    P, x, tr, ref = _oracle(inp)
    rep = compare_block(out.cpu().numpy(), idx.cpu().numpy(), x, P, k, TOL_BF16, tr=tr, ref=ref)
    assert rep.ok, str(rep)
    _check_permutation(views(blk, cfg), idx.cpu().numpy(), E)


def test_zero_tokens(cuda):
    import latent_mixture_experts_router_gb300 as lm
    w = workloads.Workload("t0", T=4, D=256, L=128, E=4, I=128, k=2)
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    x0 = inp.x[:0]
    out = blk.forward(x0)
    torch.cuda.synchronize()
    assert out.shape == (0, 256)
    assert lm.lmoe_check_status(blk.config(0), blk._ws)[0] == 0


@pytest.mark.parametrize("weights,T", [("bf16", 8), ("nvfp4", 8), ("nvfp4", 300)])
def test_capturable_in_cuda_graph(cuda, weights, T):
    # the forward enqueues work only (no host synchronisation, no allocation), side stream
    # included, so it can be captured once and replayed, as a decode loop does
    w = workloads.Workload(f"graph_{weights}_{T}", T=T, D=512, L=256, E=16, I=256, k=4, weights=weights,
                           routing="hot4")
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    out = torch.empty(T, w.D, dtype=torch.float32, device=cuda)
    ex = {"forced_idx": inp.forced_idx} if inp.forced_idx is not None else {}
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        blk.forward(inp.x, out=out, **ex)
    torch.cuda.synchronize()
    ref = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        blk.forward(inp.x, out=out, **ex)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    import latent_mixture_experts_router_gb300 as lm
    assert lm.lmoe_check_status(blk.config(T, w.act, "f32"), blk._ws)[0] == 0


def test_deterministic_and_token_order_equivariant(cuda):
    w = workloads.Workload("det", T=300, D=512, L=256, E=16, I=256, k=4)
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    a, ia, _, _ = run(inp, blk=blk)
    a = a.clone()
    b, ib, _, _ = run(inp, blk=blk)
    assert torch.equal(a, b) and torch.equal(ia, ib)
    perm = torch.randperm(w.T, generator=torch.Generator().manual_seed(0)).to(cuda)
    c, ic, _, _ = run(inp, blk=blk, x=inp.x[perm].contiguous())
    assert torch.equal(c, a[perm]) and torch.equal(ic, ia[perm])


@pytest.mark.parametrize("T,k,routing", [(16, 4, "uniform"), (40, 6, "hot4"), (100, 3, "zipf")])
def test_overlapped_and_serial_paths_agree(cuda, T, k, routing):
    # Without stage events the pooler runs on the side stream and, for at most 256 (token,
    # slot) pairs, top-k and the permutation run as one kernel; with every stage timed the
    # call runs serially through separate kernels.  Both give bit-identical results.
    import latent_mixture_experts_router_gb300 as lm
    w = workloads.Workload(f"paths_{T}_{k}", T=T, D=512, L=256, E=32, I=256, k=k, routing=routing,
                           seed=T)
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    a, ia, _, cfg = run(inp, blk=blk)
    a = a.clone()
    va = views(blk, cfg)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(lm.NUM_STAGE_EVENTS)]
    b, ib, _, _ = run(inp, blk=blk, stage_events=evs)
    vb = views(blk, cfg)
    assert torch.equal(a, b) and torch.equal(ia, ib)
    for name in ("topk_w", "counts", "offsets", "row_of", "tok_of", "n_tiles", "p", "y", "u"):
        assert np.array_equal(va[name], vb[name]), name
    _check_permutation(va, ia.cpu().numpy(), w.E)


def test_router_bias_and_forced_routing(cuda):
    w = workloads.Workload("bias", T=96, D=256, L=128, E=32, I=256, k=4, routing="zipf")
    inp = workloads.make_inputs(w, cuda)
    out, idx, _, _ = run(inp)
    P, x, tr, ref = _oracle(inp)
    rep = compare_block(out.cpu().numpy(), idx.cpu().numpy(), x, P, w.k, TOL_BF16, tr=tr, ref=ref)
    assert rep.ok, str(rep)
    w2 = workloads.Workload("forced", T=33, D=256, L=128, E=32, I=256, k=8, routing="hot4")
    inp2 = workloads.make_inputs(w2, cuda)
    out2, idx2, _, _ = run(inp2)
    assert torch.equal(idx2.cpu(), inp2.forced_idx.cpu())
    P2, x2, tr2, ref2 = _oracle(inp2)
    rep2 = compare_block(out2.cpu().numpy(), idx2.cpu().numpy(), x2, P2, w2.k, TOL_BF16, tr=tr2, ref=ref2)
    assert rep2.ok, str(rep2)


def test_bf16_output_and_host_io(cuda):
    import latent_mixture_experts_router_gb300 as lm
    w = workloads.Workload("io", T=70, D=256, L=256, E=8, I=128, k=2)
    inp = workloads.make_inputs(w, cuda)
    out32, _, blk, _ = run(inp)
    out16, _, _, _ = run(inp, out_dtype="bf16", blk=blk)
    assert out16.dtype == torch.bfloat16
    assert torch.equal(out16.float(), out32.to(torch.bfloat16).float())
    cfg = blk.config(w.T, "bf16", "f32")
    ws = torch.empty(lm.lmoe_workspace_size_host_io(cfg), dtype=torch.uint8, device=cuda)
    xh = inp.x.cpu().pin_memory()
    oh = torch.empty(w.T, w.D, dtype=torch.float32).pin_memory()
    W = blk.W
    lm.latent_moe_forward_host_io(cfg, xh, W["W_router"], W["W_pool"], W["g_pool"], W["W_gate"], W["W_up"],
                                  W["W_down"], W["g_expert"], W["W_unpool"], W["g_pre"], W["g_post"], w.k,
                                  oh, ws)
    torch.cuda.synchronize()
    assert torch.equal(oh, out32.cpu())


@pytest.mark.parametrize("routing", ["zipf", "hot4"])
def test_host_io_with_routing_controls(cuda, routing):
    # x in and out back through pinned host memory, with the router bias (Zipf) or forced
    # routing (hot experts) of lmoe_ex: the same result as the device-resident call
    import latent_mixture_experts_router_gb300 as lm
    w = workloads.Workload(f"io_{routing}", T=40, D=256, L=256, E=16, I=128, k=4, routing=routing)
    inp = workloads.make_inputs(w, cuda)
    out, _, blk, _ = run(inp)
    cfg = blk.config(w.T, "bf16", "f32")
    ws = torch.zeros(lm.lmoe_workspace_size_host_io(cfg), dtype=torch.uint8, device=cuda)
    xh = inp.x.cpu().pin_memory()
    oh = torch.empty(w.T, w.D, dtype=torch.float32).pin_memory()
    W = blk.W
    lm.latent_moe_forward_host_io_ex(cfg, xh, W["W_router"], W["W_pool"], W["g_pool"], W["W_gate"], W["W_up"],
                                     W["W_down"], W["g_expert"], W["W_unpool"], W["g_pre"], W["g_post"], w.k,
                                     oh, ws, router_bias=inp.router_bias, forced_idx=inp.forced_idx)
    torch.cuda.synchronize()
    assert torch.equal(oh, out.cpu())


@pytest.mark.parametrize("T,out_dtype", [(40, "f32"), (40, "bf16"), (300, "f32")])
def test_next_layer_pre_norm(cuda, T, out_dtype):
    # S11 also writing RMSNorm(out) * g_next (the next layer's pre-norm from the same row; at
    # T = 40 the row is split over a cluster of 4 CTAs): out itself is unchanged, and the extra
    # output is the RMSNorm of out as stored, within fp32 rounding
    w = workloads.Workload(f"next_{T}", T=T, D=1024, L=256, E=8, I=256, k=2, seed=3)
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    base, _, _, _ = run(inp, blk=blk, out_dtype=out_dtype)
    base = base.clone()
    g_next = (1.0 + 0.1 * torch.randn(w.D, generator=torch.Generator().manual_seed(5), dtype=torch.float64)
              ).to(torch.float32).to(cuda)
    nxt = torch.empty(w.T, w.D, dtype=base.dtype, device=cuda)
    out, _, _, _ = run(inp, blk=blk, out_dtype=out_dtype, next_norm_gamma=g_next, next_norm_out=nxt)
    assert torch.equal(out, base)
    ref = oracle.rms_norm(out.double().cpu().numpy(), g_next.double().cpu().numpy(), w.eps)
    err = np.abs(nxt.double().cpu().numpy() - ref).max() / np.sqrt(np.mean(ref ** 2))
    assert err < (4e-6 if out_dtype == "f32" else 1.6e-2), err   # fp32 rounding; bf16 half-ulp at |v| <= 4 RMS


@pytest.mark.parametrize("bad_row", [[3, 99], [5, 5]], ids=["out_of_range", "repeated"])
def test_bad_forced_id_is_flagged(cuda, bad_row):
    import latent_mixture_experts_router_gb300 as lm
    w = workloads.Workload("badidx", T=8, D=256, L=128, E=8, I=128, k=2)
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    forced = torch.tensor([[0, 1]] * 7 + [bad_row], dtype=torch.int32, device=cuda)
    blk.forward(inp.x, forced_idx=forced)
    st, word = lm.lmoe_check_status(blk.config(w.T), blk._ws)
    assert st == -1 and word & (1 << 3)
    # the context stays usable
    out, idx, _, _ = run(inp, blk=blk)
    assert torch.isfinite(out).all()


def test_wait_budget_runs_out_and_reports(cuda):
    import latent_mixture_experts_router_gb300 as lm
    w = workloads.Workload("tmo", T=8, D=256, L=128, E=8, I=128, k=2)
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    cfg = blk.config(w.T)
    blk.workspace(cfg)
    # a barrier nothing arrives on: the wait gives up after ~1e6 cycles and says so
    lm.lmoe_wait_selftest(cfg, blk._ws, 1_000_000)
    st, word = lm.lmoe_check_status(cfg, blk._ws)
    assert st == -6 and word != 0
    # the block itself under a 1-cycle budget: either finishes or reports the timeout,
    # and the context stays usable afterwards
    blk.forward(inp.x, wait_budget_cycles=1)
    st, _ = lm.lmoe_check_status(cfg, blk._ws)
    assert st in (0, -6)
    out, idx, _, _ = run(inp, blk=blk)
    P, x, tr, ref = _oracle(inp)
    assert compare_block(out.cpu().numpy(), idx.cpu().numpy(), x, P, w.k, TOL_BF16, tr=tr, ref=ref).ok


@pytest.mark.parametrize("T,k,weights", [(8, 2, "bf16"), (300, 4, "bf16"), (8, 2, "nvfp4"), (300, 4, "nvfp4")])
def test_nan_token_routes_to_valid_experts(cuda, T, k, weights):
    # A NaN in one token's input makes all of its router logits NaN.  The top-k orders NaN as
    # -inf, so the token still gets k distinct valid experts (the lowest ids), the call reports
    # no error, and the other tokens keep their routing and outputs (bitwise with BF16
    # weights; with NVFP4 the grouped GEMMs may pick another split count, so they are graded
    # against the oracle instead).  T = 8 takes the fused top-k + permutation kernel, T = 300
    # the separate ones.
    w = workloads.Workload(f"nan_{T}_{weights}", T=T, D=256, L=256, E=16, I=256, k=k, weights=weights, seed=2)
    inp = workloads.make_inputs(w, cuda)
    out0, idx0, blk, _ = run(inp)
    out0, idx0 = out0.clone(), idx0.clone()
    x = inp.x.clone()
    x[3, 5] = float("nan")
    out1, idx1, _, _ = run(inp, blk=blk, x=x)        # run() asserts the device status is OK
    assert idx1[3].cpu().tolist() == list(range(k))
    keep = torch.ones(T, dtype=torch.bool, device=cuda)
    keep[3] = False
    assert torch.equal(idx1[keep], idx0[keep])
    assert bool(torch.isfinite(out1[keep]).all())
    if weights == "bf16":
        assert torch.equal(out1[keep], out0[keep])
    else:
        P, xs, tr, ref = _oracle(inp)
        kk = keep.cpu().numpy()
        rep = compare_block(out1.cpu().numpy()[kk], idx1.cpu().numpy()[kk], xs[kk], P, k, 6e-2)
        assert rep.ok, str(rep)
