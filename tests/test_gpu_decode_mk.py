"""GPU parity of the single-token NVFP4 paths (lmoe_ex.single_token_path): the default —
cooperative pre and post kernels around the tensor-core expert GEMMs (0) — and the whole block
as one cooperative kernel (1).

* Against the fp64 oracle, under the NVFP4 rules (top-k exact with near ties counted, output
  within 6e-2 x RMS, near-boundary roundings accepted only as a legitimate alternative), over
  every lane layout of the dot products (64-code chunks per lane 1 to 4: D, L, I from 256 to
  8192), fp32 and bf16 inputs and outputs, zipf router bias, forced routing, E = 1024, k = 16.
* Against the kernel chain on the same call (SINGLE_TOKEN_CHAIN = 2): the same experts and
  routing tables bit for bit, and p, y, u and the output within the fp32 reordering of the
  same products (both compute every block's products exactly; the sums differ in order).
* Two launches of the library per call for the whole-block path (the kernel that clears the
  call's counters, then the block kernel); a grid barrier whose wait budget runs out ends the
  call with LMOE_ERR_TIMEOUT (bit 0x40) and leaves the context usable; stage events select the
  chain.
* The next layer's pre-norm from the same row; a cooperative launch (lmoe_ex.cooperative_launch)
  gives the same call bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle.compare import TOL_NVFP4, compare_block

from gpu_util import make_block, run, views

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    return torch.device("cuda:0")


SHAPES = [  # (D, L, E, I, k, act, routing): chunks per lane = ceil(max(D, L, I) / 2048)
    (256, 256, 4, 256, 2, "bf16", "uniform"),
    (512, 256, 8, 512, 2, "f32", "uniform"),
    (2048, 1024, 16, 512, 4, "bf16", "zipf"),
    (4096, 2048, 16, 1024, 8, "bf16", "uniform"),
    (6144, 512, 8, 512, 2, "bf16", "uniform"),
    (8192, 4096, 32, 1024, 8, "f32", "hot4"),
    (256, 256, 1024, 256, 16, "bf16", "uniform"),
]


def _workload(D, L, E, I, k, act, routing, seed=1):
    return workloads.Workload(f"mk_{D}_{L}_{E}_{I}_{k}_{act}_{routing}", T=1, D=D, L=L, E=E, I=I, k=k, act=act,
                              weights="nvfp4", routing=routing, seed=seed)


def _launches(lm, fn):
    torch.cuda.synchronize()
    n0 = lm.lmoe_kernel_launches()
    fn()
    torch.cuda.synchronize()
    return lm.lmoe_kernel_launches() - n0


@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("D,L,E,I,k,act,routing", SHAPES)
def test_single_token_parity_with_oracle(cuda, D, L, E, I, k, act, routing, path):
    import latent_mixture_experts_router_gb300 as lm
    w = _workload(D, L, E, I, k, act, routing)
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    n = _launches(lm, lambda: run(inp, blk=blk, single_token_path=path))
    chain = _launches(lm, lambda: run(inp, blk=blk, single_token_path=2))
    # the whole block as one kernel after the clear kernel; the default: the pre and post kernels
    # and the expert GEMMs
    assert (n == 2) if path == 1 else (2 < n < chain), (n, chain)
    out, idx, _, _ = run(inp, blk=blk, single_token_path=path)
    P = oracle.params_from_inputs(inp)
    x = inp.x.double().cpu().numpy()
    forced = None if inp.forced_idx is None else inp.forced_idx.cpu().numpy()
    tr = oracle.Trace()
    ref = oracle.forward_batched(x, P, k, trace=tr, forced_idx=forced)
    rep = compare_block(out.cpu().numpy(), idx.cpu().numpy(), x, P, k, TOL_NVFP4, tr=tr, ref=ref, forced_idx=forced)
    print(w.name, rep)
    assert rep.ok, str(rep)


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.sqrt(np.mean(b ** 2)), 1e-30))


@pytest.mark.parametrize("D,L,E,I,k,act,routing", [SHAPES[0], SHAPES[3], SHAPES[5], SHAPES[6]])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", [0, 1])
def test_single_token_matches_kernel_chain(cuda, D, L, E, I, k, act, routing, out_dtype, path):
    import latent_mixture_experts_router_gb300 as lm
    w = _workload(D, L, E, I, k, act, routing, seed=2)
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    assert _launches(lm, lambda: run(inp, blk=blk, out_dtype=out_dtype, single_token_path=2)) > 2
    out_c, idx_c, _, cfg = run(inp, blk=blk, out_dtype=out_dtype, single_token_path=2)
    out_c = out_c.clone()
    vc = views(blk, cfg)
    out_m, idx_m, _, _ = run(inp, blk=blk, out_dtype=out_dtype, single_token_path=path)
    vm = views(blk, cfg)
    assert torch.equal(idx_m, idx_c)
    for name in ("topk_idx", "counts", "offsets", "row_of", "tok_of", "n_tiles"):
        assert np.array_equal(vm[name], vc[name]), name
    # the row reductions run in another order (a last-bit change of a norm's scale), the router
    # reads fp32 xn where the chain reads its bf16 hi + lo split (2^-17 relative), and the same
    # exact block products are summed in another order; amplified only where a requantisation
    # rounds across a code boundary (rare: one code step of one element in a block)
    D_ = w.D
    xa_m, xa_c = vm["xa"][:, :D_] + vm["xa"][:, D_:2 * D_], vc["xa"][:, :D_] + vc["xa"][:, D_:2 * D_]
    assert _rel(xa_m, xa_c) < 2e-5   # one bf16 ulp of the low half
    assert _rel(vm["logits"], vc["logits"]) < 1e-4
    assert _rel(vm["topk_w"], vc["topk_w"]) < 1e-4
    assert _rel(vm["p"], vc["p"]) < 2e-2
    rows = vm["row_of"].reshape(-1)
    assert _rel(vm["y"][rows], vc["y"][rows]) < 2e-2
    assert _rel(vm["u"], vc["u"]) < 2e-2
    assert _rel(out_m.double().cpu().numpy(), out_c.double().cpu().numpy()) < 2e-2


@pytest.mark.parametrize("path", [0, 1])
def test_grid_barrier_timeout_is_reported_and_context_survives(cuda, path):
    import latent_mixture_experts_router_gb300 as lm
    w = _workload(2048, 1024, 16, 512, 4, "bf16", "uniform", seed=3)
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    ref, _, _, cfg = run(inp, blk=blk, single_token_path=path)
    ref = ref.clone()
    # a budget of one cycle: the waits give up (the first grid barrier at the latest)
    blk.forward(inp.x, wait_budget_cycles=1, single_token_path=path)
    st, word = lm.lmoe_check_status(cfg, blk._ws)
    assert st == -6 and word & 0x40, (st, hex(word))
    out, _, _, _ = run(inp, blk=blk, single_token_path=path)
    assert torch.equal(out, ref)


@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_single_token_next_layer_pre_norm(cuda, out_dtype, path):
    w = _workload(4096, 1024, 8, 512, 2, "bf16", "uniform", seed=4)
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    base, _, _, _ = run(inp, blk=blk, out_dtype=out_dtype, single_token_path=path)
    base = base.clone()
    g_next = (1.0 + 0.1 * torch.randn(w.D, generator=torch.Generator().manual_seed(5), dtype=torch.float64)
              ).to(torch.float32).to(cuda)
    nxt = torch.empty(1, w.D, dtype=base.dtype, device=cuda)
    out, _, _, _ = run(inp, blk=blk, out_dtype=out_dtype, next_norm_gamma=g_next, next_norm_out=nxt,
                       single_token_path=path)
    assert torch.equal(out, base)
    ref = oracle.rms_norm(out.double().cpu().numpy(), g_next.double().cpu().numpy(), w.eps)
    err = np.abs(nxt.double().cpu().numpy() - ref).max() / np.sqrt(np.mean(ref ** 2))
    assert err < (4e-6 if out_dtype == "f32" else 1.6e-2), err


def test_stage_events_take_the_chain_and_16_byte_codes_the_kernel(cuda):
    import latent_mixture_experts_router_gb300 as lm
    w = _workload(512, 256, 8, 256, 2, "bf16", "uniform", seed=5)
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(lm.NUM_STAGE_EVENTS)]
    assert _launches(lm, lambda: run(inp, blk=blk, stage_events=evs, single_token_path=1)) > 1
    ref, idx_ref, _, _ = run(inp, blk=blk, single_token_path=1)
    ref = ref.clone()
    # codes at 16 (not 32) bytes past an allocation: the bulk copies need 16
    codes, scales, s, layout = blk.W["W_pool"]
    buf = torch.empty(codes.numel() + 16, dtype=torch.uint8, device=cuda)
    shifted = buf[16:16 + codes.numel()].view_as(codes)
    shifted.copy_(codes)
    assert shifted.data_ptr() % 32 == 16
    blk.W["W_pool"] = (shifted, scales, s, layout)
    assert _launches(lm, lambda: run(inp, blk=blk, single_token_path=1)) == 2
    out, idx, _, _ = run(inp, blk=blk, single_token_path=1)
    assert torch.equal(out, ref) and torch.equal(idx, idx_ref)


def test_single_token_path_out_of_range_is_refused(cuda):
    import latent_mixture_experts_router_gb300 as lm
    w = _workload(256, 256, 4, 256, 2, "bf16", "uniform")
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    with pytest.raises(lm.LmoeError):
        blk.forward(inp.x, single_token_path=3)
    with pytest.raises(lm.LmoeError):
        blk.forward(inp.x, single_token_path=-1)


@pytest.mark.parametrize("path", [0, 1])
def test_cooperative_launch_gives_the_same_call(cuda, path):
    # lmoe_ex.cooperative_launch: the same kernels launched cooperatively, bit for bit the same
    w = _workload(4096, 2048, 16, 1024, 8, "bf16", "uniform", seed=6)
    inp = workloads.make_inputs(w, cuda)
    blk = make_block(inp)
    a, ia, _, _ = run(inp, blk=blk, single_token_path=path)
    a = a.clone()
    b, ib, _, _ = run(inp, blk=blk, single_token_path=path, cooperative_launch=True)
    assert torch.equal(a, b) and torch.equal(ia, ib)
