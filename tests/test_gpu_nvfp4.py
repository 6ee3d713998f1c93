"""GPU parity of the NVFP4 path.

* The quantiser: the same fp32 rows through lmoe_quantize_nvfp4 and through the oracle's
  rule (oracle.formats.quantize_activation, every rounding decision in fp32) give the same
  codes (compared as values, so +0 and -0 agree), block scales and row scales.
* The block with NVFP4 weights and activations against the fp64 oracle that dequantises the
  same packed weights and applies the same activation rule to its own values: top-k exact
  (near ties counted), output max-abs error <= 6e-2 x RMS."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import formats as F
from oracle.compare import TOL_NVFP4, compare_block
from workloads import rng

from gpu_util import run, views

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    return torch.device("cuda:0")


def _rows(n, K, seed):
    # wide dynamic range per row, exact zeros and a few huge blocks
    z = rng.normal(seed, 77, 0, n * K, 1.0).view(n, K)
    mag = torch.exp2(torch.arange(n, dtype=torch.float64) % 40 - 20).view(n, 1)
    v = (z * mag).to(torch.float32)
    v[1] = 0.0
    v[2, :16] = 0.0
    v[3, 32:48] *= 1e4
    return v


@pytest.mark.parametrize("row_scale", [True, False])
def test_quantizer_bit_exact_against_rule(cuda, row_scale):
    import latent_mixture_experts_router_gb300 as lm
    n, K = 64, 1024
    v = _rows(n, K, 3)
    if not row_scale:
        v = v / v.abs().amax(dim=1, keepdim=True).clamp_min(1e-30)
    dv = v.to(cuda)
    codes = torch.empty(n, K // 2, dtype=torch.uint8, device=cuda)
    scales = torch.empty(n, K // 16, dtype=torch.uint8, device=cuda)
    s = torch.empty(n, dtype=torch.float32, device=cuda)
    lm.lmoe_quantize_nvfp4(dv, codes, scales, s, row_scale=row_scale)
    torch.cuda.synchronize()
    q_ref, sc_ref, s_ref = F.quantize_activation(v.double().numpy(), row_scale=row_scale)
    q_gpu = F.nvfp4_unpack_codes(codes.cpu().numpy())
    assert np.array_equal(F.E2M1_TABLE[q_gpu], F.E2M1_TABLE[q_ref])
    assert np.array_equal(scales.cpu().numpy(), sc_ref)
    if row_scale:
        assert np.array_equal(s.cpu().numpy(), s_ref)


SHAPES = [  # (T, D, L, E, I, k)
    (1, 256, 256, 4, 256, 2),
    (37, 512, 256, 8, 256, 2),
    (130, 256, 512, 16, 512, 4),
    (257, 512, 256, 6, 256, 6),
    (2, 2048, 1024, 8, 512, 2),     # rows split over clusters of 8 CTAs
    (20, 4096, 4096, 4, 256, 2),    # clusters of 8, one quantisation block per thread
    (24, 256, 256, 1024, 256, 16),  # the header's limits: E = 1024, k = 16
    (10, 512, 256, 64, 256, 16),
]
# few rows and a long K: the grouped GEMMs split K (count picked on the device); gate/up
# splits in the first two, down in the last
SPLIT_SHAPES = [  # (T, D, L, E, I, k)
    (2, 512, 4096, 8, 1024, 2),
    (5, 256, 4096, 16, 512, 3),
    (1, 256, 256, 4, 4096, 2),
]


@pytest.mark.parametrize("T,D,L,E,I,k", SHAPES)
def test_nvfp4_block_parity(cuda, T, D, L, E, I, k):
    w = workloads.Workload(f"fp4_{T}_{D}_{L}_{E}_{I}_{k}", T=T, D=D, L=L, E=E, I=I, k=k,
                           weights="nvfp4", seed=T % 5)
    inp = workloads.make_inputs(w, cuda)
    out, idx, blk, cfg = run(inp)
    P = oracle.params_from_inputs(inp)
    x = inp.x.double().cpu().numpy()
    tr = oracle.Trace()
    ref = oracle.forward_batched(x, P, k, trace=tr)
    rep = compare_block(out.cpu().numpy(), idx.cpu().numpy(), x, P, k, TOL_NVFP4, tr=tr, ref=ref)
    print(w.name, rep)
    assert rep.ok, str(rep)


@pytest.mark.parametrize("T,D,L,E,I,k", [(130, 1024, 512, 8, 256, 2), (5, 2048, 1024, 8, 512, 2)])
def test_nvfp4_f32_activations(cuda, T, D, L, E, I, k):
    # fp32 x into the NVFP4 path: the pre-norm reads float4 chunks instead of bf16 ones
    w = workloads.Workload(f"fp4x32_{T}_{D}", T=T, D=D, L=L, E=E, I=I, k=k, weights="nvfp4", act="f32",
                           seed=T % 5)
    inp = workloads.make_inputs(w, cuda)
    assert inp.x.dtype == torch.float32
    out, idx, blk, cfg = run(inp)
    P = oracle.params_from_inputs(inp)
    x = inp.x.double().cpu().numpy()
    tr = oracle.Trace()
    ref = oracle.forward_batched(x, P, k, trace=tr)
    rep = compare_block(out.cpu().numpy(), idx.cpu().numpy(), x, P, k, TOL_NVFP4, tr=tr, ref=ref)
    assert rep.ok, str(rep)


@pytest.mark.parametrize("T,D,L,E,I,k", SPLIT_SHAPES)
def test_nvfp4_grouped_split_parity(cuda, T, D, L, E, I, k):
    import latent_mixture_experts_router_gb300 as lm
    w = workloads.Workload(f"fp4s_{T}_{D}_{L}_{E}_{I}_{k}", T=T, D=D, L=L, E=E, I=I, k=k,
                           weights="nvfp4", seed=T)
    inp = workloads.make_inputs(w, cuda)
    out, idx, blk, cfg = run(inp)
    lay = lm.lmoe_get_workspace_layout(cfg)
    o = lay["grouped_splits"]
    splits = blk._ws[o:o + 8].view(torch.int32).cpu().tolist()
    n_tiles = int(blk._ws[lay["n_tiles"]:lay["n_tiles"] + 4].view(torch.int32).item())
    # the device's choice against the rule: fill the last wave of the persistent grid best,
    # with the smallest divisor of the K blocks that gains more than 2 %
    grid = torch.cuda.get_device_properties(cuda).multi_processor_count
    s_max = min(8, max(1, (L // 128) // T))

    def rule(units, num_kb):
        if s_max <= 1 or units >= 3 * grid:
            return 1
        best, best_eff = 1, units / (-(-units // grid) * grid)
        for s in range(2, min(s_max, num_kb // 8) + 1):   # at least 8 K blocks per split
            if num_kb % s == 0:
                eff = units * s / (-(-units * s // grid) * grid)
                if eff > best_eff + 0.02:
                    best, best_eff = s, eff
        return best
    assert splits == [rule(n_tiles * (I // 128), L // 256), rule(n_tiles * (L // 128), I // 256)], splits
    assert max(splits) > 1, splits   # a grouped GEMM took the split path
    P = oracle.params_from_inputs(inp)
    x = inp.x.double().cpu().numpy()
    tr = oracle.Trace()
    ref = oracle.forward_batched(x, P, k, trace=tr)
    rep = compare_block(out.cpu().numpy(), idx.cpu().numpy(), x, P, k, TOL_NVFP4, tr=tr, ref=ref)
    print(w.name, splits, rep)
    assert rep.ok, str(rep)


def test_nvfp4_pooler_stage(cuda):
    # the pooler output against the oracle's: same packed weights, each side quantising its
    # own xn by the rule (flips at quantisation boundaries stay rare and small)
    w = workloads.Workload("fp4_stage", T=64, D=512, L=256, E=8, I=256, k=2, weights="nvfp4")
    inp = workloads.make_inputs(w, cuda)
    out, idx, blk, cfg = run(inp)
    v = views(blk, cfg)
    P = oracle.params_from_inputs(inp)
    tr = oracle.Trace()
    oracle.forward_batched(inp.x.double().cpu().numpy(), P, w.k, trace=tr)
    err = np.abs(v["p"] - tr.p)
    rms = np.sqrt(np.mean(tr.p ** 2))
    assert np.sqrt(np.mean(err ** 2)) < 2e-2 * rms and err.max() < 0.15 * rms, (err.max() / rms)


def _gaussian_packed(w, name, seed):
    """A weight drawn from a Gaussian with per-(row, 16-block) magnitudes 2^-u, u uniform in
    [0, 16], packed by the oracle's plain NVFP4 definition (one tensor scale per matrix, per
    expert for stacks): block scales then span the E4M3 range down to its subnormals."""
    import math
    from workloads import configs
    stream, per_e, rows, cols, fan_in = configs.weight_specs(w)[name]
    n = w.E if per_e else 1
    W = configs.normal_tensor(w, stream, (n, rows, cols), 1.0 / math.sqrt(fan_in), "f32").double().numpy()
    u = np.random.default_rng(seed).uniform(0, 16, size=(n, rows, cols // 16))
    W = W * np.repeat(np.exp2(-u), 16, axis=2)
    packed = [F.quantize_weight(W[e]) for e in range(n)]
    codes = torch.from_numpy(np.stack([p[0] for p in packed]))
    scales = torch.from_numpy(np.stack([p[1] for p in packed]))
    s = torch.tensor([float(p[2]) for p in packed], dtype=torch.float32)
    if not per_e:
        codes, scales = codes[0], scales[0]
    return codes, scales, s


@pytest.mark.parametrize("T,D,L,E,I,k", [(37, 512, 256, 8, 256, 2), (130, 256, 512, 16, 512, 4)])
def test_nvfp4_block_parity_gaussian_quantised_weights(cuda, T, D, L, E, I, k):
    # weights quantised from a Gaussian draw (not drawn as codes): the block-scaled MMAs see
    # subnormal, small and large E4M3 block scales and one tensor scale per matrix/expert
    import dataclasses
    w = workloads.Workload(f"fp4g_{T}_{D}", T=T, D=D, L=L, E=E, I=I, k=k, weights="nvfp4", seed=T % 5)
    inp = workloads.make_inputs(w, "cpu")
    repl = {n: _gaussian_packed(w, n, seed=i) for i, n in enumerate(("W_pool", "W_gate", "W_up", "W_down",
                                                                      "W_unpool"))}
    sc_all = np.concatenate([v[1].numpy().reshape(-1) for v in repl.values()])
    assert np.any((sc_all & 0x78) == 0) and np.any(sc_all >= 0x70), "scales do not span the range"
    inp = workloads.to_device(dataclasses.replace(inp, **repl), cuda)
    out, idx, blk, cfg = run(inp)
    P = oracle.params_from_inputs(inp)
    x = inp.x.double().cpu().numpy()
    tr = oracle.Trace()
    ref = oracle.forward_batched(x, P, k, trace=tr)
    rep = compare_block(out.cpu().numpy(), idx.cpu().numpy(), x, P, k, TOL_NVFP4, tr=tr, ref=ref)
    print(w.name, rep)
    assert rep.ok, str(rep)


def test_nvfp4_wide_dense_tiles(cuda):
    # enough rows for the pooler and unpooler to take 128 x 256 tiles (at least two waves of
    # them, unsplit), with a ragged last M tile; graded on sampled tokens (token-independent)
    T, D, L, E, I, k = 2600, 4096, 4096, 16, 256, 2
    assert -(-T // 128) * (L // 256) >= 2 * 152 and -(-T // 128) * (D // 256) >= 2 * 152
    w = workloads.Workload("fp4_wide", T=T, D=D, L=L, E=E, I=I, k=k, weights="nvfp4", seed=4)
    inp = workloads.make_inputs(w, cuda)
    out, idx, blk, cfg = run(inp)
    sample = [0, 1, 127, 128, 255, 1000, 2047, 2048, 2559, 2560, 2561, 2598, 2599]
    P = oracle.params_from_inputs(inp)
    xs = inp.x.double().cpu().numpy()[sample]
    tr = oracle.Trace()
    ref = oracle.forward_batched(xs, P, k, trace=tr)
    gidx = idx.cpu().numpy()[sample]
    rep = compare_block(out.cpu().numpy()[sample], gidx, xs, P, k, TOL_NVFP4, tr=tr, ref=ref)
    print(w.name, rep)
    assert rep.ok, str(rep)
    import latent_mixture_experts_router_gb300 as lm
    o = lm.lmoe_get_workspace_layout(cfg)["p"]
    p = blk._ws[o:o + 4 * T * L].view(torch.float32).view(T, L)[sample].double().cpu().numpy()
    err = np.abs(p - tr.p)
    rms = np.sqrt(np.mean(tr.p ** 2))
    assert np.sqrt(np.mean(err ** 2)) < 2e-2 * rms and err.max() < 0.15 * rms, (err.max() / rms)


def test_row_major_scales_refused_blocked_accepted(cuda):
    # the same weights through the C ABI: scales in the plain [rows, K/16] layout get a non-OK
    # status before any launch; converted once to the block layout they give the block's result
    import latent_mixture_experts_router_gb300 as lm
    w = workloads.Workload("fp4_layout", T=20, D=256, L=256, E=4, I=256, k=2, weights="nvfp4")
    inp = workloads.make_inputs(w, cuda)
    out_ref, _, blk, cfg = run(inp)
    ws = torch.zeros(lm.lmoe_workspace_size(cfg), dtype=torch.uint8, device=cuda)
    args = lambda W: (cfg, inp.x, inp.W_router, W["W_pool"], inp.g_pool, W["W_gate"], W["W_up"],  # noqa: E731
                      W["W_down"], inp.g_expert, W["W_unpool"], inp.g_pre, inp.g_post, w.k)
    raw = {n: getattr(inp, n) for n in ("W_pool", "W_gate", "W_up", "W_down", "W_unpool")}
    out = torch.full_like(out_ref, 7.0)
    with pytest.raises(lm.LmoeError) as ei:
        lm.latent_moe_forward(*args(raw), out, ws)
    assert ei.value.status == -2
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())              # nothing was written
    lm.latent_moe_forward(*args(blk.W), out, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, out_ref)
