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
