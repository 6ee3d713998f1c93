"""The seeded input generator and the workload shapes.

Shapes are pinned to the weight budget the vLLM day-0 post prints for Muse
Spark Open (golden fixture tests/golden/weight_budget.json).
"""
import json
import math
import os

import numpy as np
import torch

import workloads
from workloads import rng

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "weight_budget.json")


def test_hash_tensor_path_matches_pure_python():
    idx = torch.tensor([0, 1, 2, 12345, (1 << 40) - 1], dtype=torch.int64)
    for seed, stream in ((0, 0), (0, 7), (3, 65535)):
        h = rng.hash64(seed, stream, idx)
        for i, v in zip(idx.tolist(), h.tolist()):
            assert (v & ((1 << 64) - 1)) == rng.hash64_int(seed, stream, i)


def test_splitmix64_known_value():
    # First output of SplitMix64 seeded with 0: mix(0 + golden gamma) = 0xE220A8397B1DCDAF
    assert rng.mix64_int(0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF


def test_normal_moments_and_slicing():
    z = rng.normal(0, 3, 0, 400_000, 2.0)
    assert abs(float(z.mean())) < 0.01 and abs(float(z.std()) - 2.0) < 0.01
    part = rng.normal(0, 3, 1000, 500, 2.0)
    assert torch.equal(part, z[1000:1500])


def test_expert_slice_equals_full_tensor():
    w = workloads.WORKLOADS["tiny_fp32"]
    full = workloads.dense_weight(w, "W_down")
    for e in (0, 7, 15):
        assert torch.equal(full[e], workloads.dense_weight(w, "W_down", expert=e))
    x = workloads.x_tensor(w)
    assert torch.equal(workloads.x_tensor(w, rows=[3, 60]), x[[3, 60]])


def test_nvfp4_weights_have_target_std_and_layout():
    w = workloads.WORKLOADS["prefill_nvfp4"]
    codes, scales, s = workloads.nvfp4_weight(w, "W_down", expert=3)
    assert codes.shape == (w.L, w.I // 2) and scales.shape == (w.L, w.I // 16)
    from oracle import formats
    deq = formats.nvfp4_dequantize(codes[:256].numpy(), scales[:256].numpy(), float(s[0]))
    assert abs(deq.std() * math.sqrt(w.I) - 1.0) < 0.02 and abs(deq.mean()) < 1e-3 / math.sqrt(w.I) * 50


def test_forced_routing_structure():
    for T in workloads.DECODE_SWEEP_T:
        w = workloads.WORKLOADS["decode_nvfp4_hot"].with_tokens(T)
        f = workloads.forced_routing(w)
        hot = workloads.hot_experts(w)
        assert f.shape == (T, w.k)
        for t in range(T):
            assert len(set(f[t].tolist())) == w.k       # k distinct experts per token
        for e in hot:
            assert int((f == e).sum()) == (T + 1) // 2  # each hot expert takes ceil(T/2) tokens


def test_zipf_bias_is_zipf():
    w = workloads.WORKLOADS["prefill_bf16_zipf"]
    b = workloads.zipf_bias(w).double().numpy()
    r = np.sort(-b)            # -b sorted ascending = s * ln(rank)
    assert np.allclose(r, w.zipf_s * np.log(np.arange(1, w.E + 1)), atol=1e-5)


def test_shapes_match_published_weight_budget():
    g = json.load(open(GOLDEN))
    w = workloads.WORKLOADS["decode_bf16"]
    layers = g["layers"]
    experts = 3 * w.L * w.I * w.E * layers / 1e9
    latent = 2 * w.D * w.L * layers / 1e9
    assert abs(experts - g["experts_total_B"]) < 0.5 * 1            # 798.9 vs "799 B"
    assert abs(latent - g["moe_latent_projections_B"]) < 0.05       # 4.16 vs "4.2 B"
    assert (w.L, w.D) == (g["pooler_rows"], g["pooler_cols"])
    assert w.E == g["experts_per_layer"]
    # active parameters with top-8: experts + latent + router per layer, plus attention
    active = layers * (w.k * 3 * w.L * w.I + 2 * w.D * w.L + w.E * w.D) / 1e9 + g["attention_B"]
    assert abs(active - g["active_B"]) < 1.0


def test_gaussian_is_standard_normal():
    # x and the gammas: Box-Muller deviates checked against scipy's normal distribution
    # (Kolmogorov-Smirnov), its fourth moment and its tails (which an Irwin-Hall sum lacks)
    import scipy.stats as st
    z = rng.gaussian(0, 1, 0, 1_000_000, 1.0).numpy()
    assert abs(z.mean()) < 3e-3 and abs(z.std() - 1.0) < 3e-3
    assert abs(st.kurtosis(z, fisher=False) - 3.0) < 0.03
    tail = np.mean(np.abs(z) > 3.5)
    assert abs(tail - 2 * st.norm.sf(3.5)) < 1.5e-4            # 4.65e-4 expected
    assert st.kstest(z[:200_000], "norm").pvalue > 1e-3
    part = rng.gaussian(0, 1, 5000, 100, 2.0)
    assert torch.equal(part, 2.0 * rng.gaussian(0, 1, 0, 6000, 1.0)[5000:5100])


def test_x_rows_of_one_long_sequence():
    w = workloads.WORKLOADS["tiny_fp32"].with_tokens(6)
    x = workloads.x_tensor(w)
    assert torch.equal(workloads.x_tensor(w.with_tokens(3), first_token=3), x[3:6])
    assert torch.equal(workloads.x_tensor(w, rows=[5, 1]), x[[5, 1]])
