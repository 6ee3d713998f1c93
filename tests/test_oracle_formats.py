"""Pins for the oracle's number formats (E2M1, E4M3, NVFP4 packing, activation rule).

Each test checks the oracle against something other than itself: the format
definitions written out as closed-form value lists, torch's float8_e4m3fn
decoder (a library routine), and exhaustive midpoint / saturation cases.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F


def test_e2m1_table_closed_form():
    # E2M1 magnitudes: 0, 0.5 (subnormal), then (1 + m/2) * 2^(e-1) for e = 1..3
    assert list(F.E2M1_TABLE[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(F.E2M1_TABLE[8:]) == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e4m3_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.E4M3_TABLE
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all() and nan.sum() == 2          # 0x7F and 0xFF
    assert (ours[~nan] == ref[~nan]).all()
    assert np.nanmax(ours) == 448.0 and F.E4M3_TABLE[1] == 2.0 ** -9


def test_encode_decode_identity_on_all_codes():
    for c in range(16):
        v = F.E2M1_TABLE[c]
        if c == 8:   # -0 encodes with its sign bit
            assert F.e2m1_encode(np.array([-0.0]))[0] == 8
            continue
        assert F.e2m1_encode(np.array([v]))[0] == c
    for c in range(256):
        v = F.E4M3_TABLE[c]
        if np.isnan(v) or c == 0x80:
            continue
        assert F.e4m3_encode(np.array([v]))[0] == c, c


@pytest.mark.parametrize("table,enc,n", [(F.E2M1_TABLE, F.e2m1_encode, 8),
                                          (F.E4M3_TABLE, F.e4m3_encode, 127)])
def test_rne_midpoints_and_neighbours(table, enc, n):
    pos = table[:n]
    for i in range(n - 1):
        a, b = pos[i], pos[i + 1]
        mid = (a + b) / 2
        even = i if i % 2 == 0 else i + 1
        assert enc(np.array([mid]))[0] == even
        assert enc(np.array([-mid]))[0] == even | (8 if n == 8 else 0x80)
        assert enc(np.array([np.nextafter(mid, 0)]))[0] == i
        assert enc(np.array([np.nextafter(mid, np.inf)]))[0] == i + 1


def test_saturation():
    assert F.E2M1_TABLE[F.e2m1_encode(np.array([6.0, 7.0, 1e30, -1e30]))].tolist() == [6, 6, 6, -6]
    assert F.E4M3_TABLE[F.e4m3_encode(np.array([448.0, 460.0, 1e9, -1e9]))].tolist() == [448, 448, 448, -448]


def test_e4m3_encode_matches_torch_in_range():
    # torch's fp32 -> float8_e4m3fn conversion rounds to nearest-even in range
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * 30, rng.uniform(-2 ** -6, 2 ** -6, 5000)])
    v = v[np.abs(v) < 448].astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = F.e4m3_encode(v)
    ok = (ours == ref) | ((ours & 0x7F) == 0) & ((ref & 0x7F) == 0)
    assert ok.all()


def test_nvfp4_unpack_low_nibble_first():
    codes = np.array([[0x21, 0xF7]], dtype=np.uint8)
    assert F.nvfp4_unpack_codes(codes).tolist() == [[1, 2, 7, 15]]
    deq = F.nvfp4_dequantize(np.tile(codes, (1, 4)), np.array([[0x38]], np.uint8), 2.0)  # block scale 1.0
    assert deq[0, :4].tolist() == [1.0, 2.0, 12.0, -12.0]


def test_activation_rule_representable_roundtrip():
    # rows built as e2m1 * e4m3 * s with the block max at magnitude 6 and the row max
    # block scale at 448 reproduce exactly
    rng = np.random.default_rng(2)
    q = rng.integers(0, 16, size=(4, 64))
    q[:, ::16] = 7                       # each block holds a 6
    sc = rng.integers(0x20, 0x60, size=(4, 4))
    sc[:, 0] = 0x7E                      # 448 in the first block of each row
    s = np.array([0.5, 1.0, 2.0 ** -7, 3.0])
    v = F.E2M1_TABLE[q] * np.repeat(F.E4M3_TABLE[sc], 16, axis=1) * s[:, None]
    q2, sc2, s2 = F.quantize_activation(v)
    assert np.array_equal(F.dequantize_activation(q2, sc2, s2), v)
    assert np.array_equal(s2, s.astype(np.float32))


def test_activation_rule_error_bound_and_zero_rows():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((16, 256)) * np.exp(rng.uniform(-8, 8, size=(16, 1)))
    v[3] = 0.0
    deq = F.fake_quantize_activation(v)
    amax_b = np.repeat(np.abs(v).reshape(16, 16, 16).max(axis=2), 16, axis=1)
    # one E2M1 step is at most 2 units of the block scale (~amax_b/6), plus E4M3 rounding
    assert (np.abs(deq - v) <= amax_b * (1.0 / 6.0) * (1 + 2 ** -3) + 1e-300).all()
    assert (deq[3] == 0).all()
    # scale-1 rows (the SwiGLU output between the expert GEMMs)
    deq1 = F.fake_quantize_activation(v / np.maximum(np.abs(v).max(axis=1, keepdims=True), 1e-30), row_scale=False)
    assert np.isfinite(deq1).all()


# ------------------------------------------------------------------ the rule vs its fp64 form
# The oracle applies the activation rule with each rounding decision in fp32 (the precision
# the kernels use).  Its plain definition (LMSYS Muse Spark Open post, "NVFP4 as a third MMA
# type": E2M1 values with one UE4M3 scale per 16 elements and an FP32 per-token scale) is, in
# exact arithmetic:
#     s  = amax(row) / (6 * 448)      sc = E4M3_RNE(amax(block) / (6 s))
#     q  = E2M1_RNE_sat(v / (sc * s)), q = 0 where sc = 0
# The fp32 sequence may differ from it only where the exact quotient lies within a few fp32
# rounding errors of an E4M3 or E2M1 rounding boundary.
_E2M1_MID = (F.E2M1_TABLE[:7] + F.E2M1_TABLE[1:8]) / 2
_E4M3_MID = (F.E4M3_TABLE[:126] + F.E4M3_TABLE[1:127]) / 2


def _near(a, mids, rel):
    a = np.abs(np.asarray(a, dtype=np.float64))
    d = np.min(np.abs(a[..., None] - mids), axis=-1)
    return d <= rel * np.maximum(a, 1e-300)


def _rule_fp64(v, row_scale):
    rows, K = v.shape
    amax = np.max(np.abs(v), axis=1)
    s = np.where(amax > 0, amax / (6.0 * 448.0), 1.0) if row_scale else np.ones(rows)
    blocks = v.reshape(rows, K // 16, 16)
    ratio = np.max(np.abs(blocks), axis=2) / (6.0 * s[:, None])
    sc = F.e4m3_encode(ratio)
    scv = F.E4M3_TABLE[sc]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(scv[:, :, None] > 0, blocks / (scv[:, :, None] * s[:, None, None]), 0.0)
    return F.e2m1_encode(t).reshape(rows, K), sc, s, ratio, t.reshape(rows, K)


@pytest.mark.parametrize("row_scale", [True, False])
def test_activation_rule_matches_its_fp64_definition(row_scale):
    rng = np.random.default_rng(7 + row_scale)
    rows, K = 512, 512
    v = rng.standard_normal((rows, K)) * np.exp2(rng.integers(-30, 30, size=(rows, 1)))
    v[::7, :16] *= 1e3            # outlier blocks: the row scale comes from them
    v[5] = 0.0
    v[9, 32:48] = 0.0
    if not row_scale:             # scale-1 rows (the SwiGLU output): keep the block scales in range
        v = v / np.max(np.abs(v), axis=1, keepdims=True).clip(1e-300) * rng.uniform(0.01, 2000, size=(rows, 1))
    v = v.astype(np.float32).astype(np.float64)   # both sides see the same fp32 inputs
    q, sc, s = F.quantize_activation(v, row_scale=row_scale)
    q64, sc64, s64, ratio, t = _rule_fp64(v, row_scale)
    # row scales: fp32 rounding of the exact quotient
    assert np.all(np.abs(s.astype(np.float64) - s64) <= 2.0 ** -24 * s64)
    # block scales: equal except within a few fp32 roundings of an E4M3 midpoint
    sc_diff = sc != sc64
    assert np.all(_near(ratio[sc_diff], _E4M3_MID, 1e-6)), ratio[sc_diff][:8]
    assert sc_diff.mean() < 1e-3
    # codes of blocks whose scale agrees: equal as values except near an E2M1 midpoint
    same_blk = np.repeat(~sc_diff, 16, axis=1)
    q_diff = (F.E2M1_TABLE[q] != F.E2M1_TABLE[q64]) & same_blk
    assert np.all(_near(t[q_diff], _E2M1_MID, 1e-6)), t[q_diff][:8]
    assert q_diff.mean() < 1e-4, q_diff.mean()
    # and the dequantised values agree to one E2M1 step where anything differs at all
    deq = F.dequantize_activation(q, sc, s)
    deq64 = F.E2M1_TABLE[q64] * np.repeat(F.E4M3_TABLE[sc64], 16, axis=1) * s64[:, None]
    amax_b = np.repeat(np.abs(v).reshape(rows, K // 16, 16).max(axis=2), 16, axis=1)
    assert np.all(np.abs(deq - deq64) <= amax_b / 3 + 1e-300)


@pytest.mark.parametrize("mistake", ["scale_without_row_scale", "multiplies_swapped_to_divide",
                                     "row_scale_6_only", "block_amax_over_4"])
def test_fp64_definition_sees_plausible_mistakes(mistake):
    # the comparison above is sharp enough to catch a plausible slip in the fp32 sequence
    rng = np.random.default_rng(11)
    rows, K = 64, 256
    v = (rng.standard_normal((rows, K)) * np.exp2(rng.integers(-20, 20, size=(rows, 1))))
    v = v.astype(np.float32).astype(np.float64)
    f32 = np.float32
    amax = np.max(np.abs(v), axis=1).astype(f32)
    s = (amax / f32(2688.0) if mistake != "row_scale_6_only" else amax / f32(6.0)).astype(f32)
    blocks = v.astype(f32).reshape(rows, K // 16, 16)
    amax_b = np.max(np.abs(blocks), axis=2)
    if mistake == "block_amax_over_4":
        amax_b = amax_b * f32(1.5)
    den = (f32(6.0) * s).astype(f32) if mistake != "scale_without_row_scale" else np.full(rows, f32(6.0))
    sc = F.e4m3_encode((amax_b / den[:, None]).astype(f32))
    scv = F.E4M3_TABLE[sc]
    r = np.where(scv > 0, 1.0 / np.where(scv > 0, scv, 1.0), 0.0).astype(f32)
    if mistake == "multiplies_swapped_to_divide":
        scaled = (blocks / r[:, :, None].clip(1e-30)).astype(f32) / s[:, None, None]
    else:
        scaled = (blocks * r[:, :, None]).astype(f32) * (f32(1.0) / s)[:, None, None]
    q_bad = F.e2m1_encode(scaled.astype(f32)).reshape(rows, K)
    q64, sc64, *_ = _rule_fp64(v, True)
    differs = (F.E2M1_TABLE[q_bad] != F.E2M1_TABLE[q64]).mean() + (sc != sc64).mean()
    assert differs > 1e-2, (mistake, differs)


def test_quantize_weight_roundtrip_and_bound():
    # weights built as e2m1 * e4m3 * s (the largest block scale 448 and a 6 in that block)
    # come back exactly; Gaussian weights spread over 2^-20..1 land within half an E2M1 step
    # of the block scale, and their block scales reach the E4M3 subnormals
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, size=(8, 64))
    q[:, ::16] = 7
    sc = rng.integers(0x08, 0x7E, size=(8, 4))
    sc[0, 0] = 0x7E
    s = np.float32(2.0 ** -10)
    W = F.E2M1_TABLE[q] * np.repeat(F.E4M3_TABLE[sc], 16, axis=1) * float(s)
    codes, sc2, s2 = F.quantize_weight(W)
    assert s2 == s and np.array_equal(F.nvfp4_dequantize(codes, sc2, s2), W)
    G = rng.standard_normal((256, 256)) * np.exp2(-rng.uniform(0, 20, size=(256, 1)))
    codes, sc3, s3 = F.quantize_weight(G)
    deq = F.nvfp4_dequantize(codes, sc3, s3)
    unit = np.repeat(F.E4M3_TABLE[sc3], 16, axis=1) * float(s3)
    inside = np.abs(G) <= 6 * unit
    # in range: at most half of the largest E2M1 step (2 units); beyond 6 units (the block
    # scale rounded down): saturated at 6 units with the sign kept
    assert np.all(np.abs(deq - G)[inside] <= 1.0 * unit[inside] + 1e-300)
    assert np.array_equal(deq[~inside], np.sign(G[~inside]) * 6 * unit[~inside])
    assert np.any((sc3 & 0x78) == 0) and np.any(sc3 >= 0x70)  # subnormal and large scales


def test_bf16_round_matches_torch_and_ties_to_even():
    # fp32-representable inputs: torch's float32 -> bfloat16 conversion (round to nearest even)
    rng = np.random.default_rng(9)
    v = (rng.standard_normal(200_000) * np.exp2(rng.integers(-60, 60, 200_000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.bf16_round(v.astype(np.float64)), ref)
    # exact halfway cases go to the even significand; one ulp either side goes the near way
    one = 1.0 + 2.0 ** -8                 # halfway between 1 and 1 + 2^-7
    assert F.bf16_round(np.array([one, 1.0 + 3 * 2.0 ** -8, -one]))[[0, 1, 2]].tolist() == \
        [1.0, 1.0 + 2 * 2.0 ** -7, -1.0]
    assert F.bf16_round(np.array([np.nextafter(one, 2.0)]))[0] == 1.0 + 2.0 ** -7
    assert F.bf16_round(np.array([0.0, -0.0]))[1] == 0.0


def _clean_row(rng, blocks=4):
    # a row whose blocks hold a 6 (block max) and whose first block scale is 448: Q(v) = v
    q = rng.integers(0, 16, size=(blocks * 16,))
    q[::16] = 7
    sc = rng.integers(0x30, 0x50, size=(blocks,))
    sc[0] = 0x7E
    return F.E2M1_TABLE[q] * np.repeat(F.E4M3_TABLE[sc], 16) * 0.25, sc


def test_activation_choices_far_from_boundaries_is_the_rule():
    rng = np.random.default_rng(12)
    for _ in range(20):
        v = rng.standard_normal(256) * np.exp2(rng.uniform(-10, 10))
        ch = F.activation_choices(v)
        assert len(ch) == 1 and np.array_equal(ch[0], F.fake_quantize_activation(v[None])[0])


@pytest.mark.parametrize("rel,expect", [(1e-7, 2), (-1e-7, 2), (1e-3, 1)])
def test_activation_choices_flip_one_element_at_an_e2m1_midpoint(rel, expect):
    rng = np.random.default_rng(13)
    v, sc = _clean_row(rng)
    unit = F.E4M3_TABLE[sc[1]] * 0.25             # block 1's scale unit (row scale 0.25 exactly)
    v[16 + 5] = 1.25 * unit * (1 + rel)           # between 1 and 1.5, just off the midpoint
    ch = F.activation_choices(v)
    assert len(ch) == expect
    assert np.array_equal(ch[0], F.fake_quantize_activation(v[None])[0])
    if expect == 2:
        d = np.nonzero(ch[1] != ch[0])[0]
        assert d.tolist() == [21] and abs(abs(ch[1][21] - ch[0][21]) - 0.5 * unit) < 1e-12 * unit
        assert {ch[0][21], ch[1][21]} == {unit, 1.5 * unit}


def test_activation_choices_flip_one_block_scale_at_an_e4m3_midpoint():
    rng = np.random.default_rng(14)
    v, sc = _clean_row(rng)
    s = 0.25
    lo, hi = F.E4M3_TABLE[0x44], F.E4M3_TABLE[0x45]
    ratio = (lo + hi) / 2 * (1 + 1e-8)            # block 2's amax / (6 s), just above a midpoint
    v[32:48] = v[32:48] / np.max(np.abs(v[32:48])) * ratio * 6 * s
    ch = F.activation_choices(v)
    assert len(ch) == 2
    diff_blocks = sorted({int(i) // 16 for i in np.nonzero(ch[1] != ch[0])[0]})
    assert diff_blocks == [2]
    # the two scales are the midpoint's neighbours: block max at 6 units of one or the other
    m0, m1 = np.max(np.abs(ch[0][32:48])), np.max(np.abs(ch[1][32:48]))
    assert sorted([m0, m1]) == pytest.approx(sorted([6 * lo * s, 6 * hi * s]), rel=0, abs=1e-12)
