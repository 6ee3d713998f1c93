"""Number formats of the NVFP4 path, written from their definitions (oracle).

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU baseline, never by the library.

NVFP4 is dense FP4 (E2M1) with one unsigned E4M3 scale per 16 consecutive
elements, plus an fp32 second-level scale (LMSYS "SGLang and Miles Add Day-0
Support for Muse Spark Open", section "NVFP4 as a third MMA type").

* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
  0, 0.5, 1, 1.5, 2, 3, 4, 6; no inf/NaN.
* E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
  subnormals m/8 * 2^-6; S.1111.111 is NaN, so the largest finite is 448.

Encoders round to nearest with ties to the even code and saturate to the
largest finite magnitude.  They are a literal search over the code table, so
a reader can check them against the definition by eye.
"""
from __future__ import annotations

import numpy as np


def e2m1_value(code: int) -> float:
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = m * 0.5 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


def e4m3_value(code: int) -> float:
    s, e, m = (code >> 7) & 1, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)

# positive magnitudes in code order (codes 0..7 for E2M1, 0..126 for E4M3)
_E2M1_POS = E2M1_TABLE[:8]
_E4M3_POS = E4M3_TABLE[:127]


def _rne_sat_index(a: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """Index of the nearest magnitude in ascending ``pos`` to each a >= 0; ties to the even
    index; above the largest magnitude -> the largest (saturation)."""
    a = np.asarray(a, dtype=np.float64)
    hi = np.searchsorted(pos, a, side="left")          # pos[hi-1] < a <= pos[hi]
    hi = np.clip(hi, 0, len(pos) - 1)
    lo = np.clip(hi - 1, 0, len(pos) - 1)
    d_lo = a - pos[lo]
    d_hi = pos[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(a >= pos[-1], len(pos) - 1, idx)
    idx = np.where(a <= 0.0, 0, idx)
    return idx


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """fp -> E2M1 code (uint8 in 0..15), RNE, saturating at +-6; the sign bit follows the input."""
    v = np.asarray(v, dtype=np.float64)
    mag = _rne_sat_index(np.abs(v), _E2M1_POS)
    return (mag | (np.signbit(v).astype(np.int64) << 3)).astype(np.uint8)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """fp -> E4M3(fn) code, RNE, saturating at +-448 (never NaN for finite input)."""
    v = np.asarray(v, dtype=np.float64)
    mag = _rne_sat_index(np.abs(v), _E4M3_POS)
    return (mag | (np.signbit(v).astype(np.int64) << 7)).astype(np.uint8)


def nvfp4_unpack_codes(codes: np.ndarray) -> np.ndarray:
    """[.., K/2] bytes -> [.., K] E2M1 codes; the low nibble holds the even element."""
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = codes & 0xF
    out[..., 1::2] = codes >> 4
    return out


def nvfp4_dequantize(codes: np.ndarray, scales: np.ndarray, tensor_scale: float) -> np.ndarray:
    """Packed NVFP4 [rows, K/2] + E4M3 block scales [rows, K/16] + fp32 scale -> fp64 [rows, K]:
    value = e2m1(code) * e4m3(block scale) * tensor_scale."""
    q = E2M1_TABLE[nvfp4_unpack_codes(codes)]
    sc = E4M3_TABLE[np.asarray(scales, dtype=np.uint8)]
    return q * np.repeat(sc, 16, axis=-1) * float(tensor_scale)


# ------------------------------------------------------------------ bf16
def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 value (8 significant bits, ties to even), in fp64.
    bfloat16 keeps fp32's exponent range; the values rounded here (expert outputs) lie far
    inside it, so only the significand is rounded: v = m * 2^e with m in [0.5, 1), and m is
    rounded to a multiple of 2^-8 (numpy's rint rounds halves to even)."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


# ------------------------------------------------------------------ activations
# The activation rule (one fp32 scale per row, an E4M3 scale per 16-block,
# E2M1 codes) takes each rounding decision in fp32, the precision of the
# kernels that apply it, in this order:
#   s     = amax(row) / 2688                 (2688 = 6 * 448; s = 1 for a zero row,
#                                             and s = 1 where the row has no own scale)
#   sc_b  = E4M3( amax(block) / (6 * s) )
#   r_b   = fp32(1 / value(sc_b))            (0 where sc_b = 0)
#   q_i   = E2M1( (v_i * r_b) * (1 / s) )
# and the dequantised value is q_i * sc_b * s.
_F = np.float32


def quantize_activation(v: np.ndarray, row_scale: bool = True):
    """Rows of ``v`` -> (E2M1 codes [rows, K], E4M3 scale codes [rows, K/16], s fp32 [rows])."""
    v32 = np.asarray(v, dtype=np.float64).astype(_F)
    rows, K = v32.shape
    assert K % 16 == 0
    amax = np.max(np.abs(v32), axis=1)
    if row_scale:
        s = np.where(amax > 0, amax / _F(2688.0), _F(1.0)).astype(_F)
    else:
        s = np.ones(rows, dtype=_F)
    six_s = (_F(6.0) * s).astype(_F)
    inv_s = (_F(1.0) / s).astype(_F)
    blocks = v32.reshape(rows, K // 16, 16)
    amax_b = np.max(np.abs(blocks), axis=2)
    sc_code = e4m3_encode((amax_b / six_s[:, None]).astype(_F))
    sc_val = E4M3_TABLE[sc_code]
    r = np.where(sc_val > 0, (1.0 / np.where(sc_val > 0, sc_val, 1.0)), 0.0).astype(_F)
    scaled = ((blocks * r[:, :, None]).astype(_F) * inv_s[:, None, None]).astype(_F)
    q = e2m1_encode(scaled).reshape(rows, K)
    return q, sc_code, s


def dequantize_activation(q: np.ndarray, sc_code: np.ndarray, s: np.ndarray) -> np.ndarray:
    rows, K = q.shape
    return E2M1_TABLE[q] * np.repeat(E4M3_TABLE[sc_code], 16, axis=1) * np.asarray(s, np.float64)[:, None]


def fake_quantize_activation(v: np.ndarray, row_scale: bool = True) -> np.ndarray:
    """Q(v): the fp64 value the NVFP4 GEMM sees in place of the activation rows v."""
    return dequantize_activation(*quantize_activation(v, row_scale))


# ------------------------------------------------------------------ weights
def quantize_weight(W: np.ndarray):
    """Dense weight rows [rows, K] -> packed NVFP4 (codes [rows, K/2] u8, low nibble = even k;
    E4M3 block-scale codes [rows, K/16]; fp32 tensor scale), by the plain definition in fp64:
        s  = fp32(amax(W) / (6 * 448))          one second-level scale for the matrix
        sc = E4M3_RNE(amax(block) / (6 s))      one scale per 16 consecutive k
        q  = E2M1_RNE_sat(w / (sc s))           (q = 0 where sc = 0)
    (LMSYS Muse Spark Open post, "NVFP4 as a third MMA type": E2M1 values, a UE4M3 scale per
    16 elements, an FP32 tensor-level scale).  Used to pack test weights drawn from a Gaussian."""
    W = np.asarray(W, dtype=np.float64)
    rows, K = W.shape
    assert K % 16 == 0
    amax = float(np.max(np.abs(W)))
    s = float(np.float32(amax / 2688.0)) if amax > 0 else 1.0
    blocks = W.reshape(rows, K // 16, 16)
    sc = e4m3_encode(np.max(np.abs(blocks), axis=2) / (6.0 * s))
    scv = E4M3_TABLE[sc]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(scv[:, :, None] > 0, blocks / (scv[:, :, None] * s), 0.0)
    q = e2m1_encode(t).reshape(rows, K)
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return codes, sc, np.float32(s)


# ------------------------------------------------------------------ near-boundary decisions
# The activation rule rounds in fp32.  The GPU and the oracle feed it values computed in
# different orders (fp32 sums on the GPU, fp64 here), which agree to ~1e-7 relative; where
# the exact value lies that close to an E4M3 or E2M1 rounding boundary, either side of the
# boundary is a legitimate result of the rule, as either expert is at a top-k near tie.
QUANT_BAND = 1e-5   # relative distance to a rounding boundary treated as undecided


def _other_neighbour(code_mag: int, a: float, pos: np.ndarray) -> int:
    """The magnitude index on the other side of a's rounding boundary from code_mag."""
    if a >= pos[code_mag]:
        return min(code_mag + 1, len(pos) - 1)
    return max(code_mag - 1, 0)


def _rule_row(v32: np.ndarray, row_scale: bool, sc_override=None, code_override=None):
    """The rule on one fp32 row (same fp32 steps as quantize_activation), optionally with some
    block-scale codes (dict block -> E4M3 code) or element codes (dict i -> E2M1 code) forced.
    Returns the dequantised fp64 row."""
    K = v32.shape[0]
    amax = np.max(np.abs(v32))
    s = (amax / _F(2688.0)).astype(_F) if (row_scale and amax > 0) else _F(1.0)
    six_s, inv_s = _F(_F(6.0) * s), _F(_F(1.0) / s)
    blocks = v32.reshape(K // 16, 16)
    sc = e4m3_encode((np.max(np.abs(blocks), axis=1) / six_s).astype(_F))
    for b, c in (sc_override or {}).items():
        sc[b] = c
    scv = E4M3_TABLE[sc]
    r = np.where(scv > 0, 1.0 / np.where(scv > 0, scv, 1.0), 0.0).astype(_F)
    q = e2m1_encode(((blocks * r[:, None]).astype(_F) * inv_s).astype(_F)).reshape(K)
    for i, c in (code_override or {}).items():
        q[i] = c
    return E2M1_TABLE[q] * np.repeat(scv, 16) * float(s)


def activation_choices(v: np.ndarray, row_scale: bool = True, band: float = QUANT_BAND, max_choices: int = 8):
    """Q(v) of one row, followed by the rows obtained by taking one near-boundary rounding
    decision the other way: a block scale whose exact ratio amax_b / (6 s) lies within `band`
    (relative) of an E4M3 midpoint, or an element whose exact v / (sc s) lies within `band` of
    an E2M1 midpoint (one decision per variant; at most max_choices - 1 variants, nearest
    first).  Exactness here means fp64 on the oracle's own values."""
    v = np.asarray(v, dtype=np.float64)
    v32 = v.astype(_F)
    K = v.shape[0]
    base = _rule_row(v32, row_scale)
    amax = float(np.max(np.abs(v)))
    s64 = amax / 2688.0 if (row_scale and amax > 0) else 1.0
    blocks = v.reshape(K // 16, 16)
    ratio = np.max(np.abs(blocks), axis=1) / (6.0 * s64)
    sc = e4m3_encode(ratio.astype(_F))
    cand = []   # (relative distance, kind, index, code)
    mid4 = (_E4M3_POS[:-1] + _E4M3_POS[1:]) / 2
    for b in range(K // 16):
        if ratio[b] <= 0:
            continue
        d = np.min(np.abs(mid4 - ratio[b])) / ratio[b]
        if d <= band:
            alt = _other_neighbour(int(sc[b] & 0x7F), ratio[b], _E4M3_POS)
            cand.append((d, "sc", b, alt))
    mid2 = (_E2M1_POS[:-1] + _E2M1_POS[1:]) / 2
    scv = E4M3_TABLE[sc]
    for i in range(K):
        if scv[i // 16] <= 0:
            continue
        t = abs(v[i]) / (scv[i // 16] * s64)
        if t <= 0 or t >= _E2M1_POS[-1]:
            continue
        d = np.min(np.abs(mid2 - t)) / t
        if d <= band:
            q0 = int(e2m1_encode(np.array([t]))[0] & 7)
            alt = _other_neighbour(q0, t, _E2M1_POS) | (8 if np.signbit(v[i]) else 0)
            cand.append((d, "q", i, alt))
    out = [base]
    for d, kind, i, code in sorted(cand)[:max_choices - 1]:
        if kind == "sc":
            out.append(_rule_row(v32, row_scale, sc_override={i: code}))
        else:
            out.append(_rule_row(v32, row_scale, code_override={i: code}))
    return out
