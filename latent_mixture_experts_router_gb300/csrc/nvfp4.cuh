// nvfp4.cuh — NVFP4 (E2M1 values, one E4M3 scale per 16 elements, one fp32 row scale)
// quantisation on the device.
//
// Format: LMSYS "SGLang and Miles Add Day-0 Support for Muse Spark Open", section "NVFP4 as
// a third MMA type" (dense FP4 operands, UE4M3 scale per 16 elements, per-token FP32 input
// scale); the scale -> reciprocal step uses a 256-entry table indexed by the scale byte
// (section "NVFP4 requant reciprocal table").
//
// Activation rule, every rounding decision in fp32 and in this order:
//   s     = amax(row) / 2688                  (2688 = 6 * 448; s = 1 for a zero row, and
//                                              s = 1 for rows quantised without a row scale)
//   sc_b  = E4M3_rn_satfinite( amax(block) / (6 * s) )
//   r_b   = table[sc_b] = fp32(1 / value(sc_b))   (0 for sc_b = 0)
//   q_i   = E2M1_rn_satfinite( (v_i * r_b) * (1 / s) )
// Codes are packed two per byte, the even element in the low nibble.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace lmoe {

// ---- E4M3 reciprocal table, computed at compile time from the format definition
struct E4M3RecipTable {
  float v[256];
  static constexpr double pow2(int e) {
    double r = 1.0;
    if (e >= 0)
      for (int i = 0; i < e; ++i) r *= 2.0;
    else
      for (int i = 0; i < -e; ++i) r *= 0.5;
    return r;
  }
  static constexpr double value(int code) {  // magnitude of an E4M3(fn) code (sign ignored)
    const int e = (code >> 3) & 15, m = code & 7;
    return e == 0 ? (m / 8.0) * pow2(-6) : (1.0 + m / 8.0) * pow2(e - 7);
  }
  constexpr E4M3RecipTable() : v() {
    for (int c = 0; c < 256; ++c) {
      const int mag = c & 0x7F;
      v[c] = (mag == 0 || mag == 0x7F) ? 0.f : static_cast<float>(1.0 / value(mag));
    }
  }
};

// The table lives in global memory of each translation unit that includes this header: kernels
// copy it to shared memory with one coalesced load per thread (constant memory would serialise
// the 32 distinct addresses of each warp's load).
static __device__ const E4M3RecipTable g_e4m3_recip = E4M3RecipTable();

// ---- hardware conversions (round to nearest even, saturate to the largest finite)
// one byte holding E2M1(hi) in the high nibble and E2M1(lo) in the low nibble
LMOE_DEV uint32_t cvt_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}
// E4M3 code of one value
LMOE_DEV uint32_t cvt_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(v));
  return r & 0xFFu;
}

// ---- block layout of the E4M3 scales (the layout the block-scaled MMA reads through
// tcgen05.cp 32x128b): the scales of a [rows, K] matrix are stored as 512-byte blocks of
// 128 rows x 64 K, ordered [row block][K/64]; inside a block, row m = m0 + 32*m1 and 16-wide
// sub-block kk land at byte 16*m0 + 4*m1 + kk.  A stage of K = 256 of one row block is then
// 2 KB contiguous.
LMOE_DEV size_t blocked_sf_offset(long long blk, int m, int kb16, int K) {
  return (static_cast<size_t>(blk) * (K / 64) + (kb16 >> 2)) * 512 + (m & 31) * 16 + (m >> 5) * 4 +
         (kb16 & 3);
}

// Row scale of the rule: s = amax / 2688 (1 for an all-zero row).
LMOE_DEV float nvfp4_row_scale(float amax) { return amax > 0.f ? __fdiv_rn(amax, 2688.f) : 1.f; }

// Quantises 16 consecutive values with row scale s (six_s = fp32(6 s), inv_s = fp32(1/s)).
// Returns the E4M3 block-scale code; `codes` receives the 8 packed bytes (element 2i in
// the low nibble of byte i).
LMOE_DEV uint32_t nvfp4_quant16(const float (&v)[16], float six_s, float inv_s, const float* recip,
                                uint2& codes) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t sc = cvt_e4m3(__fdiv_rn(amax, six_s));
  const float r = recip[sc];
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a = __fmul_rn(__fmul_rn(v[2 * i], r), inv_s);
    const float b = __fmul_rn(__fmul_rn(v[2 * i + 1], r), inv_s);
    w[i >> 2] |= cvt_e2m1x2(b, a) << (8 * (i & 3));
  }
  codes = make_uint2(w[0], w[1]);
  return sc;
}

}  // namespace lmoe
