// decode_mk.cu — the whole latent-MoE block for one token with NVFP4 weights, as one
// persistent kernel of one CTA per SM (or its parts before and after the expert GEMMs).
//
// At one token every contraction of the block is a matrix-vector product: each weight is used
// once, so the block is bound by streaming its packed weights (Muse Spark Open shape: router
// 4 MB bf16, pooler and unpooler 18 MB each, the k = 8 selected experts' gate/up 151 MB and
// down 75 MB, codes with their scales) and, as a chain of kernels, by their launch and
// pipeline latencies.  Here one CTA per SM runs the call in four weight phases separated by
// grid barriers, each spreading its weight rows evenly over all SMs:
//   P2  router (bf16 rows, fp32 xn) and pooler (NVFP4 rows, Q(xn))          barrier 1
//   P4  gate and up rows of the k experts, SwiGLU, h requantised (scale 1)   barrier 2
//   P5  down rows of the k experts: y (bf16)                                 barrier 3
//   P7  unpooler rows (Q(c))                                                 barrier 4
// and the row steps between them — pre-norm and Q(xn) (P1), top-k, softmax, pool norm and
// Q(h0) (P3), the per-expert norms, weighted sum and Q(c) (P6), post-norm and residual (P8) —
// run redundantly in every CTA (a row of at most 8192 values) in one fixed order, so all CTAs
// hold bit-identical copies without a barrier for them.
//
// Roles: lanes 0-3 of warp 15 stream the CTA's weight rows of all four phases, in order, as
// bulk copies into a ring of 30 shared-memory stages of 4 KB (an mbarrier per stage, full and
// empty); they run ahead across the grid barriers, waiting only for the top-k before the
// expert rows.
// Warps 0-14 take the row steps (a named barrier of their own) and the stages, stage q by warp
// q mod 15; a unit of rows that spans several stages (16 rows of h, of y) is finished by the
// warp that completes it.
//
// NVFP4 dot products (both operands E2M1 values with E4M3 block scales): the 16 products of a
// block are formed in f16 — an E2M1 x E2M1 product is a multiple of 0.25 of magnitude <= 36,
// so a chain of eight of them is exact in f16 — the two halves are added in fp32 (exact),
// multiplied by the product of the two block scales (exact in fp32) and accumulated in fp32
// over the blocks; the row's fp32 scales multiply the sum.  The activation rule Q and the
// bf16 rounding of y are those of the tensor-core path (nvfp4.cuh).  A lane takes pieces of 32
// codes (16 bytes) at lane, lane + 32, ... of each row; the activation is held in shared memory
// as f16 pairs, permuted so that a warp's loads of it are contiguous; the weight scales (one
// half word of the block layout per piece) are read from global memory one stage ahead.
//
// Every wait is bounded by the call's wait budget: a wait that runs past it sets
// kErrGridBarrier, and the CTA's other waits give up at once, so the call ends with
// LMOE_ERR_TIMEOUT instead of waiting forever; the producer lets its copies in flight land
// before it leaves.
//
// Launch: programmatic dependent launch, so the CTAs start on the SMs the previous kernel
// leaves and stream their weights while the consumers wait for that kernel (griddepcontrol);
// an ordinary grid of one CTA per SM, every CTA resident at once on a GPU the call has to
// itself, or, on request, a cooperative launch, which the driver starts only once all of them
// can be resident (measured 7.6 us slower per call: the grid cannot start on part of the SMs).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "internal.h"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace lmoe {

namespace {

constexpr int kMkThreads = 512;
constexpr int kMkCWarps = 15;                  // consumer warps
constexpr int kMkConsumers = kMkCWarps * 32;
constexpr int kMkProducerWarp = kMkCWarps;
constexpr int kMkMaxK = 8192;
constexpr int kMkStageBytes = 4096;
constexpr int kMkSlots = 2 * kMkCWarps;        // ring slots: w and w + 15 belong to consumer warp w
constexpr int kMkUnitSlots = 32;               // units in flight (each its 32 sums)
// rows of at most kMkMaxK values, as chunks of 8 spread over the consumers
constexpr int kRowChunks = (kMkMaxK / 8 + kMkConsumers - 1) / kMkConsumers;

// ---- small helpers
LMOE_DEV void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kMkConsumers) : "memory"); }

LMOE_DEV uint32_t ld_acquire_u32(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
LMOE_DEV uint32_t ldg_u16(const uint8_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
LMOE_DEV void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
// two E2M1 codes (one byte, element 2i in the low nibble) as an f16 pair (exact)
LMOE_DEV __half2 e2m1x2_to_h2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
  return *reinterpret_cast<__half2*>(&r);
}
// two E4M3 codes (the low 16 bits) as fp32 values (exact, through f16)
LMOE_DEV float2 e4m3x2_to_f2(uint32_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(two & 0xFFFFu)));
  return __half22float2(*reinterpret_cast<__half2*>(&r));
}
LMOE_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// sum (or max of non-negative values) over the consumer threads
LMOE_DEV float creduce(float v, float* red, bool is_max) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  const int wp = threadIdx.x >> 5, l = threadIdx.x & 31;
  csync();
  if (l == 0) red[wp] = v;
  csync();
  if (wp == 0) {
    float t = l < kMkCWarps ? red[l] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float w = __shfl_xor_sync(0xffffffffu, t, o);
      t = is_max ? fmaxf(t, w) : t + w;
    }
    if (l == 0) red[32] = t;
  }
  csync();
  return red[32];
}
// 8 consecutive fp32 values from global memory written by this kernel (read through L2)
LMOE_DEV void ldcg8(const float* p, float (&v)[8]) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
// 8 consecutive fp32 values of a kernel input
LMOE_DEV void ldg8(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
LMOE_DEV void bf16x8(const uint4 q, float (&v)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
LMOE_DEV void load_x8(const DecodeMkArgs& a, int i, float (&v)[8]) {
  if (a.x_f32) ldg8(static_cast<const float*>(a.x) + i, v);
  else bf16x8(__ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.x) + i)), v);
}
LMOE_DEV float load_x(const DecodeMkArgs& a, int i) {
  return a.x_f32 ? static_cast<const float*>(a.x)[i] : __bfloat162float(static_cast<const __nv_bfloat16*>(a.x)[i]);
}

// Bounded wait on an mbarrier phase.  A wait that runs past the budget marks the CTA dead
// (and the call failed); once dead, every wait of the CTA gives up at once.
LMOE_DEV bool mk_wait(uint64_t* bar, uint32_t parity, long long budget, volatile int* dead, unsigned* err) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(addr, parity, 1000)) {
    if (*dead) return false;
    if (clock64() - t0 > budget) {
      *dead = 1;
      atomicOr(err, kErrGridBarrier);
      return false;
    }
  }
  return true;
}

// Arrival of this CTA's consumers at grid barrier n (0-based) and the wait until every CTA has
// arrived.  False (error bit set, CTA dead) when the wait ran past the budget.
LMOE_DEV bool grid_barrier(const DecodeMkArgs& a, int n, volatile int* dead, int* s_flag) {
  csync();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(a.bar, 1u);
    const unsigned target = static_cast<unsigned>(n + 1) * gridDim.x;
    const long long t0 = clock64();
    int ok = 1;
    while (ld_acquire_u32(a.bar) < target) {
      if (clock64() - t0 > a.budget) {
        atomicOr(a.err, kErrGridBarrier);
        *dead = 1;
        ok = 0;
        break;
      }
      __nanosleep(20);
    }
    *s_flag = ok;
  }
  csync();
  return *s_flag != 0;
}

// ---- the activation operand in shared memory
// Store of one quantised 16-block b of a row of K codes as the dot products read it: piece
// p = b / 2 of 32 codes, its f16 pairs in parts 2 (b % 2) and 2 (b % 2) + 1 (part i of piece
// p at uint4 i * (K / 32) + p); the block's scale value at asc[b].
LMOE_DEV void put_block(uint4* act, float* asc, int np, int b, uint2 q, float sc) {
  const int p = b >> 1, hf = b & 1;
  uint32_t h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __half2 v = e2m1x2_to_h2(((i < 4 ? q.x : q.y) >> (8 * (i & 3))) & 0xFFu);
    h[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  act[(2 * hf) * np + p] = make_uint4(h[0], h[1], h[2], h[3]);
  act[(2 * hf + 1) * np + p] = make_uint4(h[4], h[5], h[6], h[7]);
  asc[b] = sc;
}

// Q of a row held in shared memory (fp32 v[K]) with the row scale of the rule, stored as the
// dot products read it; returns s.  With codes_out, the packed codes also go to codes_out
// [K/2] and the scale codes to the block-layout row (M tile blk_out, its row 0) of scales_out.
// Consumers only.
LMOE_DEV float quantize_row_smem(const float* v, int K, const float* recip, float* red, uint4* act, float* asc,
                                 uint8_t* codes_out = nullptr, uint8_t* scales_out = nullptr, int blk_out = 0) {
  const float4* v4 = reinterpret_cast<const float4*>(v);
  float amax = 0.f;
  for (int i = threadIdx.x; i < K / 4; i += kMkConsumers) {
    const float4 q = v4[i];
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(q.x), fabsf(q.y)), fmaxf(fabsf(q.z), fabsf(q.w))));
  }
  const float s = nvfp4_row_scale(creduce(amax, red, true));
  const float six_s = __fmul_rn(6.f, s), inv_s = __fdiv_rn(1.f, s);
  for (int b = threadIdx.x; b < K / 16; b += kMkConsumers) {
    float blk[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // 16-byte reads: a quarter of the bank conflicts of scalar ones
      const float4 q = v4[b * 4 + i];
      blk[4 * i] = q.x;
      blk[4 * i + 1] = q.y;
      blk[4 * i + 2] = q.z;
      blk[4 * i + 3] = q.w;
    }
    uint2 q;
    const uint32_t sc = nvfp4_quant16(blk, six_s, inv_s, recip, q);
    put_block(act, asc, K / 32, b, q, e4m3x2_to_f2(sc).x);
    if (codes_out != nullptr) {
      *reinterpret_cast<uint2*>(codes_out + b * 8) = q;
      scales_out[blocked_sf_offset(blk_out, 0, b, K)] = static_cast<uint8_t>(sc);
    }
  }
  csync();
  return s;
}

// ---- weight phases
// Rows per stage: 4 for K <= 2048, 2 for K <= 4096, 1 for K <= 8192 (4 KB of codes at most).
__host__ __device__ constexpr int stage_rows(int K) { return K <= 2048 ? 4 : K <= 4096 ? 2 : 1; }
// Parts of a router row (D bf16) streamed as stages of at most 4 KB: 1, 2 or 4.
__host__ __device__ constexpr int router_parts(int D) { return D <= 2048 ? 1 : D <= 4096 ? 2 : 4; }

// One stage's rows: where each lives (codes [rows, K/2], block-layout scales).
struct StageRows {
  const uint8_t* codes[4];
  const uint8_t* scales[4];
  int row[4];
};

// The CTA's share of a phase: units [u0, u1) (contiguous, balanced to one unit), each of gpu
// stages of nr rows; n: the CTA's stages.
struct PhaseShare {
  int K, nr, gpu, lg, u0, u1, n;   // lg = log2(gpu) (gpu is a power of two)
};
LMOE_DEV PhaseShare share_of(int n_units, int K, int rows_per_unit) {
  PhaseShare s;
  s.K = K;
  s.nr = stage_rows(K);
  s.gpu = rows_per_unit / s.nr;
  s.lg = __ffs(s.gpu) - 1;
  s.u0 = static_cast<int>(static_cast<long long>(n_units) * blockIdx.x / gridDim.x);
  s.u1 = static_cast<int>(static_cast<long long>(n_units) * (blockIdx.x + 1) / gridDim.x);
  s.n = (s.u1 - s.u0) * s.gpu;
  return s;
}

// The shares of the four phases (phase 0 holds the CTA's router row parts first, each one
// stage of 2 D / rp bytes of bf16, then its pooler stages); every role computes the same values.
struct Phases {
  PhaseShare ph[4];
  int rp, r0, r1;   // parts per router row; the CTA's router parts [r0, r1) (part u: row u / rp)
};
LMOE_DEV Phases phases_of(const DecodeMkArgs& a) {
  Phases P;
  P.rp = router_parts(a.D);
  P.r0 = static_cast<int>(static_cast<long long>(P.rp) * a.E * blockIdx.x / gridDim.x);
  P.r1 = static_cast<int>(static_cast<long long>(P.rp) * a.E * (blockIdx.x + 1) / gridDim.x);
  P.ph[0] = share_of(a.L / stage_rows(a.D), a.D, stage_rows(a.D));   // pooler: a unit is one stage
  P.ph[0].n += P.r1 - P.r0;
  P.ph[1] = share_of(a.k * (a.I / 16), a.L, 32);                     // 16 h rows: 16 gate + 16 up
  P.ph[2] = share_of(a.k * (a.L / 16), a.I, 16);                     // 16 y rows of one slot
  P.ph[3] = share_of(a.D / 4, a.L, 4);                               // 4 u rows
  return P;
}

// Rows of stage q of phase `ph` (q below the CTA's stage count): 32-bit index math, one
// division at most.  Phase 1 stages hold h rows r0 .. r0 + nr/2 - 1 as [gate rows][up rows].
LMOE_DEV StageRows stage_rows_of(const DecodeMkArgs& a, const Phases& P, int ph, int q, const int* s_idx) {
  StageRows g;
  const PhaseShare& S = P.ph[ph];
  if (ph == 0) {
    const int nr_rt = P.r1 - P.r0;
    if (q < nr_rt) {   // a part of a router row: D / rp bf16
      const int u = P.r0 + q;
      g.codes[0] = reinterpret_cast<const uint8_t*>(a.W_router) + static_cast<long long>(u) * (a.D / P.rp) * 2;
      g.scales[0] = nullptr;
      g.row[0] = 0;
      return g;
    }
    const int r0 = (S.u0 + (q - nr_rt)) * S.nr;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      g.codes[r] = a.w[0].codes;
      g.scales[r] = a.w[0].scales;
      g.row[r] = r0 + r;
    }
    return g;
  }
  const int u = S.u0 + (q >> S.lg), gi = q & (S.gpu - 1);
  if (ph == 1) {
    const int nb = a.I >> 4, j = u / nb, ib = u - j * nb;
    const int base = s_idx[j] * a.I + ib * 16 + gi * (S.nr / 2);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const bool up = r >= S.nr / 2;
      g.codes[r] = up ? a.w[2].codes : a.w[1].codes;
      g.scales[r] = up ? a.w[2].scales : a.w[1].scales;
      g.row[r] = base + (up ? r - S.nr / 2 : r);
    }
  } else if (ph == 2) {
    const int nl = a.L >> 4, j = u / nl;
    const int base = s_idx[j] * a.L + (u - j * nl) * 16 + gi * S.nr;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      g.codes[r] = a.w[3].codes;
      g.scales[r] = a.w[3].scales;
      g.row[r] = base + r;
    }
  } else {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      g.codes[r] = a.w[4].codes;
      g.scales[r] = a.w[4].scales;
      g.row[r] = u * 4 + gi * S.nr + r;
    }
  }
  return g;
}

// A lane's weight scales of a stage: per row, per piece, the two E4M3 codes of its blocks.  In
// the block layout, piece p of row m (pair of 16-blocks 2p, 2p+1) sits at
// (m / 128 * K / 64 + p / 2) * 512 + (m % 32) * 16 + (m % 128 / 32) * 4 + 2 (p % 2): a per-row
// base, a per-lane offset and 16 * 512 bytes per further 32 pieces.
template <int NR, int CPW>
LMOE_DEV void stage_scales(const StageRows& g, int K, int lane, uint32_t (&sc)[NR][CPW]) {
  const int np = K >> 5;
  const int lane_off = (lane >> 1) * 512 + 2 * (lane & 1);
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const int m = g.row[r];
    const uint8_t* base = g.scales[r] + static_cast<long long>(m >> 7) * (K / 64) * 512 + (m & 31) * 16 +
                          ((m >> 5) & 3) * 4 + lane_off;
#pragma unroll
    for (int c = 0; c < CPW; ++c) sc[r][c] = lane + 32 * c < np ? ldg_u16(base + c * 8192) : 0u;
  }
}

// The stage's NR rows (codes in shared memory) dotted with the activation; sums in every lane.
template <int NR, int CPW>
LMOE_DEV void stage_dot(const uint8_t* stage, int K, const uint4* act, const float* asc, const uint32_t (&sc)[NR][CPW],
                        int lane, float (&out)[NR]) {
  const int np = K >> 5;
  float acc[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) acc[r] = 0.f;
#pragma unroll
  for (int c = 0; c < CPW; ++c) {
    const int p = lane + 32 * c;
    if (p >= np) continue;
    const uint4 a0 = act[p], a1 = act[np + p], a2 = act[2 * np + p], a3 = act[3 * np + p];
    const float2 as = reinterpret_cast<const float2*>(asc)[p];
    const uint32_t av[16] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w,
                             a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const uint4 wq = *reinterpret_cast<const uint4*>(stage + r * (K / 2) + 16 * p);
      const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
      const float2 ws = e4m3x2_to_f2(sc[r][c]);
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {   // the piece's two blocks
        __half2 h = __float2half2_rn(0.f);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          h = __hfma2(e2m1x2_to_h2((wv[2 * hb + (i >> 2)] >> (8 * (i & 3))) & 0xFFu),
                      *reinterpret_cast<const __half2*>(&av[8 * hb + i]), h);
        const float2 f = __half22float2(h);
        acc[r] = fmaf(f.x + f.y, (hb ? ws.y : ws.x) * (hb ? as.y : as.x), acc[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) out[r] = warp_sum(acc[r]);
}

// Runs body(IntC<NR>, IntC<CPW>) for a row length K: rows per stage NR and pieces of 32 codes
// per lane CPW.
template <int V>
struct IntC {
  static constexpr int value = V;
};
template <class Body>
LMOE_DEV void with_shape(int K, Body&& body) {
  if (K <= 1024) body(IntC<4>{}, IntC<1>{});
  else if (K <= 2048) body(IntC<4>{}, IntC<2>{});
  else if (K <= 4096) body(IntC<2>{}, IntC<4>{});
  else body(IntC<1>{}, IntC<8>{});
}

// ---- top-k
// The top-k of the token by warp 0: the same selection, near-tie rule and weights as the
// block's top-k kernel (ties to the lower index, NaN ordered as -inf, softmax renormalised
// over the k, the k exponentials summed in selection order); forced ids are checked as there.
// Lane j holds the j-th selection.
LMOE_DEV void mk_topk(const DecodeMkArgs& a, float* vals, int* s_idx, float* s_w, int* s_nt) {
  const int lane = threadIdx.x & 31;
  const int E = a.E, k = a.k;
  int sel = 0;
  float sval = -INFINITY;
  int nt = 0;
  if (a.forced != nullptr) {
    int e = lane < k ? a.forced[lane] : 0;
    bool bad = lane < k && (e < 0 || e >= E);
    if (bad) e = 0;
    for (int i = 0; i < k; ++i) {   // a repeated id
      const int ei = __shfl_sync(0xffffffffu, e, i);
      bad = bad || (lane < k && i < lane && ei == e);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.err, kErrBadIndex);
    sel = e;
    sval = lane < k ? vals[e] : -INFINITY;
  } else {
    for (int i = lane; i < E; i += 32)
      if (vals[i] != vals[i]) vals[i] = -INFINITY;
    __syncwarp();
    const int rounds = k < E ? k + 1 : k;
    float kth = 0.f;
    for (int j = 0; j < rounds; ++j) {
      float best = -INFINITY;
      int bi = 0x7fffffff;
      for (int i = lane; i < E; i += 32) {
        const float v = vals[i];
        if (v != v) continue;   // taken
        if (bi == 0x7fffffff || v > best || (v == best && i < bi)) {
          best = v;
          bi = i;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > best || (ov == best && oi < bi)) {
          best = ov;
          bi = oi;
        }
      }
      if (j < k) {
        if (lane == j) {
          sel = bi;
          sval = best;
        }
        if (j == k - 1) kth = best;
        if (lane == 0) vals[bi] = __int_as_float(0x7fc00000);
        __syncwarp();
      } else if ((kth - best) < 1e-3f) {
        nt = 1;
      }
    }
  }
  // softmax over the k: max, then the exponentials summed in selection order
  float m = sval;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float ex = lane < k ? expf(sval - m) : 0.f;
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
  const float inv = 1.f / sum;
  if (lane < k) {
    s_idx[lane] = sel;
    s_w[lane] = ex * inv;
  }
  if (lane == 0) *s_nt = nt;
}

// This CTA's 1 KB pieces of [p, p + bytes) into L2 (bytes a multiple of 16).
LMOE_DEV void l2_prefetch_share(const void* p, uint32_t bytes) {
  for (uint32_t off = blockIdx.x * 1024u; off < bytes; off += gridDim.x * 1024u)
    prefetch_l2_bulk(static_cast<const uint8_t*>(p) + off, min(1024u, bytes - off));
}

// The scale blocks of rows [r0, r1) of a weight with K columns (block layout: 128 rows,
// K/64 pieces of 512 bytes) into L2.  The dot products read a stage's scales from global
// memory one stage ahead; from HBM each such read would stall its stage.  (A call repeated on
// one layer finds them in L2 already — they are read with the default policy, the codes
// evict-first — and runs no faster with this; in a model the other layers evict them.)
LMOE_DEV void l2_prefetch_scales(const uint8_t* scales, int r0, int r1, int K) {
  if (r1 <= r0) return;
  const uint32_t blk = static_cast<uint32_t>(K / 64) * 512u;
  for (int b = r0 >> 7; b <= (r1 - 1) >> 7; ++b)
    for (uint32_t off = 0; off < blk; off += 4096u)
      prefetch_l2_bulk(scales + static_cast<long long>(b) * blk + off, min(4096u, blk - off));
}

// ---- shared memory: [ring of stages][region A][recip][vals][unit sums][unit counters]; region
// A holds act, asc and row (phases P1-P4, P6-P8) or, in P5, every slot's Q(h) (hact, hsc)
__host__ __device__ inline size_t mk_region_a_bytes(int D, int L, int I, int k) {
  const size_t Kmax = static_cast<size_t>(D > L ? (D > I ? D : I) : (L > I ? L : I));
  const size_t act_row = Kmax * 2 + Kmax / 16 * 4 + Kmax * 4;
  const size_t hact = static_cast<size_t>(k) * I * 2 + static_cast<size_t>(k) * (I / 16) * 4;
  return act_row > hact ? act_row : hact;
}
__host__ __device__ inline size_t mk_fixed_bytes(int D, int L, int I, int E, int k) {
  return mk_region_a_bytes(D, L, I, k) + 256 * 4 + static_cast<size_t>((E + 3) / 4 * 4) * 4 + kMkUnitSlots * 32 * 4 +
         kMkUnitSlots * 4;
}
__host__ __device__ inline size_t mk_smem_bytes(int D, int L, int I, int E, int k) {
  return mk_fixed_bytes(D, L, I, E, k) + static_cast<size_t>(kMkSlots) * kMkStageBytes;
}

template <int MODE>
__global__ void __launch_bounds__(kMkThreads, 1) decode_megakernel(const DecodeMkArgs a) {
  extern __shared__ __align__(1024) uint8_t mk_smem[];
  const int D = a.D, L = a.L, I = a.I, E = a.E, k = a.k;
  const int Kmax = max(D, max(L, I));
  uint8_t* ring = mk_smem;
  uint8_t* reg_a = mk_smem + static_cast<size_t>(kMkSlots) * kMkStageBytes;
  uint4* act = reinterpret_cast<uint4*>(reg_a);                     // [Kmax / 8]
  float* asc = reinterpret_cast<float*>(act + Kmax / 8);            // [Kmax / 16]
  float* row = asc + Kmax / 16;                                     // [Kmax]
  uint4* hact = reinterpret_cast<uint4*>(reg_a);                    // [k][I / 8]   (P5 only)
  float* hsc = reinterpret_cast<float*>(hact + k * (I / 8));        // [k][I / 16]
  float* recip = reinterpret_cast<float*>(reg_a + mk_region_a_bytes(D, L, I, k));
  float* vals = recip + 256;
  float* part_all = vals + (E + 3) / 4 * 4;                         // [kMkUnitSlots][32]
  int* ucnt = reinterpret_cast<int*>(part_all + kMkUnitSlots * 32); // [kMkUnitSlots]
  __shared__ __align__(8) uint64_t full[kMkSlots], empty[kMkSlots], route_ready;
  __shared__ float red[33];
  __shared__ int s_flag, s_idx[16], s_row[16], s_nt;
  __shared__ volatile int s_dead;
  __shared__ int s_last_issue[kMkSlots];   // per ring slot, the stage last issued into it
  __shared__ float s_w[16], s_coef[16];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const long long budget = a.budget;

  if (tid == 0) {
    for (int s = 0; s < kMkSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&route_ready, 1);
    fence_mbar_init();
    // the gammas read later by every CTA into L2 now, a 1 KB piece per CTA, before the
    // weight stream fills the memory queues
    l2_prefetch_share(a.g_pool, static_cast<uint32_t>(L) * 4u);
    l2_prefetch_share(a.g_post, static_cast<uint32_t>(D) * 4u);
    s_dead = 0;
  }
  if (tid < kMkSlots) s_last_issue[tid] = -1;
  for (int i = tid; i < 256; i += kMkThreads) recip[i] = g_e4m3_recip.v[i];
  for (int i = tid; i < kMkUnitSlots; i += kMkThreads) ucnt[i] = 0;
  __syncthreads();   // the only CTA-wide barrier: the producer takes no part in the others
  const Phases P = phases_of(a);
  if (tid == 32) {   // the scales of this CTA's pooler and unpooler rows into L2 at once
    if (MODE != kDecodeMkPost) {
      const PhaseShare& S = P.ph[0];
      l2_prefetch_scales(a.w[0].scales, S.u0 * S.nr, S.u1 * S.nr, S.K);
    }
    if (MODE != kDecodeMkPre) {
      const PhaseShare& S = P.ph[3];
      l2_prefetch_scales(a.w[4].scales, S.u0 * 4, S.u1 * 4, S.K);
    }
  }

  if (warp == kMkProducerWarp) {
    // ---- producer: lanes 0-3 of warp 15 issue the CTA's stages of all four phases, four
    // consecutive stages per pass (stage q of a phase by lane q mod 4; one thread's issue rate
    // would bound the CTA's stream).  The lanes meet after every pass, so the stages are issued
    // in order, four at a time.  Stage g (counted over the phases) goes to slot g mod 30, the
    // (g / 30)-th use of the slot; slot s is consumed by warp s mod 15 alone, its uses in order,
    // so no wait on a slot's barrier can meet a phase two uses away.
    constexpr int kLanes = 4;
    if (lane < kLanes) {
      const uint64_t pol = policy_evict_first();
      int qbase_p = 0;
      // the weights depend on no earlier kernel: the stream starts at once, while the
      // consumers wait for the previous kernel (programmatic dependent launch)
      bool ok = true;
      const int ph0 = MODE == kDecodeMkPost ? 3 : 0, ph1 = MODE == kDecodeMkPre ? 0 : 3;
      for (int ph = ph0; ph <= ph1; ++ph) {
        if (ph == 1 && ok) ok = mk_wait(&route_ready, 0, budget, &s_dead, a.err);   // expert rows need the top-k
        const PhaseShare& S = P.ph[ph];
        const int nr_rt = ph == 0 ? P.r1 - P.r0 : 0, rb = S.K / 2;
        for (int q0 = 0; q0 < S.n; q0 += kLanes) {
          __syncwarp(0xFu);
          if (s_dead) ok = false;
          const int q = q0 + lane;
          if (!ok || q >= S.n) continue;
          const int qg = qbase_p + q, s = qg % kMkSlots;
          if (!mk_wait(&empty[s], (static_cast<uint32_t>(qg / kMkSlots) & 1u) ^ 1u, budget, &s_dead, a.err)) {
            ok = false;
            continue;
          }
          s_last_issue[s] = qg;
          uint8_t* dst = ring + s * kMkStageBytes;
          if (q < nr_rt) {   // a part of a router row: D / rp bf16
            const uint32_t rbytes = static_cast<uint32_t>(D / P.rp * 2);
            mbar_arrive_expect_tx(&full[s], rbytes);
            bulk_load_hint(dst, reinterpret_cast<const uint8_t*>(a.W_router) + static_cast<long long>(P.r0 + q) * rbytes,
                           rbytes, &full[s], pol);
            continue;
          }
          const uint32_t bytes = static_cast<uint32_t>(S.nr * rb);
          mbar_arrive_expect_tx(&full[s], bytes);
          const StageRows g = stage_rows_of(a, P, ph, q, s_idx);
          if (ph == 1) {   // nr/2 gate rows, then nr/2 up rows
            bulk_load_hint(dst, g.codes[0] + static_cast<long long>(g.row[0]) * rb, bytes / 2, &full[s], pol);
            const uint8_t* up = S.nr == 4 ? g.codes[2] + static_cast<long long>(g.row[2]) * rb
                                          : g.codes[1] + static_cast<long long>(g.row[1]) * rb;
            bulk_load_hint(dst + bytes / 2, up, bytes / 2, &full[s], pol);
          } else {
            bulk_load_hint(dst, g.codes[0] + static_cast<long long>(g.row[0]) * rb, bytes, &full[s], pol);
          }
        }
        qbase_p += S.n;
      }
      __syncwarp(0xFu);
      // every copy issued lands before the CTA can leave: per slot, the phase of its last issue
      if (lane == 0)
        for (int s = 0; s < kMkSlots; ++s) {
          const int j = s_last_issue[s];
          if (j >= 0 && !mbar_wait(&full[s], static_cast<uint32_t>(j / kMkSlots) & 1u, kDrainBudget))
            atomicOr(a.err, kErrDrain);
        }
    }
    return;
  }

  // ---- consumers (warps 0 .. 14)
  int qbase = 0;   // stages of the phases before the current one
  // This warp's stages of phase `ph`: those whose stage number over the phases is warp mod 15
  // (its two slots, used in turn); the scales of its next stage are read while the current
  // one is computed.  act_of(q, act, asc) picks the stage's activation; on_router(q, stage)
  // takes a router stage, on_stage(q, sums) a weight stage.
  auto consume = [&](int ph, auto&& act_of, auto&& on_router, auto&& on_stage) {
    const PhaseShare& S = P.ph[ph];
    with_shape(S.K, [&](auto NRc, auto CPWc) {
      constexpr int NR = decltype(NRc)::value, CPW = decltype(CPWc)::value;
      uint32_t sc[NR][CPW], sn[NR][CPW];
      const int nr_rt = ph == 0 ? P.r1 - P.r0 : 0;   // router stages lead phase 0
      const int q0 = (warp - qbase % kMkCWarps + kMkCWarps) % kMkCWarps;
      if (q0 < S.n && q0 >= nr_rt) stage_scales<NR, CPW>(stage_rows_of(a, P, ph, q0, s_idx), S.K, lane, sc);
      for (int q = q0; q < S.n; q += kMkCWarps) {
        const int qn = q + kMkCWarps;
        if (qn < S.n && qn >= nr_rt) stage_scales<NR, CPW>(stage_rows_of(a, P, ph, qn, s_idx), S.K, lane, sn);
        const int qg = qbase + q;
        const int s = qg % kMkSlots;
        if (mk_wait(&full[s], static_cast<uint32_t>(qg / kMkSlots) & 1u, budget, &s_dead, a.err)) {
          const uint8_t* st = ring + static_cast<size_t>(s) * kMkStageBytes;
          if (q < nr_rt) {   // a router row part
            on_router(q, st);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
          } else {
            const uint4* qa;
            const float* qs;
            act_of(q, qa, qs);
            float d[NR];
            stage_dot<NR, CPW>(st, S.K, qa, qs, sc, lane, d);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            on_stage(q, NR, d);
          }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
          for (int c = 0; c < CPW; ++c) sc[r][c] = sn[r][c];
      }
    });
    qbase += S.n;
  };
  auto same_act = [&](int, const uint4*& qa, const float*& qs) {
    qa = act;
    qs = asc;
  };
  // the sums of a unit spanning gpu stages go to slot (q / gpu) mod kMkUnitSlots; true when
  // this stage completed the unit (the caller then finishes it; the slot is free again)
  auto unit_done = [&](int slot, int gpu) {
    if (gpu == 1) return true;
    __threadfence_block();
    const int old = atomicAdd(&ucnt[slot], 1);
    if (old != gpu - 1) return false;
    __threadfence_block();
    ucnt[slot] = 0;
    return true;
  };

  if constexpr (MODE == kDecodeMkPost) {   // the routing of the pre kernel, from the workspace
    // launched while the down GEMM drains: the producer streams the unpooler's weights at once,
    // the consumers read nothing an earlier kernel wrote before that GEMM has completed
    griddep_wait();
    if (tid < k) {
      s_idx[tid] = a.topk_idx[tid];
      s_w[tid] = a.topk_w[tid];
      s_row[tid] = a.row_of[tid];
    }
    csync();
  } else {
  // ---- P1: pre-norm (fp32 xn in `row`; this CTA's slice of xa as bf16 hi/lo), Q(xn); x is
  // read once the previous kernel of the stream has completed
  griddep_wait();
  {
    float v[kRowChunks][8], g[kRowChunks][8];
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < kRowChunks; ++c) {
      const int i = (tid + kMkConsumers * c) * 8;
      if (i < D) {
        load_x8(a, i, v[c]);
        ldg8(a.g_pre + i, g[c]);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(v[c][e], v[c][e], ss);
      }
    }
    const float rs = rsqrtf(creduce(ss, red, false) / static_cast<float>(D) + a.eps);
#pragma unroll
    for (int c = 0; c < kRowChunks; ++c) {
      const int i = (tid + kMkConsumers * c) * 8;
      if (i < D) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = v[c][e] * rs * g[c][e];
        reinterpret_cast<float4*>(row + i)[0] = make_float4(o[0], o[1], o[2], o[3]);
        reinterpret_cast<float4*>(row + i)[1] = make_float4(o[4], o[5], o[6], o[7]);
      }
    }
  }
  csync();
  {
    const int per = (D + G - 1) / G;
    for (int i = cta * per + tid; i < min(D, (cta + 1) * per); i += kMkConsumers) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(row[i]);
      a.xa[i] = hi;
      a.xa[D + i] = __float2bfloat16_rn(row[i] - __bfloat162float(hi));
    }
  }
  const float s_x = quantize_row_smem(row, D, recip, red, act, asc);

  // ---- P2: router half rows (fp32 xn against bf16) and pooler rows
  {
    const float alpha = s_x * a.w[0].tensor_scale[0];
    const int nr_rt = P.r1 - P.r0;
    consume(
        0, same_act,
        [&](int q, const uint8_t* st) {
          const int u = P.r0 + q, part = u % P.rp, nv = D / P.rp / 8;   // 16-byte pieces of the part
          const float4* xr = reinterpret_cast<const float4*>(row + part * (D / P.rp));
          float acc = 0.f;
          for (int v = lane; v < nv; v += 32) {
            float w8[8];
            bf16x8(reinterpret_cast<const uint4*>(st)[v], w8);
            const float4 x0 = xr[2 * v], x1 = xr[2 * v + 1];
            acc = fmaf(w8[0], x0.x, acc);
            acc = fmaf(w8[1], x0.y, acc);
            acc = fmaf(w8[2], x0.z, acc);
            acc = fmaf(w8[3], x0.w, acc);
            acc = fmaf(w8[4], x1.x, acc);
            acc = fmaf(w8[5], x1.y, acc);
            acc = fmaf(w8[6], x1.z, acc);
            acc = fmaf(w8[7], x1.w, acc);
          }
          acc = warp_sum(acc);
          if (lane == 0) a.router_part[part * E + u / P.rp] = acc;
        },
        [&](int q, int nr, const float* d) {
          if (lane != 0) return;
          const long long l0 = static_cast<long long>(P.ph[0].u0 + (q - nr_rt)) * nr;
          for (int r = 0; r < nr; ++r) a.p[l0 + r] = d[r] * alpha;
        });
  }
  if (!grid_barrier(a, 0, &s_dead, &s_flag)) return;

  // ---- P3: logits, top-k + softmax (warp 0), the routing tables (CTA 0), pool norm, Q(h0)
  // p and g_pool first: their loads are in flight while the top-k runs
  float pv[kRowChunks][8], pg[kRowChunks][8];
  float sp = 0.f;
#pragma unroll
  for (int c = 0; c < kRowChunks; ++c) {
    const int i = (tid + kMkConsumers * c) * 8;
    if (i < L) {
      ldcg8(a.p + i, pv[c]);
      ldg8(a.g_pool + i, pg[c]);
    }
  }
  for (int e = tid; e < E; e += kMkConsumers) {
    float lg = __ldcg(a.router_part + e);   // the row's parts in order
    for (int pi = 1; pi < P.rp; ++pi) lg += __ldcg(a.router_part + pi * E + e);
    if (cta == 0) a.logits[e] = lg;
    vals[e] = lg + (a.router_bias != nullptr ? a.router_bias[e] : 0.f);
  }
  csync();
  if (warp == 0) mk_topk(a, vals, s_idx, s_w, &s_nt);
  csync();
  if (tid < k) {   // row of each pair: expert-major order (rank among the k, ties by slot)
    const int j = tid;
    int rnk = 0;
    for (int q = 0; q < k; ++q) rnk += s_idx[q] < s_idx[j] || (s_idx[q] == s_idx[j] && q < j);
    s_row[j] = rnk;
  }
  csync();
  if (tid == 0) {
    mbar_arrive(&route_ready);   // the producer may stream the experts' rows
    // this CTA's pieces of the k routed experts' gammas into L2 for the combine
    const uint32_t rowb = static_cast<uint32_t>(L) * 4u;
    for (uint32_t pc = cta; pc < static_cast<uint32_t>(k) * (rowb / 1024u); pc += G) {
      const uint32_t j = pc / (rowb / 1024u), off = (pc % (rowb / 1024u)) * 1024u;
      prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(a.g_expert + static_cast<long long>(s_idx[j]) * L) + off, 1024u);
    }
  }
  if (cta == 0) {   // the routing tables the kernel chain writes, for inspection and validation
    for (int e = tid; e < E; e += kMkConsumers) {
      int cnt = 0, before = 0;
      for (int j = 0; j < k; ++j) {
        cnt += s_idx[j] == e;
        before += s_idx[j] < e;
      }
      a.counts[e] = cnt;
      a.offsets[e] = before;
      a.tile_base[e] = before;
    }
    if (tid < k) {
      const int j = tid, r = s_row[j];
      a.topk_idx[j] = s_idx[j];
      a.topk_w[j] = s_w[j];
      if (a.idx_copy) a.idx_copy[j] = s_idx[j];
      if (a.w_copy) a.w_copy[j] = s_w[j];
      a.row_of[j] = r;
      a.tok_of[r] = 0;
      a.tiles[r] = Tile{s_idx[j], r, 1, 0};
      a.tiles2[r] = Tile{s_idx[j], r, 1, 0};
    }
    if (tid == 0) {
      a.offsets[E] = k;
      *a.n_tiles = k;
      *a.n_tiles2 = k;
      if (s_nt) atomicAdd(a.near_tie, 1);
    }
  }
  if constexpr (MODE == kDecodeMkPre) {
    // the gate/up GEMM may be launched now: its CTAs take the SMs as these exit (its set-up
    // reads the tables above as a hint; what it computes it reads after this kernel completes)
    if (cta == 0) __threadfence();
    griddep_launch_dependents();
  }
#pragma unroll
  for (int c = 0; c < kRowChunks; ++c) {
    const int i = (tid + kMkConsumers * c) * 8;
    if (i < L) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sp = fmaf(pv[c][e], pv[c][e], sp);
    }
  }
  {
    const float rs = rsqrtf(creduce(sp, red, false) / static_cast<float>(L) + a.eps);
#pragma unroll
    for (int c = 0; c < kRowChunks; ++c) {
      const int i = (tid + kMkConsumers * c) * 8;
      if (i < L) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = pv[c][e] * rs * pg[c][e];
        reinterpret_cast<float4*>(row + i)[0] = make_float4(o[0], o[1], o[2], o[3]);
        reinterpret_cast<float4*>(row + i)[1] = make_float4(o[4], o[5], o[6], o[7]);
      }
    }
  }
  csync();
  if constexpr (MODE == kDecodeMkPre) {
    // Q(h0) as the gate/up GEMM's A row of slot j = this CTA (CTAs 0 .. k-1): its row of the
    // expert-ordered rows, whose M tile is that row (one row per expert at one token)
    const int j = cta;
    const int r = j < k ? s_row[j] : 0;
    const float s = quantize_row_smem(row, L, recip, red, act, asc, j < k ? a.xe_codes + static_cast<long long>(r) * (L / 2) : nullptr,
                                      a.xe_scales, r);
    if (j < k && tid == 0) a.xe_rowscale[r] = s;
    return;
  }
  const float s_h0 = quantize_row_smem(row, L, recip, red, act, asc);

  // ---- P4: gate and up rows of the k experts; a unit is 16 rows of h (its 16 gate and 16 up
  // rows), finished by SwiGLU and Q(h) with scale 1
  {
    const PhaseShare& S = P.ph[1];
    consume(
        1, same_act, [](int, const uint8_t*) {},
        [&](int q, int nr, const float* d) {
          if (lane != 0) return;
          const int slot = (q >> S.lg) & (kMkUnitSlots - 1), r0 = (q & (S.gpu - 1)) * (nr / 2);
          float* part = part_all + slot * 32;
          for (int r = 0; r < nr / 2; ++r) {
            part[r0 + r] = d[r];                 // gate
            part[16 + r0 + r] = d[nr / 2 + r];   // up
          }
          if (!unit_done(slot, S.gpu)) return;
          const int u = S.u0 + (q >> S.lg), nb = I / 16, j = u / nb, ib = u % nb, e = s_idx[j];
          const float ag = s_h0 * a.w[1].tensor_scale[e], au = s_h0 * a.w[2].tensor_scale[e];
          float h[16];
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            const float x = part[r] * ag;
            h[r] = __fdividef(x, 1.f + __expf(-x)) * (part[16 + r] * au);   // silu(a) * b
          }
          uint2 qc;
          const uint32_t sc = nvfp4_quant16(h, 6.f, 1.f, recip, qc);
          *reinterpret_cast<uint2*>(a.h_codes + static_cast<long long>(j) * (I / 2) + ib * 8) = qc;
          a.h_scales[static_cast<long long>(j) * (I / 16) + ib] = static_cast<uint8_t>(sc);
        });
  }
  if (!grid_barrier(a, 1, &s_dead, &s_flag)) return;

  // ---- P5: Q(h) of every slot into shared memory, then the down rows of the k experts; a
  // unit is 16 rows of y of one slot: y = bf16(s_W (Q(h) . row)), and the unit's sum of
  // squares of the rounded values
  {
    const int nq = k * (I / 64);   // chunks of 64 codes: two uint4 and one word of scales
    for (int q0 = 0; q0 < nq; q0 += 4 * kMkConsumers) {
      uint4 c0[4], c1[4];
      uint32_t sw[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int q = q0 + tid + kMkConsumers * m;
        if (q < nq) {
          c0[m] = __ldcg(reinterpret_cast<const uint4*>(a.h_codes) + 2 * q);
          c1[m] = __ldcg(reinterpret_cast<const uint4*>(a.h_codes) + 2 * q + 1);
          sw[m] = __ldcg(reinterpret_cast<const unsigned*>(a.h_scales) + q);
        }
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int q = q0 + tid + kMkConsumers * m;
        if (q >= nq) continue;
        const int j = q / (I / 64), ch = q % (I / 64);
        const float2 s01 = e4m3x2_to_f2(sw[m]), s23 = e4m3x2_to_f2(sw[m] >> 16);
        uint4* ha = hact + j * (I / 8);
        float* hs = hsc + j * (I / 16);
        put_block(ha, hs, I / 32, 4 * ch, make_uint2(c0[m].x, c0[m].y), s01.x);
        put_block(ha, hs, I / 32, 4 * ch + 1, make_uint2(c0[m].z, c0[m].w), s01.y);
        put_block(ha, hs, I / 32, 4 * ch + 2, make_uint2(c1[m].x, c1[m].y), s23.x);
        put_block(ha, hs, I / 32, 4 * ch + 3, make_uint2(c1[m].z, c1[m].w), s23.y);
      }
    }
  }
  csync();
  {
    const PhaseShare& S = P.ph[2];
    const int nl = L / 16;
    consume(
        2,
        [&](int q, const uint4*& qa, const float*& qs) {   // the unit's slot's Q(h)
          const int j = (S.u0 + (q >> S.lg)) / nl;
          qa = hact + j * (I / 8);
          qs = hsc + j * (I / 16);
        },
        [](int, const uint8_t*) {},
        [&](int q, int nr, const float* d) {
          if (lane != 0) return;
          const int slot = (q >> S.lg) & (kMkUnitSlots - 1), r0 = (q & (S.gpu - 1)) * nr;
          float* part = part_all + slot * 32;
          for (int r = 0; r < nr; ++r) part[r0 + r] = d[r];
          if (!unit_done(slot, S.gpu)) return;
          const int u = S.u0 + (q >> S.lg), j = u / nl, l0 = (u % nl) * 16;
          const float ts = a.w[3].tensor_scale[s_idx[j]];
          uint32_t yb[8];
          float sq = 0.f;
#pragma unroll
          for (int r = 0; r < 16; r += 2) {
            const __nv_bfloat162 y2 = __floats2bfloat162_rn(part[r] * ts, part[r + 1] * ts);
            const float2 f = __bfloat1622float2(y2);
            sq = fmaf(f.x, f.x, sq);
            sq = fmaf(f.y, f.y, sq);
            yb[r / 2] = *reinterpret_cast<const uint32_t*>(&y2);
          }
          uint4* dst = reinterpret_cast<uint4*>(a.y + static_cast<long long>(s_row[j]) * L + l0);
          dst[0] = make_uint4(yb[0], yb[1], yb[2], yb[3]);
          dst[1] = make_uint4(yb[4], yb[5], yb[6], yb[7]);
          a.ss_part[u] = sq;
        });
  }
  if (!grid_barrier(a, 2, &s_dead, &s_flag)) return;
  }   // the pre and expert phases

  // ---- P6: per-expert norms (the units' sums of squares, staged in shared memory and summed
  // by one warp per slot), the weighted sum in slot order, Q(c)
  if constexpr (MODE == kDecodeMkPost) {   // the down GEMM's partial sums of squares of each y row
    for (int j = warp; j < k; j += kMkCWarps) {
      float sy = 0.f;
      for (int i = lane; i < a.ld_ss_y; i += 32) sy += __ldcg(a.ss_y + static_cast<long long>(s_row[j]) * a.ld_ss_y + i);
      sy = warp_sum(sy);
      if (lane == 0) s_coef[j] = s_w[j] * rsqrtf(sy / static_cast<float>(L) + a.eps);
    }
    csync();
  }
  {
    const int nl = L / 16, n4 = MODE == kDecodeMkPost ? 0 : k * nl / 4;
    for (int q0 = 0; q0 < n4; q0 += 4 * kMkConsumers) {
      float4 v[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int q = q0 + tid + kMkConsumers * m;
        if (q < n4) v[m] = __ldcg(reinterpret_cast<const float4*>(a.ss_part) + q);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int q = q0 + tid + kMkConsumers * m;
        if (q < n4) reinterpret_cast<float4*>(row)[q] = v[m];
      }
    }
    csync();
    for (int j = warp; j < k && MODE != kDecodeMkPost; j += kMkCWarps) {
      float sy = 0.f;
      for (int i = lane; i < nl; i += 32) sy += row[j * nl + i];
      sy = warp_sum(sy);
      if (lane == 0) s_coef[j] = s_w[j] * rsqrtf(sy / static_cast<float>(L) + a.eps);
    }
    csync();
    float acc[kRowChunks][8];
#pragma unroll
    for (int c = 0; c < kRowChunks; ++c)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[c][e] = 0.f;
#pragma unroll
    for (int c = 0; c < kRowChunks; ++c) {
      const int i = (tid + kMkConsumers * c) * 8;
      if (i >= L) continue;
      for (int j0 = 0; j0 < k; j0 += 4) {   // four slots' loads in flight, summed in slot order
        uint4 yq[4];
        float g[4][8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          if (j0 + m < k) {
            yq[m] = __ldcg(reinterpret_cast<const uint4*>(a.y + static_cast<long long>(s_row[j0 + m]) * L + i));
            ldg8(a.g_expert + static_cast<long long>(s_idx[j0 + m]) * L + i, g[m]);
          }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          if (j0 + m >= k) continue;
          float yv[8];
          bf16x8(yq[m], yv);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[c][e] = fmaf(s_coef[j0 + m], yv[e] * g[m][e], acc[c][e]);
        }
      }
    }
    csync();   // the staged sums of squares are read
#pragma unroll
    for (int c = 0; c < kRowChunks; ++c) {
      const int i = (tid + kMkConsumers * c) * 8;
      if (i < L) {
        reinterpret_cast<float4*>(row + i)[0] = make_float4(acc[c][0], acc[c][1], acc[c][2], acc[c][3]);
        reinterpret_cast<float4*>(row + i)[1] = make_float4(acc[c][4], acc[c][5], acc[c][6], acc[c][7]);
      }
    }
  }
  csync();
  const float s_c = quantize_row_smem(row, L, recip, red, act, asc);

  // ---- P7: unpooler rows, 4 per unit, with the unit's sum of squares
  {
    const PhaseShare& S = P.ph[3];
    const float alpha = s_c * a.w[4].tensor_scale[0];
    float* ss_u = a.ss_part + k * (L / 16);
    consume(
        3, same_act, [](int, const uint8_t*) {},
        [&](int q, int nr, const float* d) {
          if (lane != 0) return;
          float v[4];
          if (S.gpu == 1) {   // the stage is the unit: no slot
            for (int r = 0; r < 4; ++r) v[r] = d[r] * alpha;
          } else {
            const int slot = (q >> S.lg) & (kMkUnitSlots - 1), r0 = (q & (S.gpu - 1)) * nr;
            float* part = part_all + slot * 32;
            for (int r = 0; r < nr; ++r) part[r0 + r] = d[r] * alpha;
            if (!unit_done(slot, S.gpu)) return;
            for (int r = 0; r < 4; ++r) v[r] = part[r];
          }
          const int u = S.u0 + (q >> S.lg);
          float sq = 0.f;
#pragma unroll
          for (int r = 0; r < 4; ++r) sq = fmaf(v[r], v[r], sq);
          *reinterpret_cast<float4*>(a.u + u * 4) = make_float4(v[0], v[1], v[2], v[3]);
          ss_u[u] = sq;
        });
  }
  if (!grid_barrier(a, MODE == kDecodeMkPost ? 0 : 3, &s_dead, &s_flag)) return;
  griddep_launch_dependents();   // the next kernel may be launched during the post-norm

  // ---- P8: post-norm + residual; CTA c writes its slice of the output row (and of the next
  // layer's pre-norm of it, whose row sum every CTA takes over the whole row)
  float su = 0.f;
  {
    const float* ss_u = a.ss_part + k * (L / 16);
    for (int q = tid; q < D / 16; q += kMkConsumers) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(ss_u) + q);
      su += (v.x + v.y) + (v.z + v.w);
    }
  }
  const float rs_u = rsqrtf(creduce(su, red, false) / static_cast<float>(D) + a.eps);
  auto as_stored = [&](float o) { return a.out_f32 ? o : __bfloat162float(__float2bfloat16_rn(o)); };
  float rs_next = 0.f;
  if (a.g_next != nullptr) {
    float so = 0.f;
#pragma unroll
    for (int c = 0; c < kRowChunks; ++c) {
      const int i = (tid + kMkConsumers * c) * 8;
      if (i >= D) continue;
      float xv[8], uv[8], gv[8];
      load_x8(a, i, xv);
      ldcg8(a.u + i, uv);
      ldg8(a.g_post + i, gv);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float o = as_stored(xv[e] + uv[e] * rs_u * gv[e]);
        so = fmaf(o, o, so);
      }
    }
    rs_next = rsqrtf(creduce(so, red, false) / static_cast<float>(D) + a.eps);
  }
  const int per = (D + G - 1) / G;
  for (int i = cta * per + tid; i < min(D, (cta + 1) * per); i += kMkConsumers) {
    const float o = as_stored(load_x(a, i) + __ldcg(a.u + i) * rs_u * a.g_post[i]);
    if (a.out_f32) static_cast<float*>(a.out)[i] = o;
    else static_cast<__nv_bfloat16*>(a.out)[i] = __float2bfloat16_rn(o);
    if (a.g_next != nullptr) {
      const float nx = o * rs_next * a.g_next[i];
      if (a.out_f32) static_cast<float*>(a.next_out)[i] = nx;
      else static_cast<__nv_bfloat16*>(a.next_out)[i] = __float2bfloat16_rn(nx);
    }
  }
}

}  // namespace

size_t decode_megakernel_smem(int D, int L, int I, int E, int k) { return mk_smem_bytes(D, L, I, E, k); }

bool decode_megakernel_fits(int D, int L, int I, int E, int k) {
  auto ok = [](int K) { return K >= 256 && K <= kMkMaxK && K % 256 == 0; };
  // a gate/up stage holds at least one gate and one up row: L <= 4096
  if (!ok(D) || !ok(L) || !ok(I) || L > 4096 || E < 1 || E > 1024 || k < 1 || k > 16 || k > E) return false;
  return mk_smem_bytes(D, L, I, E, k) <= static_cast<size_t>(kDecodeMkMaxSmem);
}

long long decode_megakernel_scratch_floats(int D, int L, int E, int k) {
  return static_cast<long long>(k) * (L / 16) + D / 4 + static_cast<long long>(router_parts(D)) * E;
}

// Internal linkage for the launch helpers below: a template's function-local static (the
// shared-memory attribute flag) would otherwise be one weak symbol shared by every copy of
// this library in a process (the release and the bounds-checked builds), and the second copy
// would skip setting the attribute on its own kernel.
namespace {

// The words a single-token call starts from zero (error word, near-tie count, the grid barrier
// counts), cleared once the previous kernel of the stream has completed.  It lets the kernel
// after it launch at once, which then waits for it.
__global__ void decode_clear_kernel(unsigned* w, int n) {
  griddep_launch_dependents();
  griddep_wait();
  if (static_cast<int>(threadIdx.x) < n) w[threadIdx.x] = 0u;
}

template <int MODE>
cudaError_t launch_mode(const DecodeMkArgs& d, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(decode_megakernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kDecodeMkMaxSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sm_count()));   // one CTA per SM
  cfg.blockDim = dim3(kMkThreads);
  cfg.dynamicSmemBytes = decode_megakernel_smem(d.D, d.L, d.I, d.E, d.k);
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  // cooperative: the driver starts the grid once every CTA can be resident (the grid barriers
  // wait on one another); else an ordinary grid of one CTA per SM, whose CTAs take the SMs the
  // previous kernel leaves (every CTA fits at once on an otherwise idle GPU)
  attrs[0].id = cudaLaunchAttributeCooperative;
  attrs[0].val.cooperative = d.cooperative ? 1 : 0;
  // programmatic dependent launch: the kernel's set-up and weight stream run while the previous
  // kernel finishes; its consumers wait for that kernel before reading what it wrote
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  count_launch();
  return cudaLaunchKernelEx(&cfg, decode_megakernel<MODE>, d);
}

}  // namespace

cudaError_t launch_decode_clear(unsigned* words, int n, cudaStream_t s) {
  if (n < 0 || n > 32) return cudaErrorInvalidValue;
  return launch_pdl(decode_clear_kernel, dim3(1), dim3(32), 0, s, words, n);
}

cudaError_t launch_decode_megakernel(const DecodeMkArgs& d, cudaStream_t s) {
  if (!decode_megakernel_fits(d.D, d.L, d.I, d.E, d.k)) return cudaErrorInvalidValue;
  switch (d.mode) {
    case kDecodeMkPre: return launch_mode<kDecodeMkPre>(d, s);
    case kDecodeMkPost: return launch_mode<kDecodeMkPost>(d, s);
    default: return launch_mode<kDecodeMkFull>(d, s);
  }
}

}  // namespace lmoe
