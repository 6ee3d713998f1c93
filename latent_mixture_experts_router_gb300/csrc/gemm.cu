// gemm.cu — grouped BF16 GEMM on the 5th-generation tensor cores (tcgen05), persistent.
//
// out[r, n] = sum_kb A[r, kA(kb)] * B[e*N + n, kB(kb)]  for the rows r of each M tile,
// where e is the tile's expert (0 for a plain GEMM) and the k coordinates of A and B
// wrap at their own periods, so that one operand can be paired with a hi/lo split of
// the other (K-concatenation without copying).  A and B are K-major bf16 staged in shared
// memory by TMA (128-byte swizzle); fp32 accumulators live in tensor memory.
//
// One CTA per SM walks the (128 MH) x BN output tiles in grouped order (groups of 16 M
// tiles, M fastest inside a group, ids strided by the grid size), with three roles:
//   warp 0, lane 0   TMA producer over a ring of smem stages (the ring runs on across tiles)
//   warp 1, lane 0   tcgen05.mma issuer; warp 1 also owns the TMEM allocation (512 columns)
//   warps 2..5       epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 (one row each).  (Eight
//                    epilogue warps on half the columns each measured slower here: the
//                    waiting warps take issue slots from the producer and the MMA issuer.)
// MH = 1: 128-row tiles, 4 stages, two accumulator buffers (the next tile's MMAs run while
// the epilogue drains the previous one) — the weight-streaming regime of few rows.
// MH = 2: 256-row tiles (two M = 128 MMAs per K step share each B tile), 3 stages, one
// accumulator buffer spanning the 512 columns.  A CTA can take in only about 100 GB/s of
// operands from L2 or HBM; a 128 x 256 bf16 tile needs 48 KB per 2 x 128 x 256 x 64 FLOP,
// which caps it near 70 % of the tensor rate, while the 256-row tile needs 64 KB per twice
// the work — the many-row (prefill) regime.
// Epilogues (one per use in the latent-MoE block):
//   kEpiF32     fp32 logits (router)
//   kEpiF32Ss   fp32 output plus, per row, the partial sum of squares of the values of
//               this tile's columns.  The row's RMS is finished later from these partials,
//               so no kernel re-reads the row to normalise it (the "fused per-expert
//               post-norm" of the LMSYS Muse Spark Open post: each second-GEMM tile
//               accumulates a partial sum of squares of the values it holds in registers;
//               here partials go to [rows, N/BN] without atomics, so the result is
//               deterministic).  The outputs stay fp32 because they are not tensor-core
//               operands: rounding them would only add error.
//   kEpiSwiGLU  gate and up tiles of the same columns in one CTA (two B loads per stage,
//               two accumulators), output bf16 silu(a) * b.
#include "internal.h"
#include "ptx.cuh"
#include "tiles.cuh"

namespace lmoe {

template <int BN, int EPI, int MH>
struct GemmCfg {
  static constexpr bool kDual = (EPI == kEpiSwiGLU);
  static constexpr int kStages = MH == 2 ? 3 : 4;
  static constexpr int kAHalf = kBM * kBK * 2;            // one 128-row half of A
  static constexpr int kABytes = MH * kAHalf;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes * (kDual ? 2 : 1);
  static constexpr int kAccCols = kDual ? 2 * BN : BN;   // accumulator of one M half
  static constexpr int kBufCols = MH * kAccCols;         // one accumulator buffer
  static constexpr int kAccBufs = 512 / kBufCols >= 2 ? 2 : 1;
  static constexpr int kTileRows = MH * kBM;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kEpiWarps = MH == 2 ? 8 : 4;   // 256-row tiles: twice the rows to drain
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kXposeOff = kStages * kStageBytes + 256;   // after the barriers
  static constexpr int kXposeBytes = kEpiWarps * 32 * 33 * 4;      // reserved when args.xpose
  static constexpr int kSmemBytes = kXposeOff + kXposeBytes + 1024 /*align*/;
  static_assert(kAccBufs * kBufCols <= 512, "accumulator buffers in tensor memory");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile N");
  static_assert(MH == 1 || MH == 2, "one or two M halves");
};

template <int BN, int EPI, int MH>
__global__ void __launch_bounds__(GemmCfg<BN, EPI, MH>::kThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmB2, const GemmArgs args) {
  using C = GemmCfg<BN, EPI, MH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;    // [2] MMA -> epilogue
  uint64_t* acc_empty = acc_full + 2;         // [2] epilogue (4 warps) -> MMA
  uint64_t* mma_done = acc_empty + 2;         // every MMA of this CTA has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // epilogue warp w's transpose tile for coalesced fp32 stores
  float* xpose = reinterpret_cast<float*>(smem + C::kXposeOff) + (warp >= 2 ? (warp - 2) * 32 * 33 : 0);

  // Set-up reads nothing an earlier kernel of the stream writes, so it runs before the wait,
  // overlapping the end of that kernel, and so does an L2 prefetch of this CTA's first
  // weight tile.
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], C::kEpiWarps);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (C::kDual) prefetch_tmap(&tmB2);
    int brow, kb0, kb1;
    if (first_tile_hint(args.tiles, args.n_tiles, args.max_tiles, args.n_groups, args.M, args.N, BN,
                        args.k_splits, args.num_kb, false, brow, kb0, kb1, C::kTileRows)) {
      for (int kb = kb0; kb < min(kb1, kb0 + kPrefetchKb); ++kb) {
        const int kbb = (kb % args.kb_period_b) * kBK;
        prefetch_l2_tile_2d(&tmB, kbb, brow);
        if (C::kDual) prefetch_l2_tile_2d(&tmB2, kbb, brow);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_enter();
  // CTAs past the live tile ids walk nothing and go straight to the teardown
  const TileWalk walk(args.tiles, args.n_tiles, args.M, args.N, BN, args.k_splits, args.num_kb, false,
                      C::kTileRows);
  const long long budget = args.budget;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer
      const uint64_t pol_b = args.b_stream_once ? policy_evict_first() : policy_evict_normal();
      int it = 0;
      bool ok = true;
      for (int id = blockIdx.x; ok && id < walk.n_ids; id += gridDim.x) {
        int expert, row0, nrows, ntile;
        if (!walk.at(id, expert, row0, nrows, ntile)) continue;
        const int brow = expert * args.N + ntile * BN;
        const int halves = nrows > kBM ? 2 : 1;   // a 256-row tile with at most 128 live rows
        const uint32_t tx = C::kStageBytes - (MH - halves) * C::kAHalf;   // skips its second half
        int kb0, kb1;
        walk.k_range(id, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          const int s = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, budget)) {
            atomicOr(args.err, kErrWaitProducer);
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * C::kStageBytes;
          mbar_arrive_expect_tx(&full[s], tx);
          const int ka = (kb % args.kb_period_a) * kBK;
          tma_load_2d(sa, &tmA, &full[s], ka, row0);
          if (MH == 2 && halves == 2) tma_load_2d(sa + C::kAHalf, &tmA, &full[s], ka, row0 + kBM);
          const int kbb = (kb % args.kb_period_b) * kBK;
          tma_load_2d_hint(sa + C::kABytes, &tmB, &full[s], kbb, brow, pol_b);
          if (C::kDual) tma_load_2d_hint(sa + C::kABytes + C::kBBytes, &tmB2, &full[s], kbb, brow, pol_b);
          ++it;
        }
      }
      // before leaving, let every copy this thread issued land (drain budget, independent
      // of the caller's: the CTA must not exit with a copy still writing its smem)
      for (int j = max(0, it - C::kStages); j < it; ++j)
        if (!mbar_wait(&full[j % C::kStages], (j / C::kStages) & 1, kDrainBudget))
          atomicOr(args.err, kErrDrain);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
      int it = 0, tc = 0;
      bool ok = true;
      for (int id = blockIdx.x; ok && id < walk.n_ids; id += gridDim.x) {
        int expert, row0, nrows, ntile;
        if (!walk.at(id, expert, row0, nrows, ntile)) continue;
        const int halves = nrows > kBM ? 2 : 1;
        const int buf = tc % C::kAccBufs;
        const uint32_t use = (tc / C::kAccBufs) & 1;
        if (!mbar_wait(&acc_empty[buf], use ^ 1, budget)) {   // epilogue released this buffer
          atomicOr(args.err, kErrWaitMma);
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + buf * C::kBufCols;
        int kb0, kb1;
        walk.k_range(id, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          const int s = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          if (!mbar_wait(&full[s], ph, budget)) {
            atomicOr(args.err, kErrWaitMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * C::kStageBytes);
          const uint32_t b0 = a0 + C::kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t accum = (kb > kb0 || kk > 0) ? 1u : 0u;
            const uint64_t bd = sw128_kmajor_desc(b0 + kk * 32);
            const uint64_t bd2 = sw128_kmajor_desc(b0 + C::kBBytes + kk * 32);
#pragma unroll
            for (int h = 0; h < MH; ++h) {
              if (h >= halves) break;
              const uint64_t ad = sw128_kmajor_desc(a0 + h * C::kAHalf + kk * 32);
              const uint32_t dh = acc + h * C::kAccCols;
              mma_bf16(dh, ad, bd, idesc, accum);
              if (C::kDual) mma_bf16(dh + BN, ad, bd2, idesc, accum);
            }
          }
          mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
          ++it;
        }
        mma_commit(&acc_full[buf]);  // accumulator of this tile complete (or abandoned)
        ++tc;
      }
      mma_commit(mma_done);
    }
  } else {
    // ---- epilogue: TMEM lane quadrant = warp % 4; with 8 warps, column half (warp - 2) / 4
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quad * 32 + lane;
    constexpr int kCols = BN * 4 / C::kEpiWarps;
    const int c_lo = half * kCols, c_hi = c_lo + kCols;
    int tc = 0;
    for (int id = blockIdx.x; id < walk.n_ids; id += gridDim.x) {
      int expert, row0, nrows, ntile;
      if (!walk.at(id, expert, row0, nrows, ntile)) continue;
      const int buf = tc % C::kAccBufs;
      const uint32_t use = (tc / C::kAccBufs) & 1;
      if (!mbar_wait(&acc_full[buf], use, budget)) {
        atomicOr(args.err, kErrWaitEpilogue);
        break;
      }
      tc_fence_after();
      const int halves = nrows > kBM ? 2 : 1;
      const int n0 = ntile * BN;
#pragma unroll 1
      for (int h = 0; h < halves; ++h) {
      const int rr = h * kBM + r;   // row within the tile
      const bool row_ok = rr < nrows;
      const long long grow = static_cast<long long>(row0) + rr;
      // this warp's 32 rows: the first of them, and how many hold live rows
      const long long wrow = static_cast<long long>(row0) + h * kBM + quad * 32;
      const int wvalid = min(32, max(0, nrows - (h * kBM + quad * 32)));
      const uint32_t tq = tmem + buf * C::kBufCols + h * C::kAccCols + (static_cast<uint32_t>(quad * 32) << 16);
      if (EPI != kEpiSwiGLU && walk.splits > 1) {
        // split-K: raw fp32 partial product of this K range; the reduction finishes the tile
        const long long pbase = static_cast<long long>(id % walk.splits) * args.M;
        float* prow = args.partial + (pbase + grow) * args.N;
#pragma unroll 1
        for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32cols(tq + c0, v);
          tmem_ld_wait();
          const int col = n0 + c0;
          if (args.xpose && col + 32 <= args.N) {   // warp-uniform
            warp_store_32x32_f32(xpose, v, args.partial + (pbase + wrow) * args.N + col, args.N, wvalid, lane);
          } else if (row_ok && col + 32 <= args.N) {
            store_row32_f32(prow + col, v);
          } else if (row_ok && col < args.N) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col + i < args.N) prow[col + i] = __uint_as_float(v[i]);
          }
        }
      } else if constexpr (EPI == kEpiF32) {
        float* orow = static_cast<float*>(args.out) + grow * args.ldo;
        float* wout = static_cast<float*>(args.out) + wrow * args.ldo;
#pragma unroll 1
        for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32cols(tq + c0, v);
          tmem_ld_wait();
          const int col = n0 + c0;
          if (args.xpose && col + 32 <= args.N) {   // warp-uniform
            warp_store_32x32_f32(xpose, v, wout + col, args.ldo, wvalid, lane);
          } else if (row_ok && col + 32 <= args.N) {
            store_row32_f32(orow + col, v);
          } else if (row_ok && col < args.N) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col + i < args.N) orow[col + i] = __uint_as_float(v[i]);
          }
        }
      } else if constexpr (EPI == kEpiF32Ss) {
        // row sums of squares per 128 columns ([rows, N/128]; the consumer adds them in order)
        float* orow = static_cast<float*>(args.out) + grow * args.ldo;
        float* wout = static_cast<float*>(args.out) + wrow * args.ldo;
        float ss0 = 0.f, ss1 = 0.f;   // columns [c_lo, c_lo + 128), [c_lo + 128, c_hi)
#pragma unroll 1
        for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32cols(tq + c0, v);
          tmem_ld_wait();
          const int col = n0 + c0;
          if (col + 32 > args.N) continue;   // (N is a multiple of 128 here)
          float sp = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) sp = fmaf(__uint_as_float(v[i]), __uint_as_float(v[i]), sp);
          if (c0 - c_lo < 128) ss0 += sp;
          else ss1 += sp;
          if (args.xpose) warp_store_32x32_f32(xpose, v, wout + col, args.ldo, wvalid, lane);
          else if (row_ok) store_row32_f32(orow + col, v);
        }
        if (row_ok) {
          float* srow = args.ss + grow * args.ld_ss + (n0 + c_lo) / 128;
          srow[0] = ss0;
          if (c_hi - c_lo > 128 && n0 + c_lo + 128 < args.N) srow[1] = ss1;
        }
      } else {  // kEpiSwiGLU
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(args.out) + grow * args.ldo;
#pragma unroll 1
        for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
          uint32_t g[32], u[32];
          tmem_ld_32cols(tq + c0, g);
          tmem_ld_32cols(tq + BN + c0, u);
          tmem_ld_wait();
          const int col = n0 + c0;
          if (row_ok && col + 32 <= args.N) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a0 = __uint_as_float(g[2 * i]), a1 = __uint_as_float(g[2 * i + 1]);
              const float h0 = __fdividef(a0, 1.f + __expf(-a0)) * __uint_as_float(u[2 * i]);
              const float h1 = __fdividef(a1, 1.f + __expf(-a1)) * __uint_as_float(u[2 * i + 1]);
              pk[i] = pack_bf16x2(h0, h1);
            }
            uint4* o = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      }
      }  // M halves
      // every TMEM read of this buffer is complete: hand it back to the MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
      ++tc;
    }
  }

  // ---- teardown: all MMAs of this CTA have completed before the columns are released
  if (warp == 1 && lane == 0)
    if (!mbar_wait(mma_done, 0, kDrainBudget)) atomicOr(args.err, kErrDrain);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

template <int BN, int EPI, int MH>
static cudaError_t launch_one(const CUtensorMap& tmA, const CUtensorMap& tmB,
                              const CUtensorMap& tmB2, const GemmArgs& a, int m_tiles,
                              cudaStream_t s) {
  using C = GemmCfg<BN, EPI, MH>;
  auto kern = gemm_tcgen05_kernel<BN, EPI, MH>;
  static bool attr_set = false;  // per process; the attribute is per function
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // upper bound of the tile ids (the live M-tile count of a grouped GEMM is on the device)
  const long long ids = tile_id_bound(m_tiles, a.N, BN, a.k_splits > 1 ? a.k_splits : 1);
  if (ids == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(ids < sm_count() ? ids : sm_count());
  const int smem = C::kSmemBytes - (a.xpose ? 0 : C::kXposeBytes);
  return launch_pdl(kern, dim3(grid), dim3(C::kThreads), smem, s, tmA, tmB, tmB2, a);
}

cudaError_t launch_gemm(EpiKind epi, const CUtensorMap& tmA, const CUtensorMap& tmB,
                        const CUtensorMap& tmB2, const GemmArgs& a, int m_tiles,
                        cudaStream_t s, int m_halves) {
  if (m_halves == 2) {
    switch (epi) {
      case kEpiF32: return launch_one<kBNWide, kEpiF32, 2>(tmA, tmB, tmB2, a, m_tiles, s);
      case kEpiF32Ss: return launch_one<kBNWide, kEpiF32Ss, 2>(tmA, tmB, tmB2, a, m_tiles, s);
      case kEpiSwiGLU: return launch_one<kBNSwiGLU, kEpiSwiGLU, 2>(tmA, tmB, tmB2, a, m_tiles, s);
    }
    return cudaErrorInvalidValue;
  }
  switch (epi) {
    case kEpiF32: return launch_one<kBNWide, kEpiF32, 1>(tmA, tmB, tmB2, a, m_tiles, s);
    case kEpiF32Ss: return launch_one<kBNWide, kEpiF32Ss, 1>(tmA, tmB, tmB2, a, m_tiles, s);
    case kEpiSwiGLU: return launch_one<kBNSwiGLU, kEpiSwiGLU, 1>(tmA, tmB, tmB2, a, m_tiles, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lmoe
