// gemm_fp4.cu — grouped NVFP4 x NVFP4 GEMM on the block-scaled 5th-generation tensor cores,
// persistent.
//
// out[r, n] = alpha_r,e * sum_k A[r, k] * B[e*N + n, k], with A and B packed E2M1 (two
// values per byte, K contiguous) and one UE4M3 scale per 16 consecutive k on both operands
// (LMSYS "SGLang and Miles Add Day-0 Support for Muse Spark Open", "NVFP4 as a third MMA
// type": nvfp4 x nvfp4 with 16-element UE4M3 block scales; the per-token FP32 input scale
// is applied to the accumulator).  alpha = row scale (per token / per routed row, or 1) *
// tensor scale of the weight (per expert).
//
// One CTA per SM walks the 128 x BN output tiles in grouped order (as the BF16 GEMM); a
// pipeline stage covers K = 256 (128 bytes of codes per row, and the 2 KB of scales of the
// stage's 128-row block).  The scales are kept in memory in the layout the tensor cores
// read through tcgen05.cp 32x128b (blocks of 32 lines x 16 bytes, line m0 holding the 4
// scale bytes of rows m0, m0+32, m0+64, m0+96 — the "4x32 transpose" the pages apply before
// the copy, done once when the scales are written), so a stage's scales are one bulk copy.
// Roles (224 or 352 threads):
//   warp 0 lane 0   TMA: A codes + B codes (+ B2 for gate/up) + bulk copies of their scales
//   warp 1          TMEM allocation; lane 0 issues tcgen05.mma.kind::mxf4nvf4.block_scale.
//                   scale_vec::4X
//   warps 2..        epilogue: warp w owns TMEM lanes 32*(w%4) ..; the gate/up kernel runs
//                   8 epilogue warps, warp w also taking column half (w-2)/4, so each
//                   scheduler runs two of them and a tile drains in half the time (its
//                   single accumulator waits for that); the fp32 kernels run 4
//   last warp lane 0  copies each stage's scale factors into tensor memory (tcgen05.cp) and
//                   signals them ready through its own barrier.  A thread takes about as
//                   long to issue one 512-byte scale copy as one MMA, so copies issued by
//                   the MMA thread would double its time per stage; from a second thread
//                   they overlap the MMAs of the previous stage.
// The A box covers only the tile's live rows rounded up to 32 (a decode tile holds a few
// rows of one expert), and the producer loads the next tile's table entry one tile ahead.
// Epilogues: kFp4EpiF32Ss — alpha * acc as fp32 plus per-row partial sums of squares; two
// accumulator buffers, so the next tile's MMAs overlap this tile's epilogue.  kFp4EpiBf16Ss —
// the same with the values rounded to bf16 and the sums of squares taken of the rounded values
// (the expert down projection: each tile's partial sum of squares of the bf16 values it holds).
// kFp4EpiF32SsWide / kFp4EpiBf16SsWide — those epilogues on 128 x 256 tiles (the dense
// pooler/unpooler at many rows, the grouped down projection wherever it runs unsplit): a stage
// loads the two 128-row halves of the tile's weights (as gate/up loads its two weights), so
// the A tile, its scales and the per-stage barrier and scale-copy work come once per 256
// output columns (at prefill the operand intake of an SM, ~97 GB/s measured, bounds these
// GEMMs; at decode the per-stage overheads of a 16 KB weight stage); one accumulator buffer
// of 256 columns.
// kFp4EpiSwiGLUQuant — gate and up tiles of the same columns, h = silu(alpha_g acc_g) *
// (alpha_u acc_u) requantised to NVFP4 with scale 1 (block scales only, through the
// reciprocal table) for the down projection; one accumulator buffer (two would leave no
// tensor memory for the scale factors), while TMA runs ahead.
#include "internal.h"
#include "nvfp4.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace lmoe {

namespace {

LMOE_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory descriptor of a 512-byte scale block: 4 core matrices of 8 lines x 16 B,
// contiguous (stride 128 B), no swizzle.
LMOE_DEV uint64_t sf_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

LMOE_DEV void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Instruction descriptor of kind::mxf4nvf4 block-scaled MMA: A/B E2M1 ([7,10) = 1,
// [10,13) = 1), K-major, N>>3 at [17,23), scale type UE4M3 ([23] = 0), M>>4 at [24,29),
// scale-factor ids 0 ([4,6) and [29,31)).
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

LMOE_DEV void mma_nvf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                       uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// AROWS: A rows a stage holds (128, or 32 where no tile has more than 32 rows: a few tokens).
// The MMA still takes M = 128; with 32 the rows past the A box read the stage's B bytes, and
// their accumulator rows are never stored.  The smaller A area buys a deeper ring: at a few
// rows a CTA streams its weight tiles at the rate of the bytes it keeps in flight.
template <int BN, int EPI, int AROWS = kBM>
struct Fp4Cfg {
  // kDual: two B boxes per stage into two accumulators of BN columns — gate and up tiles of the
  // same columns (SwiGLU), or the two BN-row halves of one 2*BN-wide output tile (kWide)
  static constexpr bool kWide = (EPI == kFp4EpiF32SsWide) || (EPI == kFp4EpiBf16SsWide);
  static constexpr bool kDual = (EPI == kFp4EpiSwiGLUQuant) || kWide;
  static constexpr int kTileN = kWide ? 2 * BN : BN;   // output columns of one tile
  static constexpr int kNB = kDual ? 2 : 1;
  static_assert(AROWS == kBM || AROWS == 32, "A boxes of 32 rows");
  // 128 A rows: what fits 227 KB; 32: what fits both 227 KB and the 512 TMEM columns
  static constexpr int kStages = AROWS == kBM ? (kDual ? 4 : 6) : (kDual ? 5 : 8);
  static constexpr int kKStep = 4;                 // MMAs (K = 64 each) per stage
  static constexpr int kABoxes = AROWS / 32;       // A boxes of 32, 64, 96, 128 rows usable
  static constexpr int kABytes = AROWS * 128;      // codes (at most; the box follows the live rows)
  static constexpr int kBBytes = BN * 128;
  static constexpr int kSfaBytes = 4 * 512;        // block-layout scales of the stage: one
  static constexpr int kSfbBytes = 4 * 512;        // 512-byte block per K step (B: BN-row blocks)
  // stage layout: [A codes][B codes x kNB][A scales][B scales x kNB]
  static constexpr int kOffB = kABytes;
  static constexpr int kOffSfa = kOffB + kNB * kBBytes;
  static constexpr int kOffSfb = kOffSfa + kSfaBytes;
  static constexpr int kStageBytes = kOffSfb + kNB * kSfbBytes;
  // bytes landing per stage when the A box has `arows` rows
  static constexpr __host__ __device__ uint32_t tx_bytes(int arows) {
    return static_cast<uint32_t>(arows * 128 + kSfaBytes + kNB * (kBBytes + kSfbBytes));
  }
  // tensor memory: accumulator buffer(s), then per-stage scale columns (4 per K step)
  static constexpr int kAccCols = kNB * BN;
  static constexpr int kAccBufs = kDual ? 1 : 2;   // two gate+up buffers would leave no room for scales
  static constexpr int kSfaCols = kKStep * 4;
  static constexpr int kSfbColsOne = kKStep * 4;
  static constexpr int kSfCols = kSfaCols + kNB * kSfbColsOne;
  static constexpr int kSfCol0 = kAccBufs * kAccCols;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 1024 /*recip*/ + 256;
  static constexpr int kEpiWarps = kDual ? 8 : 4;
  static constexpr int kCopyWarp = 2 + kEpiWarps;             // scale-factor copies
  static constexpr int kThreads = 32 * (kCopyWarp + 1);
  static_assert(kSfCol0 + kStages * kSfCols <= 512, "tensor memory");
  static_assert((3 * kStages + 5) * 8 + 4 <= 256, "barriers and the TMEM slot after recip");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kStageBytes % 1024 == 0, "1024-byte aligned stages");
  static_assert(BN == 128, "one 128-row scale block of B per stage");
};

// Epilogue of a 128 x 2BN tile (kWide): this warp's TMEM lanes (tq), accumulator columns
// [half BN, (half+1) BN) = output columns n0 + half BN ..; all of them are read into registers
// and the single accumulator buffer is handed back to the MMA issuer before the scaling and the
// stores.  alpha = row scale * tensor scale; split_idx >= 0: the split-K partial of that index
// (fp32, no sums of squares); else bf16 (kFp4EpiBf16SsWide: rounded values, and the sum of
// squares of the rounded values) or fp32 values with their sum of squares per 128 columns.
template <int BN, int EPI>
LMOE_DEV void epi_wide(const Fp4Args& args, uint32_t tq, int half, uint64_t* acc_empty, int lane, int n0,
                       float alpha, int split_idx, long long grow, bool row_ok) {
  const bool split = split_idx >= 0;
  // bf16 output (unsplit): rounded values, and the sum of squares of the rounded values
  const bool bf = EPI == kFp4EpiBf16SsWide && !split;
  constexpr int kCh = BN / 32;
  uint32_t v[kCh][32];
#pragma unroll
  for (int ch = 0; ch < kCh; ++ch) tmem_ld_32cols(tq + half * BN + 32 * ch, v[ch]);
  tmem_ld_wait();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(acc_empty);
  const int cbase = n0 + half * BN;
  float* orow = split ? args.partial + (static_cast<long long>(split_idx) * args.M + grow) * args.N
                      : static_cast<float*>(args.out) + grow * args.ldo;
  float ss = 0.f;
  if (row_ok && cbase + BN <= args.N) {
    if (bf) {
      __nv_bfloat16* brow = static_cast<__nv_bfloat16*>(args.out) + grow * args.ldo + cbase;
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        uint4* o = reinterpret_cast<uint4*>(brow + 32 * ch);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t w4[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float a = bf16_round(__uint_as_float(v[ch][8 * i + 2 * h]) * alpha);
            const float b = bf16_round(__uint_as_float(v[ch][8 * i + 2 * h + 1]) * alpha);
            ss = fmaf(a, a, ss);
            ss = fmaf(b, b, ss);
            w4[h] = pack_bf16x2(a, b);
          }
          o[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
    } else {
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        float4* o = reinterpret_cast<float4*>(orow + cbase + 32 * ch);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 f = make_float4(__uint_as_float(v[ch][4 * i]) * alpha, __uint_as_float(v[ch][4 * i + 1]) * alpha,
                                       __uint_as_float(v[ch][4 * i + 2]) * alpha, __uint_as_float(v[ch][4 * i + 3]) * alpha);
          ss = fmaf(f.x, f.x, ss);
          ss = fmaf(f.y, f.y, ss);
          ss = fmaf(f.z, f.z, ss);
          ss = fmaf(f.w, f.w, ss);
          o[i] = f;
        }
      }
    }
    if (!split) args.ss[grow * args.ld_ss + cbase / BN] = ss;   // one sum per 128 columns
  }
}

// Epilogue of a gate/up tile (unsplit): SwiGLU of this warp's gate and up columns [c_lo,
// c_lo + kCols) of its TMEM lanes (tq), h = silu(ag acc_g) * (au acc_u) requantised to NVFP4 with
// scale 1 (codes by row; block-layout scales by M tile mt, as the next GEMM's A operand).
template <int BN, int kCols>
LMOE_DEV void epi_swiglu_quant(const Fp4Args& args, uint32_t tq, int c_lo, uint64_t* acc_empty, int lane, int n0,
                               float ag, float au, int mt, int r, long long grow, bool row_ok, const float* recip) {
  uint8_t* crow = static_cast<uint8_t*>(args.out) + grow * (args.ldo / 2);
  const int K_h = static_cast<int>(args.ldo);   // h is the next GEMM's A: scales by M tile
  // The whole accumulator slice is read first and the buffer handed back to the MMA
  // issuer before the SwiGLU, the requantisation and the stores: there is one gate+up
  // buffer, so the next tile's MMAs would otherwise wait for all of that (measured at
  // prefill: gate/up 0.90 ms, 0.78 ms in a timing build without the epilogue's work).
  constexpr int kCh = kCols / 32;
  uint32_t g[kCh][32], u[kCh][32];
#pragma unroll
  for (int ch = 0; ch < kCh; ++ch) {
    tmem_ld_32cols(tq + c_lo + 32 * ch, g[ch]);
    tmem_ld_32cols(tq + BN + c_lo + 32 * ch, u[ch]);
  }
  tmem_ld_wait();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(acc_empty);
#pragma unroll
  for (int ch = 0; ch < kCh; ++ch) {
    const int col = n0 + c_lo + 32 * ch;
    if (!(row_ok && col + 32 <= args.N)) continue;
    uint2 q[2];
    uint32_t sc[2];
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      float h[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a = __uint_as_float(g[ch][blk * 16 + i]) * ag;
        h[i] = __fdividef(a, 1.f + __expf(-a)) * (__uint_as_float(u[ch][blk * 16 + i]) * au);  // silu(a) * b
      }
      sc[blk] = nvfp4_quant16(h, 6.f, 1.f, recip, q[blk]);
    }
    *reinterpret_cast<uint4*>(crow + col / 2) = make_uint4(q[0].x, q[0].y, q[1].x, q[1].y);
    *reinterpret_cast<uint16_t*>(args.out_scales + blocked_sf_offset(mt, r, col / 16, K_h)) =
        static_cast<uint16_t>(sc[0] | (sc[1] << 8));
  }
}

template <int BN, int EPI, int AROWS>
__global__ void __launch_bounds__(Fp4Cfg<BN, EPI, AROWS>::kThreads, 1)
    gemm_fp4_kernel(const __grid_constant__ CUtensorMap tmA32, const __grid_constant__ CUtensorMap tmA64,
                    const __grid_constant__ CUtensorMap tmA96, const __grid_constant__ CUtensorMap tmA128,
                    const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
                    const Fp4Args args) {
  using C = Fp4Cfg<BN, EPI, AROWS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* recip = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(recip + 256);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;     // [kAccBufs]
  uint64_t* acc_empty = acc_full + 2;          // [kAccBufs], 4 epilogue warps arrive
  uint64_t* mma_done = acc_empty + 2;
  uint64_t* sf_full = mma_done + 1;            // [kStages] scales of the stage are in TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_full + C::kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Set-up reads nothing an earlier kernel of the stream writes: it runs before the wait,
  // with an L2 prefetch of this CTA's first weight tile (codes and scale blocks).
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], C::kEpiWarps);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
    prefetch_tmap(&tmA128);
    prefetch_tmap(&tmB);
    if (C::kDual) prefetch_tmap(&tmB2);
    int brow, kb0, kb1;
    if (first_tile_hint(args.tiles, args.n_tiles, args.max_tiles, args.n_groups, args.M, args.N, C::kTileN,
                        args.k_splits, args.num_kb, args.adaptive_splits != 0, brow, kb0, kb1)) {
      kb1 = min(kb1, kb0 + kPrefetchKb);
      const size_t sf0 = static_cast<size_t>(brow / BN) * args.num_kb * 4 * 512;
      for (int kb = kb0; kb < kb1; ++kb) {
        prefetch_l2_tile_2d(&tmB, kb * 128, brow);
        prefetch_l2_bulk(args.b_scales + sf0 + kb * 2048, 2048u);
        if (C::kWide) {   // the tile's second BN-row half of the same weights
          prefetch_l2_tile_2d(&tmB, kb * 128, brow + BN);
          prefetch_l2_bulk(args.b_scales + sf0 + static_cast<size_t>(args.num_kb) * 4 * 512 + kb * 2048, 2048u);
        } else if (C::kDual) {
          prefetch_l2_tile_2d(&tmB2, kb * 128, brow);
          prefetch_l2_bulk(args.b2_scales + sf0 + kb * 2048, 2048u);
        }
      }
    }
  }
  if (warp >= 2 && warp < C::kCopyWarp) {
    for (int i = threadIdx.x - 64; i < 256; i += 32 * C::kEpiWarps) recip[i] = g_e4m3_recip.v[i];
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
  const TileWalk walk(args.tiles, args.n_tiles, args.M, args.N, C::kTileN, args.k_splits, args.num_kb,
                      args.adaptive_splits != 0);
  if (args.splits_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0)
    *args.splits_out = walk.splits;
  const long long budget = args.budget;
  const int nk = args.num_kb;  // stages of K = 256

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer
      const uint64_t pol_b = args.b_stream_once ? policy_evict_first() : policy_evict_normal();
      const CUtensorMap* amap[4] = {&tmA32, &tmA64, &tmA96, &tmA128};  // A box of 32/64/96/128 rows
      const int kblk = args.num_kb * 4;   // 512-byte scale blocks per row block
      int it = 0;
      bool ok = true;
      TileRef cur = find_tile(walk, blockIdx.x);
      Tile ct = cur.valid ? tile_of(walk, cur.mt) : Tile{0, 0, 0, 0};
      while (ok && cur.valid) {
        // the next tile's table entry is loaded now and used after this tile has streamed
        const TileRef nxt = find_tile(walk, cur.id + gridDim.x);
        const Tile nt = nxt.valid ? tile_of(walk, nxt.mt) : Tile{0, 0, 0, 0};
        const int row0 = ct.row0;
        const int brow = ct.expert * args.N + cur.ntile * C::kTileN;
        // A rows past the live ones are not read; a tile beyond the variant's rows (a token
        // routed twice to one expert) is flagged, and its extra rows are left unwritten
        if (ct.nrows > AROWS) atomicOr(args.err, kErrBounds);
        const int abox = min(C::kABoxes, (ct.nrows + 31) / 32);
        const CUtensorMap* tA = amap[abox - 1];
        const uint32_t tx = C::tx_bytes(abox * 32);
        const uint8_t* sfa_src = args.a_scales + static_cast<size_t>(cur.mt) * kblk * 512;
        const uint8_t* sfb_src = args.b_scales + static_cast<size_t>(brow / BN) * kblk * 512;
        // second B box: the next BN rows of the same weights (wide tile), or the up weights
        const uint8_t* sfb2_src = C::kWide ? sfb_src + static_cast<size_t>(kblk) * 512
                                  : C::kDual ? args.b2_scales + static_cast<size_t>(brow / BN) * kblk * 512
                                             : nullptr;
        const CUtensorMap* tB2 = C::kWide ? &tmB : &tmB2;
        const int brow2 = C::kWide ? brow + BN : brow;
        int kb0, kb1;
        walk.k_range(cur.id, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          const int s = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, budget)) {
            atomicOr(args.err, kErrWaitProducer);
            ok = false;
            break;
          }
          uint8_t* st = smem + s * C::kStageBytes;
          mbar_arrive_expect_tx(&full[s], tx);
          tma_load_2d(st, tA, &full[s], kb * 128, row0);
          bulk_load(st + C::kOffSfa, sfa_src + kb * 2048, C::kSfaBytes, &full[s]);
          tma_load_2d_hint(st + C::kOffB, &tmB, &full[s], kb * 128, brow, pol_b);
          bulk_load(st + C::kOffSfb, sfb_src + kb * 2048, C::kSfbBytes, &full[s]);
          if (C::kDual) {
            tma_load_2d_hint(st + C::kOffB + C::kBBytes, tB2, &full[s], kb * 128, brow2, pol_b);
            bulk_load(st + C::kOffSfb + C::kSfbBytes, sfb2_src + kb * 2048, C::kSfbBytes, &full[s]);
          }
          ++it;
        }
        cur = nxt;
        ct = nt;
      }
      for (int j = max(0, it - C::kStages); j < it; ++j)
        if (!mbar_wait(&full[j % C::kStages], (j / C::kStages) & 1, kDrainBudget))
          atomicOr(args.err, kErrDrain);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer
      constexpr uint32_t idesc = idesc_nvf4(kBM, BN);
      int it = 0, tc = 0;
      bool ok = true;
      for (int id = blockIdx.x; ok && id < walk.n_ids; id += gridDim.x) {
        int expert, row0, nrows, ntile;
        if (!walk.at(id, expert, row0, nrows, ntile)) continue;
        const int buf = tc % C::kAccBufs;
        const uint32_t use = (tc / C::kAccBufs) & 1;
        if (!mbar_wait(&acc_empty[buf], use ^ 1, budget)) {
          atomicOr(args.err, kErrWaitMma);
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + buf * C::kAccCols;
        int kb0, kb1;
        walk.k_range(id, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          const int s = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          // the stage's codes have landed and the copier has put its scales in tensor memory
          if (!mbar_wait(&full[s], ph, budget) || !mbar_wait(&sf_full[s], ph, budget)) {
            atomicOr(args.err, kErrWaitMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * C::kStageBytes);
          const uint32_t sfa = tmem + C::kSfCol0 + s * C::kSfCols;
          const uint32_t sfb = sfa + C::kSfaCols;
#pragma unroll
          for (int j = 0; j < C::kKStep; ++j) {
            const uint64_t ad = sw128_kmajor_desc(st + j * 32);
            const uint32_t accum = (kb > kb0 || j > 0) ? 1u : 0u;
            mma_nvf4(acc, ad, sw128_kmajor_desc(st + C::kOffB + j * 32), idesc, sfa + j * 4,
                     sfb + j * 4, accum);
            if (C::kDual)
              mma_nvf4(acc + BN, ad, sw128_kmajor_desc(st + C::kOffB + C::kBBytes + j * 32), idesc,
                       sfa + j * 4, sfb + C::kSfbColsOne + j * 4, accum);
          }
          mma_commit(&empty[s]);
          ++it;
        }
        mma_commit(&acc_full[buf]);
        ++tc;
      }
      mma_commit(mma_done);
    }
  } else if (warp == C::kCopyWarp) {
    if (lane == 0) {
      // ---- scale-factor copier: the stage's A and B scale blocks into the stage's columns
      // (the slot is free again once the stage has been refilled: its previous MMAs completed
      // before the producer saw the stage empty)
      int it = 0;
      bool ok = true;
      for (int id = blockIdx.x; ok && id < walk.n_ids; id += gridDim.x) {
        int expert, row0, nrows, ntile;
        if (!walk.at(id, expert, row0, nrows, ntile)) continue;
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
          const uint32_t st = smem_u32(smem + s * C::kStageBytes);
          const uint32_t sfa = tmem + C::kSfCol0 + s * C::kSfCols;
          const uint32_t sfb = sfa + C::kSfaCols;
#pragma unroll
          for (int j = 0; j < C::kKStep; ++j) {
            tmem_cp_32x128b_x4(sfa + j * 4, sf_desc(st + C::kOffSfa + j * 512));
#pragma unroll
            for (int b = 0; b < C::kNB; ++b)
              tmem_cp_32x128b_x4(sfb + b * C::kSfbColsOne + j * 4,
                                 sf_desc(st + C::kOffSfb + b * C::kSfbBytes + j * 512));
          }
          mma_commit(&sf_full[s]);
          ++it;
        }
      }
      // every copy this thread issued has completed before the CTA tears down
      for (int j = max(0, it - C::kStages); j < it; ++j)
        if (!mbar_wait(&sf_full[j % C::kStages], (j / C::kStages) & 1, kDrainBudget))
          atomicOr(args.err, kErrDrain);
    }
  } else {
    // ---- epilogue: lane quadrant warp % 4; with 8 warps, column half (warp - 2) / 4
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quad * 32 + lane;
    constexpr int kCols = BN * 4 / C::kEpiWarps;
    const int c_lo = half * kCols, c_hi = c_lo + kCols;
    int tc = 0;
    for (int id = blockIdx.x; id < walk.n_ids; id += gridDim.x) {
      int mt, expert, row0, nrows, ntile;
      if (!walk.at(id, mt, expert, row0, nrows, ntile)) continue;
      const int buf = tc % C::kAccBufs;
      const uint32_t use = (tc / C::kAccBufs) & 1;
      if (!mbar_wait(&acc_full[buf], use, budget)) {
        atomicOr(args.err, kErrWaitEpilogue);
        break;
      }
      tc_fence_after();
      bool released = false;   // the accumulator buffer handed back before the stores
      const bool row_ok = r < min(nrows, AROWS);
      const long long grow = static_cast<long long>(row0) + r;
      const int n0 = ntile * C::kTileN;
      const uint32_t tq = tmem + buf * C::kAccCols + (static_cast<uint32_t>(quad * 32) << 16);
      const float rs = (args.row_scale != nullptr && row_ok) ? args.row_scale[grow] : 1.f;
      if constexpr (C::kWide) {
        epi_wide<BN, EPI>(args, tq, half, &acc_empty[buf], lane, n0,
                          rs * args.tensor_scale[args.tiles ? expert : 0],
                          walk.splits > 1 ? id % walk.splits : -1, grow, row_ok);
        released = true;
      } else if constexpr (EPI == kFp4EpiF32Ss || EPI == kFp4EpiBf16Ss) {
        const float alpha = rs * args.tensor_scale[args.tiles ? expert : 0];
        const bool split = walk.splits > 1;   // split-K: alpha * partial product (fp32), no ss
        // bf16 output (unsplit): the values are rounded and the sum of squares is taken of
        // the rounded values (LMSYS Muse Spark Open post, "Fused per-expert post-norm")
        const bool bf = EPI == kFp4EpiBf16Ss && !split;
        float* orow = split ? args.partial + (static_cast<long long>(id % walk.splits) * args.M + grow) * args.N
                            : static_cast<float*>(args.out) + grow * args.ldo;
        __nv_bfloat16* brow = static_cast<__nv_bfloat16*>(args.out) + grow * args.ldo;
        float ss = 0.f;
#pragma unroll 1
        for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32cols(tq + c0, v);
          tmem_ld_wait();
          const int col = n0 + c0;
          if (row_ok && col + 32 <= args.N) {
            if (bf) {
              uint4* o = reinterpret_cast<uint4*>(brow + col);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t w4[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  const float a = bf16_round(__uint_as_float(v[8 * i + 2 * h]) * alpha);
                  const float b = bf16_round(__uint_as_float(v[8 * i + 2 * h + 1]) * alpha);
                  ss = fmaf(a, a, ss);
                  ss = fmaf(b, b, ss);
                  w4[h] = pack_bf16x2(a, b);
                }
                o[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
              }
            } else {
              float4* o = reinterpret_cast<float4*>(orow + col);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 f = make_float4(__uint_as_float(v[4 * i]) * alpha, __uint_as_float(v[4 * i + 1]) * alpha,
                                             __uint_as_float(v[4 * i + 2]) * alpha, __uint_as_float(v[4 * i + 3]) * alpha);
                ss = fmaf(f.x, f.x, ss);
                ss = fmaf(f.y, f.y, ss);
                ss = fmaf(f.z, f.z, ss);
                ss = fmaf(f.w, f.w, ss);
                o[i] = f;
              }
            }
          }
        }
        if (row_ok && !split) args.ss[grow * args.ld_ss + ntile] = ss;
      } else {  // kFp4EpiSwiGLUQuant
        const int e = args.tiles ? expert : 0;
        const float ag = rs * args.tensor_scale[e], au = rs * args.tensor_scale2[e];
        // split-K: the scaled gate and up partial products, [splits][rows][2N] (gate | up)
        float* prow = walk.splits > 1
                          ? args.partial + (static_cast<long long>(id % walk.splits) * args.M + grow) * 2 * args.N
                          : nullptr;
        if (prow == nullptr) {
          epi_swiglu_quant<BN, kCols>(args, tq, c_lo, &acc_empty[buf], lane, n0, ag, au, mt, r, grow, row_ok, recip);
          released = true;
        } else {
#pragma unroll 1
        for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
          uint32_t g[32], u[32];
          tmem_ld_32cols(tq + c0, g);
          tmem_ld_32cols(tq + BN + c0, u);
          tmem_ld_wait();
          const int col = n0 + c0;
          {
            if (row_ok && col + 32 <= args.N) {
              float4* og = reinterpret_cast<float4*>(prow + col);
              float4* ou = reinterpret_cast<float4*>(prow + args.N + col);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                og[i] = make_float4(__uint_as_float(g[4 * i]) * ag, __uint_as_float(g[4 * i + 1]) * ag,
                                    __uint_as_float(g[4 * i + 2]) * ag, __uint_as_float(g[4 * i + 3]) * ag);
                ou[i] = make_float4(__uint_as_float(u[4 * i]) * au, __uint_as_float(u[4 * i + 1]) * au,
                                    __uint_as_float(u[4 * i + 2]) * au, __uint_as_float(u[4 * i + 3]) * au);
              }
            }
          }
        }
        }
      }
      if (!released) {   // every TMEM read of this buffer is complete: hand it back
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      }
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

LMOE_DEV void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

LMOE_DEV int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---- The expert pair of a few tokens: the grouped gate/up GEMM (SwiGLU, Q(h)) and the grouped
// down GEMM (bf16 y and its sums of squares) in one persistent launch.  Units: gate/up tiles
// (M tile mt, 128 h columns n), then down tiles (mt, 256 y columns n), each list M-tile major;
// CTA b takes units b, b + grid, b + 2 grid, ..., so its gate/up units all come before its down
// units, and the CTAs that finish their gate/up work first take the down units whose h rows
// are complete first.  A down unit reads the h rows of its M tile, complete once every gate/up
// unit of that tile has stored its columns: each epilogue warp adds 1 to the tile's ready count
// after its stores (release), and the producer waits for all of them (acquire, bounded) before
// the unit's first A copy.  One stage layout serves both: A box of 32 rows, two 128-row B boxes
// (gate and up, or the two halves of 256 down rows) and their scales.  The separate launches
// of the two GEMMs leave SMs idle twice, in the last wave of each (measured at the Muse shapes,
// hot-expert decode: 94.0 / 295.9 / 659.8 us per call at T = 1 / 8 / 32 with the two launches,
// 86.9 / 280.3 / 654.2 with the pair).  An L2 prefetch of each CTA's next down unit at the start
// of its previous unit made it slower (102.8 / 333.2 / 802.4 us): the prefetched lines compete
// with the streamed ones for L2 and are read twice.
__global__ void __launch_bounds__(Fp4Cfg<kBNFp4, kFp4EpiSwiGLUQuant, 32>::kThreads, 1)
    gemm_fp4_pair_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                         const __grid_constant__ CUtensorMap tmB1u, const __grid_constant__ CUtensorMap tmA2,
                         const __grid_constant__ CUtensorMap tmB2, const Fp4PairArgs pa) {
  constexpr int BN = kBNFp4;
  using C = Fp4Cfg<BN, kFp4EpiSwiGLUQuant, 32>;
  using CW = Fp4Cfg<BN, kFp4EpiBf16SsWide, 32>;
  static_assert(C::kStageBytes == CW::kStageBytes && C::kAccCols == CW::kAccCols && C::kEpiWarps == CW::kEpiWarps,
                "one stage and accumulator layout for both GEMMs");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* recip = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(recip + 256);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint64_t* sf_full = mma_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_full + C::kStages);
  const Fp4Args& gu = pa.gu;
  const Fp4Args& dn = pa.dn;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt1 = (gu.N + BN - 1) / BN, nt2 = (dn.N + 2 * BN - 1) / (2 * BN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], C::kEpiWarps);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
    prefetch_tmap(&tmA1);
    prefetch_tmap(&tmB1);
    prefetch_tmap(&tmB1u);
    prefetch_tmap(&tmA2);
    prefetch_tmap(&tmB2);
    // this CTA's first unit (a gate/up tile) into L2 before the wait: the tile table read as a
    // hint, clamped (the units computed come from the table read after the wait)
    const int tm = min(max(ld_relaxed_gpu(gu.n_tiles), 0), gu.max_tiles);
    const int u = static_cast<int>(blockIdx.x);
    if (u < tm * nt1) {
      const int e = ld_relaxed_gpu(&gu.tiles[u / nt1].expert);
      if (e >= 0 && e < gu.n_groups) {
        const int brow = e * gu.N + (u % nt1) * BN;
        const size_t sf0 = static_cast<size_t>(brow / BN) * gu.num_kb * 4 * 512;
        for (int kb = 0; kb < min(gu.num_kb, kPrefetchKb); ++kb) {
          prefetch_l2_tile_2d(&tmB1, kb * 128, brow);
          prefetch_l2_bulk(gu.b_scales + sf0 + kb * 2048, 2048u);
          prefetch_l2_tile_2d(&tmB1u, kb * 128, brow);
          prefetch_l2_bulk(gu.b2_scales + sf0 + kb * 2048, 2048u);
        }
      }
    }
  }
  if (warp >= 2 && warp < C::kCopyWarp) {
    for (int i = threadIdx.x - 64; i < 256; i += 32 * C::kEpiWarps) recip[i] = g_e4m3_recip.v[i];
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
  const int total_m = min(max(*gu.n_tiles, 0), gu.max_tiles);
  const int n1 = total_m * nt1, n_units = n1 + total_m * nt2;
  if (blockIdx.x == 0 && threadIdx.x == 0) {   // both GEMMs unsplit
    if (gu.splits_out != nullptr) *gu.splits_out = 1;
    if (dn.splits_out != nullptr) *dn.splits_out = 1;
  }
  // unit u: g = 0 gate/up, 1 down; its M tile and N tile
  auto unit_of = [&](int u, int& g, int& mt, int& ntile) {
    g = u >= n1 ? 1 : 0;
    const int v = g ? u - n1 : u, nt = g ? nt2 : nt1;
    mt = v / nt;
    ntile = v % nt;
  };
  const long long budget = gu.budget;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer
      const uint64_t pol_b = policy_evict_first();
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        int g, mt, ntile;
        unit_of(u, g, mt, ntile);
        const Tile t = pa.tiles[mt];
        const Fp4Args& A = g ? dn : gu;
        const int kblk = A.num_kb * 4;   // 512-byte scale blocks per 128-row block
        const int brow = t.expert * A.N + ntile * (g ? 2 * BN : BN);
        const int brow2 = g ? brow + BN : brow;
        const uint8_t* sfa_src = A.a_scales + static_cast<size_t>(mt) * kblk * 512;
        const uint8_t* sfb_src = A.b_scales + static_cast<size_t>(brow / BN) * kblk * 512;
        const uint8_t* sfb2_src = g ? sfb_src + static_cast<size_t>(kblk) * 512
                                    : gu.b2_scales + static_cast<size_t>(brow / BN) * kblk * 512;
        const CUtensorMap* tA = g ? &tmA2 : &tmA1;
        const CUtensorMap* tB = g ? &tmB2 : &tmB1;
        const CUtensorMap* tB2 = g ? &tmB2 : &tmB1u;
        if (t.nrows > 32) atomicOr(A.err, kErrBounds);   // rows past 32 are left unwritten
        if (g) {
          // the M tile's h rows: every gate/up epilogue warp of its nt1 units has counted them
          const int target = nt1 * C::kEpiWarps;
          const long long t0 = clock64();
          while (ld_acquire_gpu(&pa.tiles[mt].ready) < target) {
            if (clock64() - t0 > budget) {
              atomicOr(A.err, kErrWaitProducer);
              ok = false;
              break;
            }
            __nanosleep(64);
          }
          if (!ok) break;
          fence_proxy_async_global();   // written by generic stores, read by the copies below
        }
        const uint32_t tx = C::tx_bytes(32);
        for (int kb = 0; kb < A.num_kb; ++kb) {
          const int s = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, budget)) {
            atomicOr(A.err, kErrWaitProducer);
            ok = false;
            break;
          }
          uint8_t* st = smem + s * C::kStageBytes;
          mbar_arrive_expect_tx(&full[s], tx);
          tma_load_2d(st, tA, &full[s], kb * 128, t.row0);
          bulk_load(st + C::kOffSfa, sfa_src + kb * 2048, C::kSfaBytes, &full[s]);
          tma_load_2d_hint(st + C::kOffB, tB, &full[s], kb * 128, brow, pol_b);
          bulk_load(st + C::kOffSfb, sfb_src + kb * 2048, C::kSfbBytes, &full[s]);
          tma_load_2d_hint(st + C::kOffB + C::kBBytes, tB2, &full[s], kb * 128, brow2, pol_b);
          bulk_load(st + C::kOffSfb + C::kSfbBytes, sfb2_src + kb * 2048, C::kSfbBytes, &full[s]);
          ++it;
        }
      }
      for (int j = max(0, it - C::kStages); j < it; ++j)
        if (!mbar_wait(&full[j % C::kStages], (j / C::kStages) & 1, kDrainBudget))
          atomicOr(gu.err, kErrDrain);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer: the same two MMAs per K step for both GEMMs
      constexpr uint32_t idesc = idesc_nvf4(kBM, BN);
      int it = 0, tc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        int g, mt, ntile;
        unit_of(u, g, mt, ntile);
        const int nkb = g ? dn.num_kb : gu.num_kb;
        const int buf = tc % C::kAccBufs;
        const uint32_t use = (tc / C::kAccBufs) & 1;
        if (!mbar_wait(&acc_empty[buf], use ^ 1, budget)) {
          atomicOr(gu.err, kErrWaitMma);
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + buf * C::kAccCols;
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          if (!mbar_wait(&full[s], ph, budget) || !mbar_wait(&sf_full[s], ph, budget)) {
            atomicOr(gu.err, kErrWaitMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * C::kStageBytes);
          const uint32_t sfa = tmem + C::kSfCol0 + s * C::kSfCols;
          const uint32_t sfb = sfa + C::kSfaCols;
#pragma unroll
          for (int j = 0; j < C::kKStep; ++j) {
            const uint64_t ad = sw128_kmajor_desc(st + j * 32);
            const uint32_t accum = (kb > 0 || j > 0) ? 1u : 0u;
            mma_nvf4(acc, ad, sw128_kmajor_desc(st + C::kOffB + j * 32), idesc, sfa + j * 4, sfb + j * 4, accum);
            mma_nvf4(acc + BN, ad, sw128_kmajor_desc(st + C::kOffB + C::kBBytes + j * 32), idesc, sfa + j * 4,
                     sfb + C::kSfbColsOne + j * 4, accum);
          }
          mma_commit(&empty[s]);
          ++it;
        }
        mma_commit(&acc_full[buf]);
        ++tc;
      }
      mma_commit(mma_done);
    }
  } else if (warp == C::kCopyWarp) {
    if (lane == 0) {
      // ---- scale-factor copier
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        int g, mt, ntile;
        unit_of(u, g, mt, ntile);
        const int nkb = g ? dn.num_kb : gu.num_kb;
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          if (!mbar_wait(&full[s], ph, budget)) {
            atomicOr(gu.err, kErrWaitMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * C::kStageBytes);
          const uint32_t sfa = tmem + C::kSfCol0 + s * C::kSfCols;
          const uint32_t sfb = sfa + C::kSfaCols;
#pragma unroll
          for (int j = 0; j < C::kKStep; ++j) {
            tmem_cp_32x128b_x4(sfa + j * 4, sf_desc(st + C::kOffSfa + j * 512));
#pragma unroll
            for (int b = 0; b < C::kNB; ++b)
              tmem_cp_32x128b_x4(sfb + b * C::kSfbColsOne + j * 4, sf_desc(st + C::kOffSfb + b * C::kSfbBytes + j * 512));
          }
          mma_commit(&sf_full[s]);
          ++it;
        }
      }
      for (int j = max(0, it - C::kStages); j < it; ++j)
        if (!mbar_wait(&sf_full[j % C::kStages], (j / C::kStages) & 1, kDrainBudget))
          atomicOr(gu.err, kErrDrain);
    }
  } else {
    // ---- epilogue: lane quadrant warp % 4, column half (warp - 2) / 4
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quad * 32 + lane;
    constexpr int kCols = BN * 4 / C::kEpiWarps;
    const int c_lo = half * kCols;
    int tc = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      int g, mt, ntile;
      unit_of(u, g, mt, ntile);
      const Tile t = pa.tiles[mt];
      const int buf = tc % C::kAccBufs;
      const uint32_t use = (tc / C::kAccBufs) & 1;
      if (!mbar_wait(&acc_full[buf], use, budget)) {
        atomicOr(gu.err, kErrWaitEpilogue);
        break;
      }
      tc_fence_after();
      const bool row_ok = r < min(t.nrows, 32);
      const long long grow = static_cast<long long>(t.row0) + r;
      const uint32_t tq = tmem + buf * C::kAccCols + (static_cast<uint32_t>(quad * 32) << 16);
      if (g == 0) {
        const float rs = (gu.row_scale != nullptr && row_ok) ? gu.row_scale[grow] : 1.f;
        epi_swiglu_quant<BN, kCols>(gu, tq, c_lo, &acc_empty[buf], lane, ntile * BN, rs * gu.tensor_scale[t.expert],
                                    rs * gu.tensor_scale2[t.expert], mt, r, grow, row_ok, recip);
        // this warp's part of the tile's h rows is stored: counted for the down units (each
        // lane's stores fenced, then the count released by lane 0 after the warp's barrier)
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          atomicAdd(&pa.tiles[mt].ready, 1);
        }
      } else {
        const float rs = (dn.row_scale != nullptr && row_ok) ? dn.row_scale[grow] : 1.f;
        epi_wide<BN, kFp4EpiBf16SsWide>(dn, tq, half, &acc_empty[buf], lane, ntile * 2 * BN,
                                        rs * dn.tensor_scale[t.expert], -1, grow, row_ok);
      }
      ++tc;
    }
  }

  // ---- teardown: all MMAs of this CTA have completed before the columns are released
  if (warp == 1 && lane == 0)
    if (!mbar_wait(mma_done, 0, kDrainBudget)) atomicOr(gu.err, kErrDrain);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN, int EPI, int AROWS>
cudaError_t launch_fp4_one(const CUtensorMap* maps, const Fp4Args& a, int m_tiles, cudaStream_t s) {
  using C = Fp4Cfg<BN, EPI, AROWS>;
  auto kern = gemm_fp4_kernel<BN, EPI, AROWS>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long long ids = tile_id_bound(m_tiles, a.N, C::kTileN, a.k_splits > 1 ? a.k_splits : 1);
  if (ids == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(ids < sm_count() ? ids : sm_count());
  return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, maps[0], maps[1], maps[2], maps[3],
                    maps[4], maps[5], a);
}

template <int AROWS>
cudaError_t launch_fp4_rows(Fp4EpiKind epi, const CUtensorMap* maps, const Fp4Args& a, int m_tiles,
                            cudaStream_t s) {
  switch (epi) {
    case kFp4EpiF32Ss: return launch_fp4_one<kBNFp4, kFp4EpiF32Ss, AROWS>(maps, a, m_tiles, s);
    case kFp4EpiSwiGLUQuant: return launch_fp4_one<kBNFp4, kFp4EpiSwiGLUQuant, AROWS>(maps, a, m_tiles, s);
    case kFp4EpiBf16Ss: return launch_fp4_one<kBNFp4, kFp4EpiBf16Ss, AROWS>(maps, a, m_tiles, s);
    case kFp4EpiF32SsWide: return launch_fp4_one<kBNFp4, kFp4EpiF32SsWide, AROWS>(maps, a, m_tiles, s);
    case kFp4EpiBf16SsWide: return launch_fp4_one<kBNFp4, kFp4EpiBf16SsWide, AROWS>(maps, a, m_tiles, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm_fp4_pair(const CUtensorMap* maps, const Fp4PairArgs& a, int m_tiles, cudaStream_t s) {
  using C = Fp4Cfg<kBNFp4, kFp4EpiSwiGLUQuant, 32>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_fp4_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long long units = static_cast<long long>(m_tiles) *
                          ((a.gu.N + kBNFp4 - 1) / kBNFp4 + (a.dn.N + 2 * kBNFp4 - 1) / (2 * kBNFp4));
  if (units == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(units < sm_count() ? units : sm_count());
  return launch_pdl(gemm_fp4_pair_kernel, dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, maps[0], maps[1],
                    maps[2], maps[3], maps[4], a);
}

cudaError_t launch_gemm_fp4(Fp4EpiKind epi, const CUtensorMap* maps, const Fp4Args& a, int m_tiles,
                            int tile_rows, cudaStream_t s) {
  return tile_rows <= 32 ? launch_fp4_rows<32>(epi, maps, a, m_tiles, s)
                         : launch_fp4_rows<kBM>(epi, maps, a, m_tiles, s);
}

}  // namespace lmoe
