// internal.h — declarations shared by the library's translation units (not public).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace lmoe {

constexpr int kBM = 128;            // rows of one GEMM tile (tcgen05 M)
constexpr int kBK = 64;             // K elements of one pipeline stage (128 B of bf16)
constexpr int kBNWide = 256;        // N of the single-B GEMM tiles
constexpr int kBNSwiGLU = 128;      // N of each of the gate and up tiles
constexpr int kBNFp4 = 128;         // N of the NVFP4 tiles (each of gate and up for SwiGLU)
// K blocks of its first weight tile a dense GEMM CTA prefetches into L2 before it waits on
// the previous kernel
constexpr int kPrefetchKb = 64;
constexpr long long kDefaultWaitBudget = 4000000000LL;  // ~2 s of SM clock
constexpr long long kDrainBudget = 4000000000LL;        // waits for a CTA's own async work

// error-word bits written by device code
enum : uint32_t {
  kErrWaitProducer = 1u << 0,
  kErrWaitMma = 1u << 1,
  kErrWaitEpilogue = 1u << 2,
  kErrBadIndex = 1u << 3,
  kErrDrain = 1u << 4,
  kErrBounds = 1u << 5,   // routing structures failed validation (launch_validate_routing)
  kErrGridBarrier = 1u << 6,   // a grid barrier of the single-token kernel gave up waiting
};

enum EpiKind : int {
  kEpiF32 = 0,      // fp32 store (router logits)
  kEpiF32Ss = 1,    // fp32 store + per-row partial sum of squares of the stored values
  kEpiSwiGLU = 2,   // two accumulators a, b -> bf16 silu(a) * b
};

enum Fp4EpiKind : int {
  kFp4EpiF32Ss = 0,         // alpha * acc as fp32 + per-row partial sums of squares
  kFp4EpiSwiGLUQuant = 1,   // silu(alpha_g a) * (alpha_u b), requantised to NVFP4 (scale 1)
  kFp4EpiBf16Ss = 2,        // alpha * acc rounded to bf16 + partial sums of squares of the
                            // rounded values (the expert down projection's y)
  kFp4EpiF32SsWide = 3,     // as kFp4EpiF32Ss, with 128 x 256 output tiles (dense GEMMs of many
                            // rows: the two 128-row halves of the tile's weights per stage)
  kFp4EpiBf16SsWide = 4,    // as kFp4EpiBf16Ss, with 128 x 256 output tiles (the grouped down
                            // projection wherever it runs unsplit)
};

// One M tile of a grouped GEMM: rows [row0, row0 + nrows) of A, all of expert `expert`.
struct Tile {
  int expert, row0, nrows;
  // written as 0 with the tile; the expert-pair GEMM counts in it the gate/up epilogue warps
  // done with the tile's h rows (gemm_fp4.cu)
  int ready;
};

struct GemmArgs {
  int M;                   // rows of A when tiles == nullptr (dense tiling)
  int N;                   // output columns (rows of one expert's B)
  int num_kb;              // k-blocks of the reduction (K / kBK)
  int kb_period_a;         // A's k coordinate is (kb % kb_period_a) * kBK
  int kb_period_b;         // B's k coordinate is (kb % kb_period_b) * kBK
  const Tile* tiles;       // grouped tiles, or nullptr
  const int* n_tiles;      // number of valid grouped tiles (device)
  void* out;               // [rows, ldo] fp32 or bf16
  long long ldo;           // elements
  float* ss;               // [rows, ld_ss] partial sums of squares (kEpiF32Ss)
  int ld_ss;
  unsigned* err;           // device error word
  long long budget;        // wait budget, SM cycles
  int b_stream_once;       // B tiles are read by ~one M tile each: stream them evict-first
  int k_splits;            // > 1: split-K; the epilogue writes raw fp32 partial products
  float* partial;          // [k_splits][rows][N] (split-K), reduced by launch_splitk_reduce
  int max_tiles;           // grouped: capacity of the tile table
  int n_groups;            // grouped: experts (B holds n_groups * N rows)
  int xpose;               // fp32 stores through a per-warp transpose tile (many rows per tile;
                           // the launch then reserves the tile's shared memory)
};

struct Fp4Args {
  int M;                     // rows of A when tiles == nullptr
  int N;                     // output columns (rows of one expert's B)
  int num_kb;                // K / 256
  const Tile* tiles;
  const int* n_tiles;
  void* out;                 // fp32 [rows, ldo] (kFp4EpiF32Ss) or codes [rows, ldo/2] (quant)
  long long ldo;             // output row length in elements
  uint8_t* out_scales;       // quant: E4M3 block scales [rows, ldo/16]
  float* ss;                 // kFp4Epi*Ss: [rows, ld_ss] partial sums of squares
  int ld_ss;
  const float* row_scale;    // per A row fp32 scale, or nullptr (1)
  const float* tensor_scale; // per expert (grouped) or [0]: scale of B
  const float* tensor_scale2;// quant: scale of B2 (up)
  const uint8_t* a_scales;   // block-layout scales of A: row block = M tile (grouped) or row/128
  const uint8_t* b_scales;   // block-layout scales of B and B2 (row block = row / 128)
  const uint8_t* b2_scales;
  unsigned* err;
  long long budget;
  int b_stream_once;         // B tiles are read by ~one M tile each: stream them evict-first
  int k_splits;              // > 1: split-K; the epilogue writes alpha * partial products
  float* partial;            // [k_splits][rows][N] (split-K), reduced by launch_splitk_reduce
  // Grouped GEMMs only: with adaptive_splits, k_splits is an upper bound and the kernel picks
  // the split count from the live tile count (choose_splits, tiles.cuh); the count used is
  // stored at splits_out (if set), where the reduce kernel reads it.  SwiGLU partials hold
  // gate and up side by side: [splits][rows][2N].
  int adaptive_splits;
  int* splits_out;
  int max_tiles;             // grouped: capacity of the tile table
  int n_groups;              // grouped: experts (B holds n_groups * N rows)
};

// The grouped gate/up (kFp4EpiSwiGLUQuant) and down (kFp4EpiBf16SsWide) GEMMs of a few tokens
// as one persistent launch, both unsplit, every M tile of at most 32 rows; gu.out / gu.out_scales
// (h) are dn's A operand.  tiles: the table of gu and dn, writable (Tile::ready).  maps = {A of
// gu (box of 32 rows), gate codes, up codes, A of dn (h, box of 32 rows), down codes}.
struct Fp4PairArgs {
  Fp4Args gu, dn;
  Tile* tiles;
};
cudaError_t launch_gemm_fp4_pair(const CUtensorMap* maps, const Fp4PairArgs& a, int m_tiles, cudaStream_t s);

// NVFP4 GEMM; maps = {A codes with boxes of 32, 64, 96, 128 rows, B codes, B2 codes}; scales
// come from the Fp4Args pointers (block layout; B in blocks of the tile's N rows).  tile_rows
// bounds the rows of every M tile (at most 32: the variant with a 32-row A area per stage).
cudaError_t launch_gemm_fp4(Fp4EpiKind epi, const CUtensorMap* maps, const Fp4Args& a, int m_tiles,
                            int tile_rows, cudaStream_t s);

// NVFP4 row kernels (rowops.cu)
cudaError_t launch_prenorm_nvfp4(const void* x, bool x_f32, const float* g_pre, int T, int D,
                                 float eps, __nv_bfloat16* xa, int xa_cols, uint8_t* codes,
                                 uint8_t* scales, float* s_row, unsigned* status2, cudaStream_t s);
cudaError_t launch_poolnorm_scatter_nvfp4(const float* p, const float* ss_p, int ld_ss,
                                          const float* g_pool, const int32_t* row_of,
                                          const int32_t* idx, const int32_t* offsets,
                                          const int32_t* tile_base, int T, int L, int k, float eps,
                                          uint8_t* codes, uint8_t* scales, float* s_rows,
                                          cudaStream_t s);
// row-major E4M3 scales [rows, K/16] -> block layout with blocks of block_rows (64 or 128) rows
cudaError_t launch_nvfp4_block_scales(const uint8_t* src, long long rows, int K, int block_rows,
                                      uint8_t* dst, cudaStream_t s);
// y: [T*k, L] bf16 (y_bf16) or fp32
cudaError_t launch_combine_nvfp4(const void* y, bool y_bf16, const float* ss_y, int ld_ss,
                                 const int32_t* row_of, const int32_t* idx, const float* w,
                                 const float* g_expert, int T, int L, int k, float eps, uint8_t* codes,
                                 uint8_t* scales, float* s_row, cudaStream_t s);
cudaError_t launch_quantize_nvfp4(const float* src, long long rows, int K, bool row_scale,
                                  uint8_t* codes, uint8_t* scales, float* s_row, cudaStream_t s);

// Streaming multiprocessors of the current device (persistent grids).
int sm_count();

// Sums split-K partials [splits][rows][N] in split order into out [rows, ldo] (fp32, or bf16
// when out_bf16: then the sums of squares are those of the rounded values) and, when
// ss != nullptr, writes per-row partial sums of squares per group of `group` columns.  With
// splits_dev != nullptr the split count is read there on the device (adaptive grouped GEMMs)
// and `splits` is only its upper bound; a count of 1 means the GEMM wrote out itself.
cudaError_t launch_splitk_reduce(const float* partial, int splits, int rows, int N, void* out,
                                 long long ldo, float* ss, int ld_ss, int group, cudaStream_t s,
                                 const int* splits_dev = nullptr, bool out_bf16 = false);
// Grouped SwiGLU after an adaptive split-K gate/up GEMM: sums the [splits][rows][2N] partials
// (gate | up, already scaled), h = silu(gate) * up, quantised to NVFP4 with scale 1: codes
// [rows, N/2] and E4M3 block scales in the block layout of M tile `mt` (the h operand of the
// down GEMM).  Does nothing when the split count at splits_dev is 1.
cudaError_t launch_swiglu_reduce_nvfp4(const float* partial, const int* splits_dev, int rows, int N,
                                       const Tile* tiles, const int* n_tiles, int max_tiles,
                                       uint8_t* codes, uint8_t* scales, cudaStream_t s);

// Counts every kernel launch of the library (lmoe_kernel_launches).
void count_launch();

// Launches `kern` with programmatic stream serialisation and counts it; with cluster > 1
// also as clusters of `cluster` CTAs along x.  The kernel must call
// griddep_wait() (ptx.cuh) before it reads anything an earlier kernel of the stream wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Launches one persistent tcgen05 GEMM: out = A * B^T over m_tiles M tiles (an upper bound
// for grouped GEMMs) of 128 * m_halves rows (m_halves = 2: tiles of 256 rows, for many rows;
// a grouped GEMM then takes a table of 256-row tiles).
cudaError_t launch_gemm(EpiKind epi, const CUtensorMap& tmA, const CUtensorMap& tmB,
                        const CUtensorMap& tmB2, const GemmArgs& a, int m_tiles,
                        cudaStream_t s, int m_halves);

// Row kernels (rowops.cu).  The pre-norm kernels, the first of a call, also zero the two
// status words at status2 (error word, near-tie count) when status2 != nullptr.
cudaError_t launch_prenorm(const void* x, bool x_f32, const float* g_pre, int T, int D, float eps,
                           __nv_bfloat16* xa, int xa_cols, unsigned* status2, cudaStream_t s);
// S3 and S4 in one CTA for few (token, slot) pairs (route_small_fits); same outputs as
// launch_topk followed by launch_permute.
bool route_small_fits(int T, int k, int E);
// rsplits > 1: the logits are summed here from the router's split-K partials rpart
// [rsplits][T][E] (in split order, as the reduction kernel does) and written to `logits`.
cudaError_t launch_route_small(float* logits, int ld, const float* rpart, int rsplits, const float* bias,
                               const int32_t* forced,
                               int T, int E, int k, int32_t* idx, float* w, int32_t* near_tie,
                               int32_t* idx_copy, float* w_copy, unsigned* err, int32_t* counts,
                               int32_t* offsets, int32_t* row_of, int32_t* tok_of, Tile* tiles,
                               int32_t* n_tiles, int32_t* tile_base, Tile* tiles2, int32_t* n_tiles2,
                               cudaStream_t s);
cudaError_t launch_topk(const float* logits, int ld, const float* bias, const int32_t* forced,
                        int T, int E, int k, int32_t* idx, float* w, int32_t* near_tie,
                        int32_t* idx_copy, float* w_copy, unsigned* err, cudaStream_t s);
// tile_base (optional, [E]): first M tile of each expert in the tile table
// chunk_hist / chunk_base: [perm_chunks(T k)][E] int32 scratch; with them, from
// kPermChunkedMinPairs pairs the permutation runs chunked (histogram, scan, rank kernels)
// instead of one CTA per expert reading every id
constexpr int kPermChunkedMinPairs = 16384;   // below: too few chunks for the GPU (measured at 8192: slower)
int perm_chunks(long long pairs);
cudaError_t launch_permute(const int32_t* idx, int T, int k, int E, int32_t* counts,
                           int32_t* offsets, int32_t* row_of, int32_t* tok_of, Tile* tiles,
                           int32_t* n_tiles, cudaStream_t s, int32_t* tile_base = nullptr,
                           Tile* tiles2 = nullptr, int32_t* n_tiles2 = nullptr,
                           int32_t* chunk_hist = nullptr, int32_t* chunk_base = nullptr);
cudaError_t launch_poolnorm_scatter(const float* p, const float* ss_p, int ld_ss,
                                    const float* g_pool, const int32_t* row_of, int T, int L,
                                    int k, float eps, __nv_bfloat16* xe, cudaStream_t s);
cudaError_t launch_combine(const float* y, const float* ss_y, int ld_ss,
                           const int32_t* row_of, const int32_t* idx, const float* w,
                           const float* g_expert, int T, int L, int k, float eps,
                           __nv_bfloat16* c, cudaStream_t s);
// usplits > 1: u is summed here from the unpooler's split-K partials upart [usplits][T][D] and
// written to u, and the row's sum of squares is taken from it (ss_u is not read).  g_next:
// also next_out = RMSNorm(out) * g_next (out as stored), the next layer's pre-norm.
cudaError_t launch_postnorm_residual(const void* x, bool x_f32, float* u,
                                     const float* ss_u, int ld_ss, const float* g_post, int T,
                                     int D, float eps, void* out, bool out_f32, cudaStream_t s,
                                     const float* upart = nullptr, int usplits = 1,
                                     const float* g_next = nullptr, void* next_out = nullptr);
cudaError_t launch_wait_selftest(long long budget, unsigned* err, cudaStream_t s);

// ---- the single-token NVFP4 block as persistent kernels of one CTA per SM (decode_mk.cu)
constexpr int kDecodeMkMaxSmem = 225 * 1024;   // dynamic; the static part stays under 2 KB
struct DecodeMkWeight {
  const uint8_t* codes;        // [rows, K/2] E2M1 pairs
  const uint8_t* scales;       // E4M3 block scales, block layout of 128-row blocks
  const float* tensor_scale;   // [1] or [E]
};
struct DecodeMkArgs {
  const void* x;               // [D] bf16 or fp32 (x_f32)
  int x_f32;
  const __nv_bfloat16* W_router;   // [E, D]
  const float* router_bias;    // [E] or nullptr
  const int32_t* forced;       // [k] or nullptr
  const float *g_pre, *g_pool, *g_expert, *g_post;
  DecodeMkWeight w[5];         // pooler, gate, up, down, unpooler
  int D, L, E, I, k;
  float eps;
  void* out;                   // [D] bf16 or fp32 (out_f32)
  int out_f32;
  const float* g_next;         // [D] or nullptr: also next_out = RMSNorm(out as stored) * g_next
  void* next_out;
  // workspace (the block's layout at T = 1)
  __nv_bfloat16* xa;           // [2D] xn as bf16 hi | lo
  float* logits;               // [E]
  int32_t *topk_idx, *idx_copy, *near_tie, *counts, *offsets, *row_of, *tok_of, *n_tiles, *tile_base, *n_tiles2;
  float *topk_w, *w_copy;
  Tile *tiles, *tiles2;
  float* p;                    // [L]
  uint8_t* h_codes;            // [k][I/2] by slot
  uint8_t* h_scales;           // [k][I/16] E4M3 codes by slot
  __nv_bfloat16* y;            // [k][L], slot j at row row_of[j]
  float* u;                    // [D]
  float* ss_part;              // [k L/16 + D/4] sums of squares of 16 values of y, of 4 of u
  float* router_part;          // [rp][E] the logits over the rp parts of each router row
  unsigned* bar;               // grid barrier arrivals, zero at the launch
  unsigned* err;
  long long budget;
  // kDecodeMkFull: the whole block.  kDecodeMkPre: pre-norm, router, pooler, top-k and pool
  // norm, ending with Q(h0) written as the grouped gate/up GEMM's A rows (xe codes, block-layout
  // scales, row scales) for the k routed rows.  kDecodeMkPost: from the down GEMM's bf16 y and
  // its partial sums of squares ss_y (ld_ss_y per row): combine, unpooler, post-norm.
  int mode;
  int cooperative;             // launched cooperatively (else an ordinary grid of one CTA per SM)
  uint8_t* xe_codes;
  uint8_t* xe_scales;
  float* xe_rowscale;
  const float* ss_y;
  int ld_ss_y;
};
enum : int { kDecodeMkFull = 0, kDecodeMkPre = 1, kDecodeMkPost = 2 };
// Shapes the kernel takes: D, L, I multiples of 256 up to 8192, E <= 1024, k <= 16, and the
// shared memory it needs within kDecodeMkMaxSmem.
bool decode_megakernel_fits(int D, int L, int I, int E, int k);
size_t decode_megakernel_smem(int D, int L, int I, int E, int k);
long long decode_megakernel_scratch_floats(int D, int L, int E, int k);
// One launch of one CTA per SM; the caller zeroes *bar (and the status words) before it.
// Zeroes words[0, n) (n <= 32) after the previous kernel of the stream (decode_mk.cu).
cudaError_t launch_decode_clear(unsigned* words, int n, cudaStream_t s);
cudaError_t launch_decode_megakernel(const DecodeMkArgs& d, cudaStream_t s);
// Checks the routing structures one call left in its workspace: ids in [0, E); offsets start
// at 0, never decrease, end at R = T k and agree with counts; every pair's row lies in its
// expert's range and every row is the row of exactly one pair (row_of / tok_of: the scatter
// targets); every M tile (and 256-row tile) lies inside its expert's rows with 1..128 (256)
// rows, the tiles cover R rows, the tile counts are within the tables, and each expert's first
// tile (tile_base) is a tile of that expert.  A violation sets kErrBounds in *err; with
// `sanitize` the call's routing is also replaced by one that every later kernel reads in bounds
// (no tiles; every pair to row 0 of expert 0), so the rest of the call runs harmlessly.
cudaError_t launch_validate_routing(int32_t* idx, int T, int k, int E, const int32_t* counts, int32_t* offsets,
                                    int32_t* row_of, const int32_t* tok_of, const Tile* tiles, int32_t* n_tiles,
                                    int max_tiles, int32_t* tile_base, const Tile* tiles2, int32_t* n_tiles2,
                                    int max_tiles2, unsigned* err, bool sanitize, cudaStream_t s);
// fp32 weight [rows, K] -> bf16 [rows, parts*K]: part q is W_hi when bit q of lo_mask is 0,
// else W_lo = bf16(W - W_hi).  [hi | hi | lo] pairs with activations [x_hi | x_lo | x_hi];
// [hi | lo] pairs with one activation read twice.
cudaError_t launch_weight_split(const float* W, long long rows, int K, int parts,
                                unsigned lo_mask, __nv_bfloat16* dst, cudaStream_t s);

}  // namespace lmoe
