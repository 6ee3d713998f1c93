// api.cu — the C ABI of include/latent_moe.h: argument checks, workspace layout,
// TMA tensor maps, and the launch sequence of one latent-MoE block call.
//
// Launch sequence (one stream, no host synchronisation):
//   prenorm -> router GEMM (fp32 logits) -> top-k/softmax -> expert histogram +
//   stable scatter (expert-contiguous rows, M-tile table) -> pooler GEMM (+ row
//   sums of squares) -> pool norm, copied to the k expert rows -> grouped gate/up
//   GEMM with SwiGLU epilogue -> grouped down GEMM (+ per-expert row sums of
//   squares) -> combine (per-expert RMSNorm, routing weight, fp32 sum in slot
//   order) -> unpooler GEMM (+ row sums of squares) -> post-norm + residual.
// Grouped GEMMs read their tile table on the device, so per-expert row counts
// never travel to the host.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/latent_moe.h"
#include "internal.h"
#include "tiles.cuh"

using namespace lmoe;

namespace lmoe {
static std::atomic<unsigned long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace lmoe

namespace {

constexpr size_t kAlign = 256;
// Every workspace sub-buffer is followed by a guard band of LMOE_GUARD_BYTES that no kernel
// writes (lmoe_workspace_guards lists them): a write past the end of a sub-buffer lands there
// and shows as a changed canary.
constexpr size_t kGuard = LMOE_GUARD_BYTES;
constexpr int kMaxGuards = 64;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int cdiv(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

struct Layout {
  lmoe_workspace_layout pub;
  long long near_tie;
  long long tile_base;  // [E] first M tile of each expert
  long long partial;    // split-K partial products of the dense and grouped GEMMs
  long long partial_pool;  // the pooler's own (it may run beside the router on a side stream)
  long long splits_dev; // [2] split counts the grouped NVFP4 GEMMs chose (gate/up, down)
  long long tiles2, n_tiles2;  // table of 256-row tiles (BF16 grouped GEMMs of many rows)
  long long perm_hist, perm_base;  // [chunks][E] each: the chunked permutation of many pairs
  long long mk_scratch;  // single-token NVFP4 kernel: logit halves and sums of squares (or -1)
  // fp32-weight mode: bf16 copies of the weights
  long long w_router, w_pool, w_gate, w_up, w_down, w_unpool;
  long long x_stage, out_stage, host_io_total;
  int ld_logits, ld_ss_p, ld_ss_y, ld_ss_u, max_tiles, max_tiles2;
  long long guards[kMaxGuards];   // start of the guard band after each sub-buffer
  int n_guards;
};

// Upper bound of the split count of the grouped NVFP4 GEMMs (the kernel picks the count from
// the live tiles).  Split-K adds 8 bytes per partial element (write + read) on top of the
// weight stream; with R = T k rows each expert row block reads at least k of the E experts'
// weights, so the bound keeps the partial traffic a few percent of the weights'.
int grouped_max_splits(const lmoe_config* c) {
  if (c->weight_dtype != LMOE_NVFP4 || c->T <= 0) return 1;
  const long long sp = (c->d_latent / 128) / c->T;
  return sp >= 8 ? 8 : (sp < 1 ? 1 : static_cast<int>(sp));
}

// Split-K for dense GEMMs with few output tiles (small T): enough K ranges to give the 152
// SMs of a GB300 work, at least `min_kb` K blocks each, at most 32.  A fixed SM count keeps
// the workspace layout independent of the device a call runs on.
constexpr int kSplitSms = 152;

// The expert pair (lmoe_expert_pair): NVFP4, T <= 32, L a multiple of 256 and gate/up tiles
// for every SM of a GB300 (a token's k experts are distinct, so there are at least
// max(k, T k / 128) M tiles of I / 128 tiles each).
bool expert_pair_rule(const lmoe_config* c) {
  if (c->weight_dtype != LMOE_NVFP4 || c->T < 1 || c->T > 32 || c->d_latent % 256 != 0) return false;
  const long long R = 1LL * c->T * c->top_k;
  const long long lo_tiles = std::max<long long>(c->top_k, (R + kBM - 1) / kBM);
  return lo_tiles * ((c->d_ff + kBNFp4 - 1) / kBNFp4) >= kSplitSms;
}

// The pooler runs beside the router (side stream): at small T its split count is sized for
// about two thirds of the SMs, so that the router's CTAs find SMs of their own.
constexpr int kPoolerSms = 100;
// BF16 GEMMs with fp32 outputs store them through the epilogue's transpose tiles (whole-line
// stores) from this many rows per weight matrix (T for the dense GEMMs, R/E for the grouped
// ones); below it the tiles hold few rows and the smaller shared-memory footprint lets the next
// kernel's CTAs become resident beside the GEMM's
constexpr long long kXposeRows = 64;
int dense_splits(int T, int N, int bn, int num_kb, int min_kb, int sms = kSplitSms, int tile_rows = kBM) {
  const long long tiles = static_cast<long long>((T + tile_rows - 1) / tile_rows) * ((N + bn - 1) / bn);
  if (tiles == 0 || tiles * 2 >= sms) return 1;
  long long sp = sms / tiles;
  if (sp > num_kb / min_kb) sp = num_kb / min_kb;
  if (sp > 32) sp = 32;
  return sp < 1 ? 1 : static_cast<int>(sp);
}

struct DenseSplits {
  int router, pooler, unpool;
  int router_mh;   // M halves of the router's tiles
};
// The router's B (all experts' rows, K = 2D or 3D) is re-read by every M tile, so its tiles are
// bound by what an SM can take in; 256-row tiles, split along K to keep every SM busy, halve
// that traffic per row.  Measured on GB300 (E = 256, D = 8192): faster at 4096 tokens (the
// router stage 58 -> 52 us), slower at 1024 (more splits than K blocks allow) and at 16384
// (2 splits: the partials' round trip costs more than the tiles save).
constexpr int kRouterWideMinT = 2048, kRouterWideMaxT = 8192;
DenseSplits dense_split_plan(const lmoe_config* c) {
  const bool f32w = c->weight_dtype == LMOE_F32, fp4 = c->weight_dtype == LMOE_NVFP4;
  const int D = c->d_model, L = c->d_latent;
  const int xa_cols = (f32w ? 3 : 2) * D, wsplit = f32w ? 2 : 1;
  DenseSplits d;
  d.router_mh = c->T >= kRouterWideMinT && c->T <= kRouterWideMaxT ? 2 : 1;
  d.router = dense_splits(c->T, c->n_experts, kBNWide, xa_cols / kBK, 4, kSplitSms, kBM * d.router_mh);
  if (fp4) {
    d.pooler = dense_splits(c->T, L, kBNFp4, D / 256, 2, kPoolerSms);
    d.unpool = dense_splits(c->T, D, kBNFp4, L / 256, 2);
  } else {
    d.pooler = dense_splits(c->T, L, kBNWide, (f32w ? 3 * D : D) / kBK, 4, kPoolerSms);
    d.unpool = dense_splits(c->T, D, kBNWide, wsplit * L / kBK, 4);
  }
  return d;
}

lmoe_status check_config(const lmoe_config* c) {
  if (c == nullptr) return LMOE_ERR_ARG;
  if (c->T < 0 || c->T > (1 << 20)) return LMOE_ERR_ARG;
  if (c->d_model <= 0 || c->d_latent <= 0 || c->d_ff <= 0 || c->n_experts <= 0)
    return LMOE_ERR_ARG;
  if (c->top_k < 1 || c->top_k > 16 || c->top_k > c->n_experts) return LMOE_ERR_ARG;
  if (c->n_experts > 1024) return LMOE_ERR_UNSUPPORTED;
  if (c->d_model % 128 || c->d_latent % 128 || c->d_ff % 128) return LMOE_ERR_UNSUPPORTED;
  if (c->d_model > 65536 || c->d_latent > 65536 || c->d_ff > 65536) return LMOE_ERR_UNSUPPORTED;
  if (!(c->eps >= 0.f)) return LMOE_ERR_ARG;
  if (c->act_dtype != LMOE_F32 && c->act_dtype != LMOE_BF16) return LMOE_ERR_UNSUPPORTED;
  if (c->out_dtype != LMOE_F32 && c->out_dtype != LMOE_BF16) return LMOE_ERR_UNSUPPORTED;
  if (c->weight_dtype != LMOE_F32 && c->weight_dtype != LMOE_BF16 && c->weight_dtype != LMOE_NVFP4)
    return LMOE_ERR_UNSUPPORTED;
  if (c->weight_dtype == LMOE_NVFP4) {
    // NVFP4 GEMM stages cover K = 256; the quantising row kernels hold one row in smem
    if (c->d_model % 256 || c->d_latent % 256 || c->d_ff % 256) return LMOE_ERR_UNSUPPORTED;
    if (c->d_model > 32768 || c->d_latent > 32768 || c->d_ff > 32768) return LMOE_ERR_UNSUPPORTED;
  }
  return LMOE_OK;
}

void make_layout(const lmoe_config* c, Layout* L) {
  const long long T = c->T, D = c->d_model, Ld = c->d_latent, E = c->n_experts, I = c->d_ff,
                  k = c->top_k, R = T * k;
  const bool f32w = c->weight_dtype == LMOE_F32;
  size_t off = 0;
  memset(L, 0xff, sizeof(*L));
  L->n_guards = 0;
  auto take = [&](size_t bytes) -> long long {
    const long long o = static_cast<long long>(off);
    off = align_up(off + bytes, kAlign);
    if (L->n_guards < kMaxGuards) L->guards[L->n_guards++] = static_cast<long long>(off);
    off += kGuard;
    return o;
  };
  lmoe_workspace_layout& P = L->pub;
  P.xa_cols = static_cast<int>((f32w ? 3 : 2) * D);
  L->ld_logits = static_cast<int>(align_up(E, 32));
  const int bn_ss = 128;   // the GEMM epilogues write one row sum of squares per 128 columns
  L->ld_ss_p = cdiv(Ld, bn_ss);
  L->ld_ss_y = cdiv(Ld, bn_ss);
  L->ld_ss_u = cdiv(D, bn_ss);
  L->max_tiles = cdiv(R, kBM) + static_cast<int>(E < R ? E : R);
  L->max_tiles2 = cdiv(R, 2 * kBM) + static_cast<int>(E < R ? E : R);
  P.err = take(kAlign);  // error word; the near-tie counter and the single-token kernels' grid
                         // barrier counters (words 2 and 3) share this line
  L->near_tie = P.err + 4;
  P.xa = take(T * P.xa_cols * 2);
  P.logits = take(T * L->ld_logits * 4);
  P.topk_idx = take(R * 4);
  P.topk_w = take(R * 4);
  P.counts = take(E * 4);
  P.offsets = take((E + 1) * 4);
  P.row_of = take(R * 4);
  P.tok_of = take(R * 4);
  P.tiles = take(static_cast<size_t>(L->max_tiles) * sizeof(Tile));
  P.n_tiles = take(4);
  L->tile_base = take(E * 4);
  L->tiles2 = take(static_cast<size_t>(L->max_tiles2) * sizeof(Tile));
  L->n_tiles2 = take(4);
  L->perm_hist = take(static_cast<size_t>(perm_chunks(R)) * E * 4);
  L->perm_base = take(static_cast<size_t>(perm_chunks(R)) * E * 4);
  P.p = take(T * Ld * 4);
  P.ss_p = take(T * L->ld_ss_p * 4);
  const bool fp4 = c->weight_dtype == LMOE_NVFP4;
  // NVFP4 block scales are kept in the tensor cores' block layout: whole 128-row blocks, one
  // per 128 rows of a dense operand, one per M tile of a grouped one
  const long long tb = cdiv(T, kBM) * static_cast<long long>(kBM);
  const long long gb = static_cast<long long>(L->max_tiles) * kBM;
  if (fp4) {  // quantised GEMM inputs: codes (2 per byte), E4M3 block scales, fp32 row scales
    P.xq = take(T * D / 2);
    P.xq_scale = take(tb * D / 16);
    P.xq_rowscale = take(T * 4);
    P.xe = take(R * Ld / 2);
    P.xe_scale = take(gb * Ld / 16);
    P.xe_rowscale = take(R * 4);
    P.h = take(R * I / 2);
    P.h_scale = take(gb * I / 16);
  } else {
    P.xe = take(R * Ld * 2);
    P.h = take(R * I * 2);
  }
  P.y = take(R * Ld * (fp4 ? 2 : 4));   // bf16 with NVFP4 weights, fp32 otherwise
  P.ss_y = take(R * L->ld_ss_y * 4);
  if (fp4) {
    P.c = take(T * Ld / 2);
    P.c_scale = take(tb * Ld / 16);
    P.c_rowscale = take(T * 4);
  } else {
    P.c = take(T * Ld * 2);
  }
  P.u = take(T * D * 4);
  P.ss_u = take(T * L->ld_ss_u * 4);
  if (f32w) {  // bf16 hi/lo splits of fp32 weights: [hi|hi|lo] (router, pooler), [hi|lo] (rest)
    L->w_router = take(E * 3 * D * 2);
    L->w_pool = take(Ld * 3 * D * 2);
    L->w_gate = take(E * I * 2 * Ld * 2);
    L->w_up = take(E * I * 2 * Ld * 2);
    L->w_down = take(E * Ld * 2 * I * 2);
    L->w_unpool = take(D * 2 * Ld * 2);
  }
  {  // split-K partials: the largest of the router's and unpooler's [splits][T][N] and the
     // grouped GEMMs' [splits][R][2I] (gate | up) and [splits][R][L]; the pooler's apart
    const DenseSplits d = dense_split_plan(c);
    long long need = 0;
    if (d.router > 1) need = std::max(need, d.router * T * E);
    if (d.unpool > 1) need = std::max(need, d.unpool * T * D);
    L->partial_pool = d.pooler > 1 ? take(d.pooler * T * Ld * 4) : -1;
    const long long gs = grouped_max_splits(c);
    if (gs > 1) need = std::max(need, gs * R * std::max(2 * I, Ld));
    L->partial = need > 0 ? take(need * 4) : -1;
    L->splits_dev = take(2 * 4);
    P.grouped_splits = c->weight_dtype == LMOE_NVFP4 ? L->splits_dev : -1;
  }
  // one token with NVFP4 weights runs through the persistent kernels of decode_mk.cu where they fit
  L->mk_scratch = fp4 && T == 1 && decode_megakernel_fits(static_cast<int>(D), static_cast<int>(Ld),
                                                          static_cast<int>(I), static_cast<int>(E),
                                                          static_cast<int>(k))
                      ? take(decode_megakernel_scratch_floats(static_cast<int>(D), static_cast<int>(Ld),
                                                              static_cast<int>(E), static_cast<int>(k)) * 4)
                      : -1;
  P.total = static_cast<long long>(off);
  L->x_stage = take(T * D * (c->act_dtype == LMOE_F32 ? 4 : 2));
  L->out_stage = take(T * D * (c->out_dtype == LMOE_F32 ? 4 : 2));
  L->host_io_total = static_cast<long long>(off);
}

// ------------------------------------------------------------------ tensor maps
// cuTensorMapEncodeTiled is a driver entry point; it is resolved through the runtime
// once per process so the library does not link libcuda directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode_bf16_2d(CUtensorMap* m, const void* base, unsigned long long cols,
                    unsigned long long rows, unsigned long long row_stride_bytes,
                    unsigned box_cols, unsigned box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const CUresult r = enc(
      m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D uint8 map (NVFP4 codes or block scales): [rows, cols] bytes, rows `row_stride` apart.
bool encode_u8_2d(CUtensorMap* m, const void* base, unsigned long long cols, unsigned long long rows,
                  unsigned long long row_stride, unsigned box_cols, unsigned box_rows, bool swizzle) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_stride};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define LMOE_CUDA(call)                       \
  do {                                        \
    if ((call) != cudaSuccess) return LMOE_ERR_CUDA; \
  } while (0)

lmoe_status run_gemm(EpiKind epi, const void* A, long long a_rows, long long a_cols_used,
                     long long a_row_stride_elems, const void* B, long long b_rows,
                     long long b_cols, const void* B2, int N, int num_kb,
                     const Tile* tiles, const int* n_tiles, int m_tiles, void* out,
                     long long ldo, float* ss, int ld_ss, unsigned* err, long long budget,
                     cudaStream_t s, long long rows_per_b, int splits = 1,
                     float* partial = nullptr, int m_halves = 1, bool reduce = true) {
  const unsigned bn = epi == kEpiSwiGLU ? kBNSwiGLU : kBNWide;
  CUtensorMap ta, tb, tb2;
  if (!encode_bf16_2d(&ta, A, a_cols_used, a_rows, a_row_stride_elems * 2, kBK, kBM))
    return LMOE_ERR_CUDA;
  if (!encode_bf16_2d(&tb, B, b_cols, b_rows, b_cols * 2, kBK, bn)) return LMOE_ERR_CUDA;
  tb2 = tb;
  if (B2 && !encode_bf16_2d(&tb2, B2, b_cols, b_rows, b_cols * 2, kBK, bn)) return LMOE_ERR_CUDA;
  GemmArgs a{};
  a.M = static_cast<int>(a_rows);
  a.N = N;
  a.num_kb = num_kb;
  a.kb_period_a = static_cast<int>(a_cols_used / kBK);
  a.kb_period_b = static_cast<int>(b_cols / kBK);
  a.tiles = tiles;
  a.n_tiles = n_tiles;
  a.out = out;
  a.ldo = ldo;
  a.ss = ss;
  a.ld_ss = ld_ss;
  a.err = err;
  a.budget = budget;
  // evict-first only where (nearly) every B tile meets one M tile: at a mean near kBM rows
  // per expert, many experts spill into a second M tile that re-reads B from L2
  a.b_stream_once = rows_per_b <= kBM / 2;
  a.k_splits = splits > 1 ? splits : 1;
  a.partial = partial;
  a.max_tiles = m_tiles;
  a.n_groups = static_cast<int>(b_rows / N);
  a.xpose = epi != kEpiSwiGLU && rows_per_b >= kXposeRows ? 1 : 0;   // fp32 outputs only
  LMOE_CUDA(launch_gemm(epi, ta, tb, tb2, a, m_tiles, s, m_halves));
  if (splits > 1 && reduce)   // else the consumer sums the partials
    LMOE_CUDA(launch_splitk_reduce(partial, splits, static_cast<int>(a_rows), N, static_cast<float*>(out),
                                   ldo, ss, ld_ss, 128, s));
  return LMOE_OK;
}

// One NVFP4 operand: codes [rows, K/2] and block scales [rows, K/16], both K contiguous.
struct Fp4Operand {
  const uint8_t* codes;
  const uint8_t* scales;
};

lmoe_status run_gemm_fp4(Fp4EpiKind epi, Fp4Operand A, long long a_rows, int K, Fp4Operand B,
                         long long b_rows, const Fp4Operand* B2, int N, const Tile* tiles,
                         const int* n_tiles, int m_tiles, void* out, long long ldo,
                         uint8_t* out_scales, float* ss, int ld_ss, const float* row_scale,
                         const float* ts, const float* ts2, unsigned* err, long long budget,
                         cudaStream_t s, long long rows_per_b, int tile_rows, int splits = 1,
                         float* partial = nullptr, int* splits_dev = nullptr,
                         bool reduce = true) {
  CUtensorMap maps[6];
  const unsigned long long kc = K / 2;
  const unsigned bn = kBNFp4;
  for (int i = 0; i < 4; ++i)  // A boxes of 32, 64, 96, 128 rows (the tile's live rows)
    if (!encode_u8_2d(&maps[i], A.codes, kc, a_rows, kc, 128, 32 * (i + 1), true)) return LMOE_ERR_CUDA;
  if (!encode_u8_2d(&maps[4], B.codes, kc, b_rows, kc, 128, bn, true)) return LMOE_ERR_CUDA;
  maps[5] = maps[4];
  if (B2 && !encode_u8_2d(&maps[5], B2->codes, kc, b_rows, kc, 128, bn, true)) return LMOE_ERR_CUDA;
  Fp4Args a{};
  a.M = static_cast<int>(a_rows);
  a.N = N;
  a.num_kb = K / 256;
  a.tiles = tiles;
  a.n_tiles = n_tiles;
  a.out = out;
  a.ldo = ldo;
  a.out_scales = out_scales;
  a.ss = ss;
  a.ld_ss = ld_ss;
  a.row_scale = row_scale;
  a.tensor_scale = ts;
  a.tensor_scale2 = ts2;
  a.a_scales = A.scales;
  a.b_scales = B.scales;
  a.b2_scales = B2 ? B2->scales : nullptr;
  a.err = err;
  a.budget = budget;
  // evict-first only where (nearly) every B tile meets one M tile: at a mean near kBM rows
  // per expert, many experts spill into a second M tile that re-reads B from L2
  a.b_stream_once = rows_per_b <= kBM / 2;
  a.k_splits = splits > 1 ? splits : 1;
  a.partial = partial;
  a.max_tiles = m_tiles;
  a.n_groups = static_cast<int>(b_rows / N);
  // grouped: `splits` bounds the count the kernel picks and leaves at splits_dev
  const bool adaptive = tiles != nullptr && splits > 1;
  a.adaptive_splits = adaptive ? 1 : 0;
  a.splits_out = tiles != nullptr ? splits_dev : nullptr;
  if (adaptive && (partial == nullptr || splits_dev == nullptr)) return LMOE_ERR_WORKSPACE;
  LMOE_CUDA(launch_gemm_fp4(epi, maps, a, m_tiles, tile_rows, s));
  if (splits > 1 && reduce) {   // else the consumer sums the partials
    if (epi == kFp4EpiSwiGLUQuant)
      LMOE_CUDA(launch_swiglu_reduce_nvfp4(partial, splits_dev, static_cast<int>(a_rows), N, tiles,
                                           n_tiles, m_tiles, static_cast<uint8_t*>(out), out_scales, s));
    else
      LMOE_CUDA(launch_splitk_reduce(partial, splits, static_cast<int>(a_rows), N, out, ldo, ss, ld_ss, 128, s,
                                     adaptive ? splits_dev : nullptr,
                                     epi == kFp4EpiBf16Ss || epi == kFp4EpiBf16SsWide));
  }
  return LMOE_OK;
}

// The grouped gate/up and down GEMMs of a few tokens (every M tile at most 32 rows) as one
// launch: xe (R rows, K = Ld) times the gate and up weights into h (codes and block-layout
// scales, the down GEMM's A), then h (K = I) times the down weights into bf16 y with its sums
// of squares per 128 columns.  Both unsplit; the split counts left for inspection are 1.
lmoe_status run_gemm_fp4_pair(Fp4Operand xe, const float* xe_s, Fp4Operand gate, Fp4Operand up, Fp4Operand down,
                              const float* ts_g, const float* ts_u, const float* ts_d, long long R, int Ld, int I,
                              long long E, Tile* tiles, const int* n_tiles, int m_tiles, uint8_t* h, uint8_t* h_scales,
                              void* y, float* ss_y, int ld_ss_y, int* splits_dev, unsigned* err,
                              long long budget, cudaStream_t s) {
  CUtensorMap maps[5];
  const unsigned long long k1 = Ld / 2, k2 = I / 2;
  if (!encode_u8_2d(&maps[0], xe.codes, k1, R, k1, 128, 32, true) ||
      !encode_u8_2d(&maps[1], gate.codes, k1, E * I, k1, 128, kBNFp4, true) ||
      !encode_u8_2d(&maps[2], up.codes, k1, E * I, k1, 128, kBNFp4, true) ||
      !encode_u8_2d(&maps[3], h, k2, R, k2, 128, 32, true) ||
      !encode_u8_2d(&maps[4], down.codes, k2, E * Ld, k2, 128, kBNFp4, true))
    return LMOE_ERR_CUDA;
  Fp4PairArgs a{};
  Fp4Args& g = a.gu;
  g.M = static_cast<int>(R);
  g.N = I;
  g.num_kb = Ld / 256;
  g.tiles = tiles;
  g.n_tiles = n_tiles;
  g.out = h;
  g.ldo = I;
  g.out_scales = h_scales;
  g.row_scale = xe_s;
  g.tensor_scale = ts_g;
  g.tensor_scale2 = ts_u;
  g.a_scales = xe.scales;
  g.b_scales = gate.scales;
  g.b2_scales = up.scales;
  g.err = err;
  g.budget = budget;
  g.b_stream_once = 1;
  g.k_splits = 1;
  g.splits_out = splits_dev;
  g.max_tiles = m_tiles;
  g.n_groups = static_cast<int>(E);
  Fp4Args& d = a.dn;
  d.M = static_cast<int>(R);
  d.N = Ld;
  d.num_kb = I / 256;
  d.tiles = tiles;
  d.n_tiles = n_tiles;
  d.out = y;
  d.ldo = Ld;
  d.ss = ss_y;
  d.ld_ss = ld_ss_y;
  d.tensor_scale = ts_d;
  d.a_scales = h_scales;
  d.b_scales = down.scales;
  d.err = err;
  d.budget = budget;
  d.b_stream_once = 1;
  d.k_splits = 1;
  d.splits_out = splits_dev != nullptr ? splits_dev + 1 : nullptr;
  d.max_tiles = m_tiles;
  d.n_groups = static_cast<int>(E);
  a.tiles = tiles;
  LMOE_CUDA(launch_gemm_fp4_pair(maps, a, m_tiles, s));
  return LMOE_OK;
}

// ------------------------------------------------------------------ side stream
// The pooler reads only the pre-norm output, so it runs on a side stream while the router,
// top-k and permutation run on the caller's stream (all three are latency-bound at small T).
// One side stream and one fork/join event pair per device; the mutex keeps a fork, the
// pooler and the matching join of one call together when several host threads call at once.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex mu;
  bool ok = false;
};
constexpr int kMaxDevices = 64;

SideStream* side_stream() {
  static SideStream side[kMaxDevices];
  static std::once_flag once[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream& ss = side[dev];
  std::call_once(once[dev], [&ss] {
    ss.ok = cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) == cudaSuccess;
  });
  return ss.ok ? &ss : nullptr;
}

lmoe_status forward_impl(const lmoe_config* cfg, const void* x, const void* W_router,
                         const void* W_pool, const float* g_pool, const void* W_gate,
                         const void* W_up, const void* W_down, const float* g_expert,
                         const void* W_unpool, const float* g_pre, const float* g_post,
                         int top_k, void* out, void* workspace, size_t ws_bytes, cudaStream_t s,
                         const lmoe_ex* ex) {
  lmoe_status st = check_config(cfg);
  if (st != LMOE_OK) return st;
  if (top_k != cfg->top_k) return LMOE_ERR_ARG;
  if (ex != nullptr && (ex->next_norm_gamma == nullptr) != (ex->next_norm_out == nullptr)) return LMOE_ERR_ARG;
  if (ex != nullptr && (ex->single_token_path < LMOE_SINGLE_TOKEN_DEFAULT || ex->single_token_path > LMOE_SINGLE_TOKEN_CHAIN))
    return LMOE_ERR_ARG;
  if (ex != nullptr && ex->next_norm_out != nullptr &&
      (!aligned16(ex->next_norm_out) || !aligned16(ex->next_norm_gamma)))
    return LMOE_ERR_ALIGN;
  if (cfg->T == 0) {  // no rows: nothing is read; only the error word is cleared
    Layout L0;
    make_layout(cfg, &L0);
    if (workspace != nullptr && ws_bytes >= static_cast<size_t>(L0.pub.total))
      LMOE_CUDA(cudaMemsetAsync(static_cast<char*>(workspace) + L0.pub.err, 0, 8, s));
    return LMOE_OK;
  }
  const void* ptrs[] = {x, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert,
                        W_unpool, g_pre, g_post, out};
  for (const void* p : ptrs)
    if (p == nullptr) return LMOE_ERR_ARG;
  const bool fp4 = cfg->weight_dtype == LMOE_NVFP4;
  // NVFP4 weights arrive as host structs of device pointers: check what they point to
  const lmoe_nvfp4_weight* q4[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  if (fp4) {
    const void* wv[5] = {W_pool, W_gate, W_up, W_down, W_unpool};
    for (int i = 0; i < 5; ++i) {
      q4[i] = static_cast<const lmoe_nvfp4_weight*>(wv[i]);
      if (!q4[i]->data || !q4[i]->scales || !q4[i]->tensor_scale) return LMOE_ERR_ARG;
      // the kernels read the block layout only: row-major scales must be converted first
      if (q4[i]->scale_layout != LMOE_NVFP4_SCALES_BLOCKED) return LMOE_ERR_UNSUPPORTED;
      if (!aligned16(q4[i]->data) || !aligned16(q4[i]->scales) || !aligned16(q4[i]->tensor_scale))
        return LMOE_ERR_ALIGN;
    }
  }
  for (const void* p : ptrs) {
    const bool host_struct = fp4 && (p == W_pool || p == W_gate || p == W_up || p == W_down ||
                                     p == W_unpool);
    if (!host_struct && !aligned16(p)) return LMOE_ERR_ALIGN;
  }
  if (x == out) return LMOE_ERR_ARG;
  Layout L;
  make_layout(cfg, &L);
  if (workspace == nullptr || ws_bytes < static_cast<size_t>(L.pub.total)) return LMOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return LMOE_ERR_ALIGN;
  if (ex && ex->router_bias && !aligned16(ex->router_bias)) return LMOE_ERR_ALIGN;

  const int T = cfg->T, D = cfg->d_model, Ld = cfg->d_latent, E = cfg->n_experts,
            I = cfg->d_ff, k = cfg->top_k;
  const long long R = static_cast<long long>(T) * k;
  const float eps = cfg->eps;
  const bool x_f32 = cfg->act_dtype == LMOE_F32, f32w = cfg->weight_dtype == LMOE_F32;
  const long long budget =
      (ex && ex->wait_budget_cycles > 0) ? ex->wait_budget_cycles : kDefaultWaitBudget;
  char* ws = static_cast<char*>(workspace);
  auto at = [&](long long o) { return static_cast<void*>(ws + o); };
  unsigned* err = static_cast<unsigned*>(at(L.pub.err));
  int32_t* near_tie = static_cast<int32_t*>(at(L.near_tie));
  __nv_bfloat16* xa = static_cast<__nv_bfloat16*>(at(L.pub.xa));
  float* logits = static_cast<float*>(at(L.pub.logits));
  int32_t* tk_idx = static_cast<int32_t*>(at(L.pub.topk_idx));
  float* tk_w = static_cast<float*>(at(L.pub.topk_w));
  int32_t* counts = static_cast<int32_t*>(at(L.pub.counts));
  int32_t* offsets = static_cast<int32_t*>(at(L.pub.offsets));
  int32_t* row_of = static_cast<int32_t*>(at(L.pub.row_of));
  int32_t* tok_of = static_cast<int32_t*>(at(L.pub.tok_of));
  Tile* tiles = static_cast<Tile*>(at(L.pub.tiles));
  int32_t* n_tiles = static_cast<int32_t*>(at(L.pub.n_tiles));
  float* p = static_cast<float*>(at(L.pub.p));
  float* ss_p = static_cast<float*>(at(L.pub.ss_p));
  __nv_bfloat16* xe = static_cast<__nv_bfloat16*>(at(L.pub.xe));
  __nv_bfloat16* h = static_cast<__nv_bfloat16*>(at(L.pub.h));
  float* y = static_cast<float*>(at(L.pub.y));
  float* ss_y = static_cast<float*>(at(L.pub.ss_y));
  __nv_bfloat16* c = static_cast<__nv_bfloat16*>(at(L.pub.c));
  float* u = static_cast<float*>(at(L.pub.u));
  float* ss_u = static_cast<float*>(at(L.pub.ss_u));

  cudaEvent_t* ev = ex ? ex->stage_events : nullptr;
  auto mark = [&](int i) -> bool {
    return ev == nullptr || ev[i] == nullptr || cudaEventRecord(ev[i], s) == cudaSuccess;
  };
#define LMOE_MARK(i) \
  if (!mark(i)) return LMOE_ERR_CUDA;

  // One token with NVFP4 weights (not when stages are timed): by default the steps around the
  // expert GEMMs run as two persistent kernels of one CTA per SM (decode_mk.cu) — pre-norm,
  // router, pooler, top-k and pool norm before, combine, unpooler and post-norm after — with the
  // tensor-core grouped gate/up and down GEMMs between (the expert pair where it applies;
  // measured the fastest at the Muse shapes); or the whole block as one such kernel, or the
  // stage kernels, when the caller asks for them.
  const int stp = ex ? ex->single_token_path : LMOE_SINGLE_TOKEN_DEFAULT;
  const bool mk_ok = fp4 && L.mk_scratch >= 0 && ev == nullptr;
  const bool mk = mk_ok && stp == LMOE_SINGLE_TOKEN_KERNEL;
  const bool hybrid = mk_ok && stp == LMOE_SINGLE_TOKEN_DEFAULT;
  DecodeMkArgs d{};
  if (mk || hybrid) {
    // the error word, the near-tie counter and the arrival counts of the grid barriers (the
    // whole-block or pre kernel's; the post kernel's) start at zero
    LMOE_CUDA(launch_decode_clear(err, 4, s));
    d.x = x;
    d.x_f32 = x_f32;
    d.W_router = static_cast<const __nv_bfloat16*>(W_router);
    d.router_bias = ex ? ex->router_bias : nullptr;
    d.forced = ex ? ex->forced_idx : nullptr;
    d.g_pre = g_pre;
    d.g_pool = g_pool;
    d.g_expert = g_expert;
    d.g_post = g_post;
    for (int i = 0; i < 5; ++i)
      d.w[i] = DecodeMkWeight{static_cast<const uint8_t*>(q4[i]->data), static_cast<const uint8_t*>(q4[i]->scales),
                              q4[i]->tensor_scale};
    d.D = D;
    d.L = Ld;
    d.E = E;
    d.I = I;
    d.k = k;
    d.eps = eps;
    d.out = out;
    d.out_f32 = cfg->out_dtype == LMOE_F32;
    d.g_next = ex ? ex->next_norm_gamma : nullptr;
    d.next_out = ex ? ex->next_norm_out : nullptr;
    d.xa = xa;
    d.logits = logits;
    d.topk_idx = tk_idx;
    d.topk_w = tk_w;
    d.idx_copy = ex ? ex->topk_idx_out : nullptr;
    d.w_copy = ex ? ex->topk_w_out : nullptr;
    d.near_tie = near_tie;
    d.counts = counts;
    d.offsets = offsets;
    d.row_of = row_of;
    d.tok_of = tok_of;
    d.tiles = tiles;
    d.n_tiles = n_tiles;
    d.tile_base = static_cast<int32_t*>(at(L.tile_base));
    d.tiles2 = static_cast<Tile*>(at(L.tiles2));
    d.n_tiles2 = static_cast<int32_t*>(at(L.n_tiles2));
    d.p = p;
    d.h_codes = static_cast<uint8_t*>(at(L.pub.h));
    d.h_scales = static_cast<uint8_t*>(at(L.pub.h_scale));
    d.y = static_cast<__nv_bfloat16*>(at(L.pub.y));
    d.u = u;
    d.ss_part = static_cast<float*>(at(L.mk_scratch));
    d.router_part = d.ss_part + 1LL * k * (Ld / 16) + D / 4;
    d.bar = err + 2;
    d.err = err;
    d.budget = budget;
    d.mode = mk ? kDecodeMkFull : kDecodeMkPre;
    d.cooperative = ex && ex->cooperative_launch ? 1 : 0;
    d.xe_codes = static_cast<uint8_t*>(at(L.pub.xe));
    d.xe_scales = static_cast<uint8_t*>(at(L.pub.xe_scale));
    d.xe_rowscale = static_cast<float*>(at(L.pub.xe_rowscale));
    d.ss_y = static_cast<const float*>(at(L.pub.ss_y));
    d.ld_ss_y = L.ld_ss_y;
    LMOE_CUDA(launch_decode_megakernel(d, s));
  }
  if (mk) {
#if LMOE_BOUNDS_CHECKS
    LMOE_CUDA(launch_validate_routing(tk_idx, T, k, E, counts, offsets, row_of, tok_of, tiles, n_tiles, L.max_tiles,
                                      d.tile_base, d.tiles2, d.n_tiles2, L.max_tiles2, err, false, s));
#endif
    if (ex && ex->near_tie_count_out)
      LMOE_CUDA(cudaMemcpyAsync(ex->near_tie_count_out, near_tie, 4, cudaMemcpyDeviceToDevice, s));
    return LMOE_OK;
  }

  LMOE_MARK(LMOE_STAGE_PRENORM);
  // the error word and near-tie counter start at zero on every call: the pre-norm kernel
  // clears them, unless weight conversions run first (they are cleared before those)
  if (f32w) LMOE_CUDA(cudaMemsetAsync(err, 0, 8, s));
  unsigned* status2 = f32w ? nullptr : err;

  // weights as bf16 K-major operands; fp32 weights become hi/lo bf16 pairs laid side by
  // side along K, so every product keeps ~16 significant bits of the weight
  const void *wr = W_router, *wp = W_pool, *wg = W_gate, *wu = W_up, *wd = W_down,
             *wun = W_unpool;
  const int wsplit = f32w ? 2 : 1;  // K multiplier of expert/unpooler weights
  if (f32w) {
    const struct { const void* src; long long dst; long long rows; int K; int parts; unsigned lo; } cv[] = {
        {W_router, L.w_router, E, D, 3, 4u},      {W_pool, L.w_pool, Ld, D, 3, 4u},
        {W_gate, L.w_gate, 1LL * E * I, Ld, 2, 2u}, {W_up, L.w_up, 1LL * E * I, Ld, 2, 2u},
        {W_down, L.w_down, 1LL * E * Ld, I, 2, 2u}, {W_unpool, L.w_unpool, D, Ld, 2, 2u}};
    for (const auto& c : cv)
      LMOE_CUDA(launch_weight_split(static_cast<const float*>(c.src), c.rows, c.K, c.parts, c.lo,
                                    static_cast<__nv_bfloat16*>(at(c.dst)), s));
    wr = at(L.w_router);
    wp = at(L.w_pool);
    wg = at(L.w_gate);
    wu = at(L.w_up);
    wd = at(L.w_down);
    wun = at(L.w_unpool);
  }
  const int xa_cols = L.pub.xa_cols;
  const DenseSplits dsp = dense_split_plan(cfg);
  float* partial = L.partial >= 0 ? static_cast<float*>(at(L.partial)) : nullptr;

  // S1 pre-norm (NVFP4: xn is also quantised per token for the pooler)
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  if (hybrid) {
    // S1-S6 ran in the pre kernel
  } else if (fp4)
    LMOE_CUDA(launch_prenorm_nvfp4(x, x_f32, g_pre, T, D, eps, xa, xa_cols, wsb + L.pub.xq,
                                   wsb + L.pub.xq_scale, reinterpret_cast<float*>(wsb + L.pub.xq_rowscale),
                                   status2, s));
  else
    LMOE_CUDA(launch_prenorm(x, x_f32, g_pre, T, D, eps, xa, xa_cols, status2, s));
  const int m_tiles_T = cdiv(T, kBM);
  // NVFP4 operands (offsets of fields a BF16 layout lacks are -1: null pointers then)
  auto wsp = [&](long long off) -> uint8_t* { return off >= 0 ? wsb + off : nullptr; };
  const Fp4Operand xq{wsp(L.pub.xq), wsp(L.pub.xq_scale)};
  const Fp4Operand xeq{wsp(L.pub.xe), wsp(L.pub.xe_scale)};
  const Fp4Operand hq{wsp(L.pub.h), wsp(L.pub.h_scale)};
  const Fp4Operand cq{wsp(L.pub.c), wsp(L.pub.c_scale)};
  float* xq_s = reinterpret_cast<float*>(wsp(L.pub.xq_rowscale));
  float* xe_s = reinterpret_cast<float*>(wsp(L.pub.xe_rowscale));
  float* c_s = reinterpret_cast<float*>(wsp(L.pub.c_rowscale));
  auto op = [](const lmoe_nvfp4_weight* w) { return Fp4Operand{w->data, w->scales}; };
  float* partial_pool = L.partial_pool >= 0 ? static_cast<float*>(at(L.partial_pool)) : nullptr;

  // S5 pooler, enqueued on stream `ps`: NVFP4 p = s_x * s_W * (Q(xn) . W_pool^T) (block-scaled
  // FP4 MMA), else p = xn_hi . W_pool^T; both with row partial sums of squares
  // BF16 GEMMs over many rows take 256-row tiles (two MMAs share each weight tile): the
  // pooler and unpooler from 512 rows when not split along K and where the 256-row tiles
  // still give every SM one, grouped ones at >= 256 rows per expert on average (they then
  // walk the table of 256-row tiles); the router has its own plan (dense_split_plan)
  auto dense_mh_n = [&](int splits, int n_tiles) {
    return splits <= 1 && T >= 4 * kBM && 1LL * cdiv(T, 2 * kBM) * n_tiles >= kSplitSms ? 2 : 1;
  };
  const int pool_mh = dense_mh_n(dsp.pooler, cdiv(Ld, kBNWide));
  const int unpool_mh = dense_mh_n(dsp.unpool, cdiv(D, kBNWide));
  // NVFP4 dense GEMMs of many rows (unsplit, at least two waves of 128 x 256 tiles) take the
  // 256-wide tiles: the A tile is then read once per 256 output columns
  auto fp4_dense_epi = [&](int splits, int N) {
    return splits <= 1 && N % 256 == 0 && 1LL * m_tiles_T * (N / 256) >= 2 * kSplitSms ? kFp4EpiF32SsWide
                                                                                         : kFp4EpiF32Ss;
  };
  auto pooler = [&](cudaStream_t ps) -> lmoe_status {
    if (fp4)
      return run_gemm_fp4(fp4_dense_epi(dsp.pooler, Ld), xq, T, D, op(q4[0]), Ld, nullptr, Ld, nullptr, nullptr, m_tiles_T,
                          p, Ld, nullptr, ss_p, L.ld_ss_p, xq_s, q4[0]->tensor_scale, nullptr, err, budget,
                          ps, T, T, dsp.pooler, partial_pool);
    const int pool_k = f32w ? 3 * D : D;
    return run_gemm(kEpiF32Ss, xa, T, pool_k, xa_cols, wp, Ld, pool_k, nullptr, Ld, pool_k / kBK,
                    nullptr, nullptr, cdiv(T, kBM * pool_mh), p, Ld, ss_p, L.ld_ss_p, err, budget, ps, T,
                    dsp.pooler, partial_pool, pool_mh);
  };
  // The pooler needs only xn: it runs on the side stream beside S2-S4 unless the caller
  // times those stages (their events pin every stage to the caller's stream).
  bool staged = false;
  for (int i = LMOE_STAGE_PRENORM; ev != nullptr && i <= LMOE_STAGE_POOLNORM; ++i)
    staged = staged || ev[i] != nullptr;
  SideStream* side = staged || hybrid ? nullptr : side_stream();
  std::unique_lock<std::mutex> side_lock;
  struct Join {  // the caller's stream waits for the side stream on every way out
    cudaStream_t s;
    SideStream* side;
    bool join() {
      SideStream* q = side;
      side = nullptr;
      return q == nullptr || cudaStreamWaitEvent(s, q->join, 0) == cudaSuccess;
    }
    ~Join() { join(); }
  } joiner{s, nullptr};
  if (side != nullptr) {
    side_lock = std::unique_lock<std::mutex>(side->mu);
    LMOE_CUDA(cudaEventRecord(side->fork, s));
    LMOE_CUDA(cudaStreamWaitEvent(side->stream, side->fork, 0));
    joiner.side = side;
    st = pooler(side->stream);
    if (cudaEventRecord(side->join, side->stream) != cudaSuccess) {
      joiner.side = nullptr;   // nothing to wait on; the error is reported
      return LMOE_ERR_CUDA;
    }
    if (st != LMOE_OK) return st;
  }

  LMOE_MARK(LMOE_STAGE_ROUTER);
  // S2 router logits = [xn_hi | xn_lo (| xn_hi)] . [W | W (| W_lo)]^T
  // few pairs: top-k and the permutation run as one kernel, which also sums the router's
  // split-K partials when they are few (one launch less on the chain)
  const bool fused_route = route_small_fits(T, k, E) && (ev == nullptr || ev[LMOE_STAGE_PERMUTE] == nullptr);
  const int rsplits = fused_route && dsp.router > 1 && 1LL * T * dsp.router * E <= 65536 ? dsp.router : 1;
  const int router_mh = dsp.router_mh;
  if (!hybrid) st = run_gemm(kEpiF32, xa, T, xa_cols, xa_cols, wr, E, f32w ? 3LL * D : D, nullptr, E,
                xa_cols / kBK, nullptr, nullptr, cdiv(T, kBM * router_mh), logits, L.ld_logits, nullptr, 0,
                err, budget, s, T, dsp.router, partial, router_mh, rsplits == 1);
  if (st != LMOE_OK) return st;
  LMOE_MARK(LMOE_STAGE_TOPK);
  // S3 top-k + softmax, S4 permutation (one kernel for few pairs unless S4 is timed apart)
  const float* bias = ex ? ex->router_bias : nullptr;
  const int32_t* forced = ex ? ex->forced_idx : nullptr;
  int32_t* tile_base = static_cast<int32_t*>(at(L.tile_base));
  Tile* tiles2 = static_cast<Tile*>(at(L.tiles2));
  int32_t* n_tiles2 = static_cast<int32_t*>(at(L.n_tiles2));
  if (hybrid) {
  } else if (fused_route) {
    LMOE_CUDA(launch_route_small(logits, L.ld_logits, partial, rsplits, bias, forced, T, E, k, tk_idx, tk_w,
                                 near_tie,
                                 ex ? ex->topk_idx_out : nullptr, ex ? ex->topk_w_out : nullptr, err,
                                 counts, offsets, row_of, tok_of, tiles, n_tiles, tile_base, tiles2,
                                 n_tiles2, s));
    LMOE_MARK(LMOE_STAGE_PERMUTE);
  } else {
    LMOE_CUDA(launch_topk(logits, L.ld_logits, bias, forced, T, E, k, tk_idx, tk_w, near_tie,
                          ex ? ex->topk_idx_out : nullptr, ex ? ex->topk_w_out : nullptr, err, s));
    LMOE_MARK(LMOE_STAGE_PERMUTE);
    LMOE_CUDA(launch_permute(tk_idx, T, k, E, counts, offsets, row_of, tok_of, tiles, n_tiles, s,
                             tile_base, tiles2, n_tiles2, static_cast<int32_t*>(at(L.perm_hist)),
                             static_cast<int32_t*>(at(L.perm_base))));
  }
#if LMOE_BOUNDS_CHECKS
  // checked build: the routing structures are validated before any kernel follows them; on a
  // violation the error word says so and the rest of the call runs on a harmless routing
  LMOE_CUDA(launch_validate_routing(tk_idx, T, k, E, counts, offsets, row_of, tok_of, tiles, n_tiles, L.max_tiles,
                                    tile_base, tiles2, n_tiles2, L.max_tiles2, err, true, s));
#endif
  if (ex && ex->near_tie_count_out)
    LMOE_CUDA(cudaMemcpyAsync(ex->near_tie_count_out, near_tie, 4, cudaMemcpyDeviceToDevice, s));
  if (side != nullptr) {
    if (!joiner.join()) return LMOE_ERR_CUDA;
    side_lock.unlock();
  } else if (!hybrid) {
    LMOE_MARK(LMOE_STAGE_POOLER);
    st = pooler(s);
    if (st != LMOE_OK) return st;
  }
  if (fp4) {
    LMOE_MARK(LMOE_STAGE_POOLNORM);
    // S6 pool norm, quantised per token, copied to the k expert rows
    if (!hybrid)
      LMOE_CUDA(launch_poolnorm_scatter_nvfp4(p, ss_p, L.ld_ss_p, g_pool, row_of, tk_idx, offsets,
                                            tile_base, T, Ld, k, eps, wsb + L.pub.xe,
                                            wsb + L.pub.xe_scale, xe_s, s));
    LMOE_MARK(LMOE_STAGE_GATE_UP);
    // S7 grouped gate/up + SwiGLU, h requantised to NVFP4 (scale 1); at small T split-K
    // with the split count picked on the device from the live tiles
    int* splits_dev = static_cast<int*>(at(L.splits_dev));
    // the live tile count lies in [max(k, R/128), max_tiles] (a token's k experts are
    // distinct); where no count in that range splits, the GEMM runs unsplit with no reduce
    const int lo_tiles = std::max(k, cdiv(R, kBM));
    auto grouped_splits = [&](int N, int num_kb) -> int {
      const int gs = grouped_max_splits(cfg);
      if (gs <= 1) return 1;
      const long long ids = tile_id_bound(L.max_tiles, N, kBNFp4, gs);
      const int grid = static_cast<int>(std::min<long long>(ids, sm_count()));
      return grouped_split_possible(lo_tiles, L.max_tiles, cdiv(N, kBNFp4), num_kb, grid, gs) ? gs : 1;
    };
    const Fp4Operand up = op(q4[2]);
    // a few tokens (M tiles of at most 32 rows) and gate/up tiles for at least every SM: S7 and
    // S8 as one launch, whose down tiles fill the SMs that finish their gate/up tiles first
    if (expert_pair_rule(cfg) && !(ex && ex->separate_expert_gemms)) {
      st = run_gemm_fp4_pair(xeq, xe_s, op(q4[1]), up, op(q4[3]), q4[1]->tensor_scale, q4[2]->tensor_scale,
                             q4[3]->tensor_scale, R, Ld, I, E, tiles, n_tiles, L.max_tiles, wsb + L.pub.h,
                             wsb + L.pub.h_scale, y, ss_y, L.ld_ss_y, splits_dev, err, budget, s);
      if (st != LMOE_OK) return st;
      LMOE_MARK(LMOE_STAGE_DOWN);   // the down stage of a recorded call is empty
    } else {
      st = run_gemm_fp4(kFp4EpiSwiGLUQuant, xeq, R, Ld, op(q4[1]), 1LL * E * I, &up, I, tiles, n_tiles,
                        L.max_tiles, wsb + L.pub.h, I, wsb + L.pub.h_scale, nullptr, 0, xe_s,
                        q4[1]->tensor_scale, q4[2]->tensor_scale, err, budget, s, R / E, T,
                        grouped_splits(I, Ld / 256), partial, splits_dev);
      if (st != LMOE_OK) return st;
      LMOE_MARK(LMOE_STAGE_DOWN);
      // S8 grouped down: y rounded to bf16, with per-row partial sums of squares of those values;
      // unsplit on 128 x 256 tiles, which read each expert's h tile (and pay each stage's A box,
      // scale copies and barriers) once per 256 output columns: measured faster at every T
      const int down_splits = grouped_splits(Ld, I / 256);
      const Fp4EpiKind down_epi = down_splits <= 1 && Ld % 256 == 0 ? kFp4EpiBf16SsWide : kFp4EpiBf16Ss;
      st = run_gemm_fp4(down_epi, hq, R, I, op(q4[3]), 1LL * E * Ld, nullptr, Ld, tiles, n_tiles,
                        L.max_tiles, y, Ld, nullptr, ss_y, L.ld_ss_y, nullptr, q4[3]->tensor_scale,
                        nullptr, err, budget, s, R / E, T, down_splits, partial, splits_dev + 1);
      if (st != LMOE_OK) return st;
    }
    if (hybrid) {   // S9-S11 in the post kernel, with a barrier counter of its own
      d.bar = err + 3;
      d.mode = kDecodeMkPost;
      LMOE_CUDA(launch_decode_megakernel(d, s));
      return LMOE_OK;
    }
    LMOE_MARK(LMOE_STAGE_COMBINE);
    // S9 combine, c quantised per token
    LMOE_CUDA(launch_combine_nvfp4(y, true, ss_y, L.ld_ss_y, row_of, tk_idx, tk_w, g_expert, T, Ld, k, eps,
                                   wsb + L.pub.c, wsb + L.pub.c_scale, c_s, s));
    LMOE_MARK(LMOE_STAGE_UNPOOLER);
    // S10 unpooler u = s_c * s_W * (Q(c) . W_unpool^T)
    st = run_gemm_fp4(fp4_dense_epi(dsp.unpool, D), cq, T, Ld, op(q4[4]), D, nullptr, D, nullptr, nullptr, m_tiles_T, u,
                      D, nullptr, ss_u, L.ld_ss_u, c_s, q4[4]->tensor_scale, nullptr, err, budget, s, T, T,
                      dsp.unpool, partial, nullptr, false);
    if (st != LMOE_OK) return st;
  } else {
  LMOE_MARK(LMOE_STAGE_POOLNORM);
  // S6 pool norm, scattered to the k expert-contiguous rows of each token
  LMOE_CUDA(launch_poolnorm_scatter(p, ss_p, L.ld_ss_p, g_pool, row_of, T, Ld, k, eps, xe, s));
  LMOE_MARK(LMOE_STAGE_GATE_UP);
  // S7 grouped gate/up + SwiGLU
  const int gmh = R / E >= 2 * kBM ? 2 : 1;
  const Tile* gtiles = gmh == 2 ? tiles2 : tiles;
  const int* gn_tiles = gmh == 2 ? n_tiles2 : n_tiles;
  const int gmax = gmh == 2 ? L.max_tiles2 : L.max_tiles;
  st = run_gemm(kEpiSwiGLU, xe, R, Ld, Ld, wg, 1LL * E * I, 1LL * wsplit * Ld, wu, I,
                wsplit * Ld / kBK, gtiles, gn_tiles, gmax, h, I, nullptr, 0, err, budget, s, R / E, 1,
                nullptr, gmh);
  if (st != LMOE_OK) return st;
  LMOE_MARK(LMOE_STAGE_DOWN);
  // S8 grouped down (fp32 y), with per-row partial sums of squares
  st = run_gemm(kEpiF32Ss, h, R, I, I, wd, 1LL * E * Ld, 1LL * wsplit * I, nullptr, Ld,
                wsplit * I / kBK, gtiles, gn_tiles, gmax, y, Ld, ss_y, L.ld_ss_y, err, budget, s, R / E, 1,
                nullptr, gmh);
  if (st != LMOE_OK) return st;
  LMOE_MARK(LMOE_STAGE_COMBINE);
  // S9 combine: per-expert RMSNorm, routing weight, fp32 sum in slot order
  LMOE_CUDA(launch_combine(y, ss_y, L.ld_ss_y, row_of, tk_idx, tk_w, g_expert, T, Ld, k, eps, c, s));
  LMOE_MARK(LMOE_STAGE_UNPOOLER);
  // S10 unpooler u = c . W_unpool^T with row partial sums of squares
  st = run_gemm(kEpiF32Ss, c, T, Ld, Ld, wun, D, 1LL * wsplit * Ld, nullptr, D, wsplit * Ld / kBK,
                nullptr, nullptr, cdiv(T, kBM * unpool_mh), u, D, ss_u, L.ld_ss_u, err, budget, s, T,
                dsp.unpool, partial, unpool_mh, false);
  if (st != LMOE_OK) return st;
  }
  LMOE_MARK(LMOE_STAGE_POSTNORM);
  // S11 post-norm + residual
  // S11 reads the unpooler's split-K partials itself when it ran split (no reduction launch)
  LMOE_CUDA(launch_postnorm_residual(x, x_f32, u, ss_u, L.ld_ss_u, g_post, T, D, eps, out,
                                     cfg->out_dtype == LMOE_F32, s, partial, dsp.unpool,
                                     ex ? ex->next_norm_gamma : nullptr, ex ? ex->next_norm_out : nullptr));
  LMOE_MARK(LMOE_STAGE_END);
#undef LMOE_MARK
  return LMOE_OK;
}

}  // namespace

extern "C" {

lmoe_status lmoe_workspace_size(const lmoe_config* cfg, size_t* bytes) {
  const lmoe_status st = check_config(cfg);
  if (st != LMOE_OK) return st;
  if (bytes == nullptr) return LMOE_ERR_ARG;
  Layout L;
  make_layout(cfg, &L);
  *bytes = static_cast<size_t>(L.pub.total);
  return LMOE_OK;
}

lmoe_status lmoe_expert_pair(const lmoe_config* cfg, int* used) {
  const lmoe_status st = check_config(cfg);
  if (st != LMOE_OK) return st;
  if (used == nullptr) return LMOE_ERR_ARG;
  *used = expert_pair_rule(cfg) ? 1 : 0;
  return LMOE_OK;
}

lmoe_status lmoe_workspace_size_host_io(const lmoe_config* cfg, size_t* bytes) {
  const lmoe_status st = check_config(cfg);
  if (st != LMOE_OK) return st;
  if (bytes == nullptr) return LMOE_ERR_ARG;
  Layout L;
  make_layout(cfg, &L);
  *bytes = static_cast<size_t>(L.host_io_total);
  return LMOE_OK;
}

lmoe_status lmoe_get_workspace_layout(const lmoe_config* cfg, lmoe_workspace_layout* layout) {
  const lmoe_status st = check_config(cfg);
  if (st != LMOE_OK) return st;
  if (layout == nullptr) return LMOE_ERR_ARG;
  Layout L;
  make_layout(cfg, &L);
  *layout = L.pub;
  return LMOE_OK;
}

lmoe_status latent_moe_forward(const lmoe_config* cfg, const void* x, const void* W_router,
                               const void* W_pool, const float* g_pool, const void* W_gate,
                               const void* W_up, const void* W_down, const float* g_expert,
                               const void* W_unpool, const float* g_pre, const float* g_post,
                               int top_k, void* out, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
  return forward_impl(cfg, x, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert, W_unpool,
                      g_pre, g_post, top_k, out, workspace, workspace_bytes, stream, nullptr);
}

lmoe_status latent_moe_forward_ex(const lmoe_config* cfg, const void* x, const void* W_router,
                                  const void* W_pool, const float* g_pool, const void* W_gate,
                                  const void* W_up, const void* W_down, const float* g_expert,
                                  const void* W_unpool, const float* g_pre, const float* g_post,
                                  int top_k, void* out, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream, const lmoe_ex* ex) {
  return forward_impl(cfg, x, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert, W_unpool,
                      g_pre, g_post, top_k, out, workspace, workspace_bytes, stream, ex);
}

lmoe_status latent_moe_forward_host_io_ex(const lmoe_config* cfg, const void* x_host,
                                          const void* W_router, const void* W_pool,
                                          const float* g_pool, const void* W_gate, const void* W_up,
                                          const void* W_down, const float* g_expert,
                                          const void* W_unpool, const float* g_pre,
                                          const float* g_post, int top_k, void* out_host,
                                          void* workspace, size_t workspace_bytes,
                                          cudaStream_t stream, const lmoe_ex* ex) {
  const lmoe_status st = check_config(cfg);
  if (st != LMOE_OK) return st;
  if (x_host == nullptr || out_host == nullptr) return LMOE_ERR_ARG;
  Layout L;
  make_layout(cfg, &L);
  if (workspace == nullptr || workspace_bytes < static_cast<size_t>(L.host_io_total))
    return LMOE_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  const size_t xb = static_cast<size_t>(cfg->T) * cfg->d_model * (cfg->act_dtype == LMOE_F32 ? 4 : 2);
  const size_t ob = static_cast<size_t>(cfg->T) * cfg->d_model * (cfg->out_dtype == LMOE_F32 ? 4 : 2);
  if (cfg->T == 0) return LMOE_OK;
  if (cudaMemcpyAsync(ws + L.x_stage, x_host, xb, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  const lmoe_status s2 =
      forward_impl(cfg, ws + L.x_stage, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert,
                   W_unpool, g_pre, g_post, top_k, ws + L.out_stage, workspace,
                   static_cast<size_t>(L.pub.total), stream, ex);
  if (s2 != LMOE_OK) return s2;
  if (cudaMemcpyAsync(out_host, ws + L.out_stage, ob, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

lmoe_status latent_moe_forward_host_io(const lmoe_config* cfg, const void* x_host,
                                       const void* W_router, const void* W_pool,
                                       const float* g_pool, const void* W_gate, const void* W_up,
                                       const void* W_down, const float* g_expert,
                                       const void* W_unpool, const float* g_pre,
                                       const float* g_post, int top_k, void* out_host,
                                       void* workspace, size_t workspace_bytes,
                                       cudaStream_t stream) {
  return latent_moe_forward_host_io_ex(cfg, x_host, W_router, W_pool, g_pool, W_gate, W_up, W_down,
                                       g_expert, W_unpool, g_pre, g_post, top_k, out_host, workspace,
                                       workspace_bytes, stream, nullptr);
}

lmoe_status lmoe_check_status(const lmoe_config* cfg, void* workspace, cudaStream_t stream,
                              uint32_t* detail) {
  const lmoe_status st = check_config(cfg);
  if (st != LMOE_OK) return st;
  if (workspace == nullptr) return LMOE_ERR_WORKSPACE;
  Layout L;
  make_layout(cfg, &L);
  uint32_t word = 0;
  unsigned* err = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + L.pub.err);
  if (cudaMemcpyAsync(&word, err, 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return LMOE_ERR_CUDA;
  if (cudaMemsetAsync(err, 0, 4, stream) != cudaSuccess) return LMOE_ERR_CUDA;
  if (detail) *detail = word;
  if (word & (kErrWaitProducer | kErrWaitMma | kErrWaitEpilogue | kErrDrain | kErrGridBarrier))
    return LMOE_ERR_TIMEOUT;
  if (word & (kErrBadIndex | kErrBounds)) return LMOE_ERR_ARG;
  return LMOE_OK;
}

lmoe_status lmoe_workspace_guards(const lmoe_config* cfg, int host_io, long long* offsets, int capacity,
                                  int* count) {
  const lmoe_status st = check_config(cfg);
  if (st != LMOE_OK) return st;
  if (count == nullptr || capacity < 0) return LMOE_ERR_ARG;
  Layout L;
  make_layout(cfg, &L);
  // the bands after the two host-I/O staging buffers are the last two
  const int n = host_io ? L.n_guards : L.n_guards - 2;
  *count = n;
  if (offsets != nullptr)
    for (int i = 0; i < n && i < capacity; ++i) offsets[i] = L.guards[i];
  return LMOE_OK;
}

lmoe_status lmoe_validate_routing(const lmoe_config* cfg, void* workspace, cudaStream_t stream) {
  const lmoe_status st = check_config(cfg);
  if (st != LMOE_OK) return st;
  if (workspace == nullptr) return LMOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return LMOE_ERR_ALIGN;
  Layout L;
  make_layout(cfg, &L);
  char* ws = static_cast<char*>(workspace);
  auto at = [&](long long o) { return static_cast<void*>(ws + o); };
  if (launch_validate_routing(static_cast<int32_t*>(at(L.pub.topk_idx)), cfg->T, cfg->top_k, cfg->n_experts,
                              static_cast<const int32_t*>(at(L.pub.counts)), static_cast<int32_t*>(at(L.pub.offsets)),
                              static_cast<int32_t*>(at(L.pub.row_of)), static_cast<const int32_t*>(at(L.pub.tok_of)),
                              static_cast<const Tile*>(at(L.pub.tiles)), static_cast<int32_t*>(at(L.pub.n_tiles)),
                              L.max_tiles, static_cast<int32_t*>(at(L.tile_base)),
                              static_cast<const Tile*>(at(L.tiles2)),
                              static_cast<int32_t*>(at(L.n_tiles2)), L.max_tiles2,
                              static_cast<unsigned*>(at(L.pub.err)), false, stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

lmoe_status lmoe_quantize_nvfp4(const float* src, long long rows, int K, int row_scale,
                                uint8_t* codes, uint8_t* scales, float* s_row,
                                cudaStream_t stream) {
  if (rows < 0 || rows > (1LL << 31) - 1 || K <= 0 || K % 16 || K > 32768) return LMOE_ERR_ARG;
  if (rows == 0) return LMOE_OK;
  if (src == nullptr || codes == nullptr || scales == nullptr) return LMOE_ERR_ARG;
  if (!aligned16(src) || (reinterpret_cast<uintptr_t>(codes) & 7u)) return LMOE_ERR_ALIGN;
  if (launch_quantize_nvfp4(src, rows, K, row_scale != 0, codes, scales, s_row, stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

lmoe_status lmoe_nvfp4_block_scales(const uint8_t* src, long long rows, int K, int block_rows,
                                    uint8_t* dst, cudaStream_t stream) {
  if (block_rows != 64 && block_rows != 128) return LMOE_ERR_ARG;
  if (rows < 0 || rows % block_rows || K <= 0 || K % 64) return LMOE_ERR_ARG;
  if (rows == 0) return LMOE_OK;
  if (src == nullptr || dst == nullptr || src == dst) return LMOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(dst) & 3u) || (reinterpret_cast<uintptr_t>(src) & 3u))
    return LMOE_ERR_ALIGN;
  if (launch_nvfp4_block_scales(src, rows, K, block_rows, dst, stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

lmoe_status lmoe_wait_selftest(const lmoe_config* cfg, void* workspace, long long budget_cycles,
                               cudaStream_t stream) {
  const lmoe_status st = check_config(cfg);
  if (st != LMOE_OK) return st;
  if (workspace == nullptr) return LMOE_ERR_WORKSPACE;
  Layout L;
  make_layout(cfg, &L);
  const long long b = budget_cycles < 1 ? 1 : (budget_cycles > 4000000000LL ? 4000000000LL : budget_cycles);
  unsigned* err = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + L.pub.err);
  if (launch_wait_selftest(b, err, stream) != cudaSuccess) return LMOE_ERR_CUDA;
  return LMOE_OK;
}

unsigned long long lmoe_kernel_launches(void) { return g_launches.load(); }

const char* lmoe_status_string(lmoe_status s) {
  switch (s) {
    case LMOE_OK: return "ok";
    case LMOE_ERR_ARG: return "invalid argument";
    case LMOE_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case LMOE_ERR_ALIGN: return "pointer not aligned (16 B for tensors, 256 B for workspace)";
    case LMOE_ERR_WORKSPACE: return "workspace missing or too small";
    case LMOE_ERR_CUDA: return "CUDA call failed";
    case LMOE_ERR_TIMEOUT: return "a device wait exceeded its budget";
  }
  return "unknown status";
}

}  // extern "C"
