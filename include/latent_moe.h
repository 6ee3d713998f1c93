/*
 * latent_moe.h — C ABI of a GB300 (sm_103a) implementation of the Muse Spark
 * Open latent mixture-of-experts decoder block:
 *
 *     out = x + RMSNorm_post( F( RMSNorm_pre(x) ) )
 *
 * with F = full-width router (softmax over all experts, top-k, weights
 * renormalised over the k) ; pooler d_model -> d_latent and RMSNorm ; routed
 * SwiGLU experts at width d_latent ; each selected expert's output
 * RMS-normalised with its own gamma BEFORE it is multiplied by its routing
 * weight ; FP32 weighted sum ; unpooler d_latent -> d_model.
 *
 * Sources: LMSYS "SGLang and Miles Add Day-0 Support for Muse Spark Open",
 * section "MoE with pooler, unpooler and per-expert normalization" (router on
 * the full-width input, pooled input normalised before the experts, per-expert
 * RMSNorm before the weighted sum, then unpool), "Fused per-expert post-norm"
 * (partial sums of squares of the bf16 values of each down-projection tile,
 * one scalar per selected expert read at combine), "Reinforcement learning"
 * (weighted sum in FP32), "NVFP4 as a third MMA type" (E2M1 data, UE4M3 scale
 * per 16 elements, per-token FP32 input scale); vLLM "Day 0 support for Muse
 * Spark Open", sections "Sandwich normalization" and "Latent MoE".
 *
 * Conventions
 *  - Every pointer named in a signature as device memory must be a CUDA
 *    device pointer of the current device, 16-byte aligned.  Host-memory
 *    arguments are marked "host".
 *  - Every weight matrix is "out x in", row-major, K (the "in" dimension)
 *    contiguous: W_router [E, D], W_pool [L, D], W_gate/W_up [E, I, L],
 *    W_down [E, L, I], W_unpool [D, L].
 *  - The caller owns all memory (inputs, out, workspace).  The library
 *    allocates no device memory in any call.
 *  - Calls are asynchronous on `stream`; nothing synchronises the host.
 *  - Host-detectable errors return a negative status before any launch and
 *    leave out/workspace untouched.  A launch error maps to LMOE_ERR_CUDA.
 *    A device-side wait that exceeds its budget sets an error word in the
 *    workspace, which lmoe_check_status() reads back (LMOE_ERR_TIMEOUT).
 *  - Calls that share one workspace must not overlap on the GPU.
 */
#ifndef LATENT_MOE_H_
#define LATENT_MOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LMOE_OK = 0,
  LMOE_ERR_ARG = -1,          /* null pointer, bad size, top_k out of range            */
  LMOE_ERR_UNSUPPORTED = -2,  /* a shape or dtype combination the kernels do not cover */
  LMOE_ERR_ALIGN = -3,        /* a device pointer not 16-byte aligned                  */
  LMOE_ERR_WORKSPACE = -4,    /* workspace null or smaller than lmoe_workspace_size()  */
  LMOE_ERR_CUDA = -5,         /* a CUDA runtime/driver call failed                     */
  LMOE_ERR_TIMEOUT = -6       /* a device wait ran past its budget                     */
} lmoe_status;

typedef enum { LMOE_F32 = 0, LMOE_BF16 = 1, LMOE_NVFP4 = 2 } lmoe_dtype;

/* Block shape and dtypes.
 *  T          tokens (rows of x), 0 <= T <= 1<<20 (T = 0 is a no-op)
 *  d_model    D, multiple of 128           d_latent  L, multiple of 128
 *  n_experts  E, 1..1024                   d_ff      I, multiple of 128
 *  top_k      k, 1..min(E, 16)             eps       RMSNorm epsilon (all four norms)
 *             (NVFP4 weights: D, L, I multiples of 256 and at most 32768)
 *  act_dtype  dtype of x: LMOE_F32 or LMOE_BF16
 *  weight_dtype  LMOE_F32, LMOE_BF16, or LMOE_NVFP4 (pooler, experts, unpooler packed;
 *             the router then stays LMOE_BF16)
 *  out_dtype  LMOE_F32 or LMOE_BF16                                                  */
typedef struct {
  int T, d_model, d_latent, n_experts, d_ff, top_k;
  float eps;
  lmoe_dtype act_dtype, weight_dtype, out_dtype;
} lmoe_config;

/* Layouts of the E4M3 block scales of an NVFP4 weight (lmoe_nvfp4_weight.scale_layout). */
typedef enum {
  /* [rows, K/16] row-major, one scale per 16 consecutive k: the plain layout.  The forward
   * entry points do not read it (they return LMOE_ERR_UNSUPPORTED before any launch):
   * convert it once with lmoe_nvfp4_block_scales() and pass LMOE_NVFP4_SCALES_BLOCKED.     */
  LMOE_NVFP4_SCALES_ROW_MAJOR = 0,
  /* the tensor cores' block layout: 512-byte blocks of 128 rows x 64 k, ordered
   * [rows/128][K/64]; inside a block the scale of row m = m0 + 32*m1 and 16-wide group kk
   * sits at byte 16*m0 + 4*m1 + kk (what lmoe_nvfp4_block_scales() writes).                */
  LMOE_NVFP4_SCALES_BLOCKED = 1
} lmoe_nvfp4_scale_layout;

/* One NVFP4-packed weight (host struct holding device pointers), "out x in" [rows, K]:
 *  data          [rows, K/2] bytes, two E2M1 codes per byte, the low nibble holds the even k
 *  scales        E4M3 block-scale codes (one per 16 consecutive k), in `scale_layout`
 *                (for expert stacks, rows = E*rows_per_expert)
 *  tensor_scale  fp32 second-level scale: 1 value, or one per expert for expert stacks
 *  scale_layout  an lmoe_nvfp4_scale_layout; a zero-initialised struct declares row-major
 *                scales, which the forward refuses, so scales in the wrong layout are never
 *                read as if they were blocked
 *  value = e2m1(code) * e4m3(scale) * tensor_scale.                                    */
typedef struct {
  const uint8_t* data;
  const uint8_t* scales;
  const float* tensor_scale;
  int scale_layout;
} lmoe_nvfp4_weight;

/* Stage boundaries of one call, for stage_events (see lmoe_ex).  Event i is recorded on
 * the call's stream just before stage i is enqueued; event LMOE_STAGE_END after the last. */
enum {
  LMOE_STAGE_PRENORM = 0,   /* pre-norm (and fp32 weight splits)              */
  LMOE_STAGE_ROUTER = 1,    /* router GEMM                                     */
  LMOE_STAGE_TOPK = 2,      /* softmax + top-k                                 */
  LMOE_STAGE_PERMUTE = 3,   /* expert histogram + stable scatter               */
  LMOE_STAGE_POOLER = 4,    /* pooler GEMM                                     */
  LMOE_STAGE_POOLNORM = 5,  /* pool norm, copied to expert rows                */
  LMOE_STAGE_GATE_UP = 6,   /* grouped gate/up GEMM + SwiGLU                   */
  LMOE_STAGE_DOWN = 7,      /* grouped down GEMM                               */
  LMOE_STAGE_COMBINE = 8,   /* per-expert norm, routing weight, weighted sum   */
  LMOE_STAGE_UNPOOLER = 9,  /* unpooler GEMM                                   */
  LMOE_STAGE_POSTNORM = 10, /* post-norm + residual                            */
  LMOE_STAGE_END = 11,
  LMOE_NUM_STAGE_EVENTS = 12
};

/* Optional extensions of one call (host struct; every member may be NULL/0).
 *  router_bias       [E] fp32 device: added to the router logits before softmax/top-k
 *  forced_idx        [T, k] int32 device: use these experts (distinct per row) instead of
 *                    the top-k; weights are the softmax of the logits renormalised over them.
 *                    An id outside [0, E) or repeated within a row is flagged on the
 *                    device (lmoe_check_status then returns LMOE_ERR_ARG).
 *  topk_idx_out      [T, k] int32 device: selected experts, descending logit
 *  topk_w_out        [T, k] fp32 device: their routing weights
 *  near_tie_count_out  [1] int32 device: tokens whose k-th and (k+1)-th logits differ by < 1e-3
 *  wait_budget_cycles  SM clock cycles a device wait may spin before it gives up (0: default)
 *  next_norm_gamma   [D] fp32 device, with next_norm_out [T, D] device (out_dtype): S11 also
 *                    writes RMSNorm(out) * next_norm_gamma — the next layer's pre-norm taken
 *                    from the same row in the same kernel (LMSYS Muse Spark Open post,
 *                    § "Kernel optimizations": FFN post-norm, residual add and the next
 *                    pre-norm as one kernel).  Both NULL: not written.  One alone: ERR_ARG.
 *  stage_events      host array of LMOE_NUM_STAGE_EVENTS caller-created cudaEvent_t, or NULL:
 *                    recorded on the stream at the stage boundaries above (timing only);
 *                    a NULL entry is skipped.  Kernels of one call are launched with
 *                    programmatic dependent launch, so a kernel's set-up overlaps the end of
 *                    the previous one; an event between two kernels serialises them fully.
 *  single_token_path  with NVFP4 weights and T = 1 (one decode token), which kernels run
 *                    (ignored otherwise, and when a stage event is set; a value outside the
 *                    three below: LMOE_ERR_ARG):
 *                    LMOE_SINGLE_TOKEN_DEFAULT (0): two persistent kernels of one CTA per SM
 *                      around the tensor-core grouped gate/up and down GEMMs (as one launch
 *                      where lmoe_expert_pair() says so), after a one-warp kernel that zeroes
 *                      the call's status and barrier words: before them the
 *                      pre-norm, router, pooler, top-k, routing tables and pool norm (writing
 *                      the gate/up GEMM's NVFP4 input rows), after them the per-expert norms,
 *                      combine, unpooler and post-norm; each streams its weights into shared
 *                      memory by bulk copies and dots them on the CUDA cores, the row steps
 *                      redundant in every CTA;
 *                    LMOE_SINGLE_TOKEN_KERNEL (1): the whole block as one such kernel, the
 *                      expert weights on the CUDA cores too (four weight phases behind grid
 *                      barriers);
 *                    LMOE_SINGLE_TOKEN_CHAIN (2): the stage kernels, as at T > 1.
 *                    On a GB300 at the Muse shapes the default is the fastest of the three.
 *                    The persistent kernels take D and I multiples of 256 up to 8192, L up to
 *                    4096 and E <= 1024 (else the stage kernels run), with the same arithmetic
 *                    as the chain up to the order of fp32 sums; after them the workspace holds
 *                    xa, the logits, the routing tables, p, y and u as after the chain, but not
 *                    every quantised operand nor every partial sum of squares.  A grid barrier
 *                    or stage wait past wait_budget_cycles sets bit 0x40 of the error word
 *                    (LMOE_ERR_TIMEOUT).
 *  cooperative_launch  nonzero: those persistent kernels are launched cooperatively, so the
 *                    driver starts one only once every CTA can be resident; needed where other
 *                    work may hold SMs meanwhile (another stream or process; two such calls at
 *                    once on two streams).  0 (default): launched as ordinary grids of one CTA
 *                    per SM with programmatic dependent launch, so each starts on the SMs the
 *                    previous kernel leaves while it drains (measured 7.6 us faster per call at
 *                    the Muse shapes); their grid barriers assume the call has the SMs to itself,
 *                    and give up after wait_budget_cycles (LMOE_ERR_TIMEOUT) otherwise.
 *  separate_expert_gemms  nonzero: the grouped gate/up and down GEMMs run as two launches
 *                    even where lmoe_expert_pair() says they run as one (for inspection:
 *                    both compute the same values bit for bit). */
enum {
  LMOE_SINGLE_TOKEN_DEFAULT = 0,
  LMOE_SINGLE_TOKEN_KERNEL = 1,
  LMOE_SINGLE_TOKEN_CHAIN = 2
};
typedef struct {
  const float* router_bias;
  const int32_t* forced_idx;
  int32_t* topk_idx_out;
  float* topk_w_out;
  int32_t* near_tie_count_out;
  long long wait_budget_cycles;
  cudaEvent_t* stage_events;
  const float* next_norm_gamma;
  void* next_norm_out;
  int single_token_path;
  int separate_expert_gemms;
  int cooperative_launch;
} lmoe_ex;

/* Whether a call with this config runs the grouped gate/up (S7) and down (S8) GEMMs as one
 * persistent launch, the expert pair (host arithmetic only; *used = 1 or 0): NVFP4 weights,
 * T <= 32 (every expert's rows fit one 32-row tile), d_latent a multiple of 256, and at
 * least 152 gate/up tiles of 128 columns (top_k * d_ff / 128, or more rows' worth).  The
 * down tiles of an expert start once all of its gate/up tiles have stored h (a count per
 * tile in the workspace, waited on with wait_budget_cycles; past it: LMOE_ERR_TIMEOUT), so
 * the SMs that finish their gate/up tiles first take the down tiles.  With stage events the
 * gate_up stage then spans both GEMMs and the down stage is empty.                      */
lmoe_status lmoe_expert_pair(const lmoe_config* cfg, int* used);

/* Bytes of device workspace a call with this config needs (host out-parameter). */
lmoe_status lmoe_workspace_size(const lmoe_config* cfg, size_t* bytes);

/* The block.  Device pointers:
 *  x         [T, D]   act_dtype
 *  W_router  [E, D]   fp32 when weight_dtype is LMOE_F32, else bf16
 *  W_pool    [L, D]   } bf16/fp32 per weight_dtype, or, for LMOE_NVFP4, a HOST pointer to
 *  W_gate    [E, I, L]}  an lmoe_nvfp4_weight (expert stacks: data [E, rows, K/2], scales of
 *  W_up      [E, I, L]}  E*rows rows, tensor_scale [E]; W_gate and W_up may use different
 *  W_down    [E, L, I]}  scales; scale_layout must be LMOE_NVFP4_SCALES_BLOCKED, else
 *                        LMOE_ERR_UNSUPPORTED)
 *  W_unpool  [D, L]   }
 *  g_pool [L], g_expert [E, L], g_pre [D], g_post [D]   fp32 RMSNorm gammas
 *  top_k     must equal cfg->top_k
 *  out       [T, D]   out_dtype (may not alias x)
 *  workspace device buffer of at least lmoe_workspace_size() bytes, 256-byte aligned  */
lmoe_status latent_moe_forward(const lmoe_config* cfg, const void* x, const void* W_router,
                               const void* W_pool, const float* g_pool, const void* W_gate,
                               const void* W_up, const void* W_down, const float* g_expert,
                               const void* W_unpool, const float* g_pre, const float* g_post,
                               int top_k, void* out, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/* latent_moe_forward with the extensions of `ex` (host pointer, may be NULL). */
lmoe_status latent_moe_forward_ex(const lmoe_config* cfg, const void* x, const void* W_router,
                                  const void* W_pool, const float* g_pool, const void* W_gate,
                                  const void* W_up, const void* W_down, const float* g_expert,
                                  const void* W_unpool, const float* g_pre, const float* g_post,
                                  int top_k, void* out, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream, const lmoe_ex* ex);

/* latent_moe_forward with x and out in HOST memory (pinned for asynchronous copies):
 * copies x to the workspace, runs the block, copies out back, all on `stream`.
 * The weights stay device pointers.  workspace must hold lmoe_workspace_size() plus
 * the x and out staging bytes reported by lmoe_workspace_size_host_io().             */
lmoe_status lmoe_workspace_size_host_io(const lmoe_config* cfg, size_t* bytes);
lmoe_status latent_moe_forward_host_io(const lmoe_config* cfg, const void* x_host,
                                       const void* W_router, const void* W_pool,
                                       const float* g_pool, const void* W_gate, const void* W_up,
                                       const void* W_down, const float* g_expert,
                                       const void* W_unpool, const float* g_pre,
                                       const float* g_post, int top_k, void* out_host,
                                       void* workspace, size_t workspace_bytes,
                                       cudaStream_t stream);
/* latent_moe_forward_host_io with the extensions of `ex` (host pointer, may be NULL; the
 * pointers inside it stay device pointers, as for latent_moe_forward_ex). */
lmoe_status latent_moe_forward_host_io_ex(const lmoe_config* cfg, const void* x_host,
                                          const void* W_router, const void* W_pool,
                                          const float* g_pool, const void* W_gate, const void* W_up,
                                          const void* W_down, const float* g_expert,
                                          const void* W_unpool, const float* g_pre,
                                          const float* g_post, int top_k, void* out_host,
                                          void* workspace, size_t workspace_bytes,
                                          cudaStream_t stream, const lmoe_ex* ex);

/* Reads (synchronising `stream`) and clears the device error word of `workspace`.
 * Returns LMOE_OK, LMOE_ERR_TIMEOUT (a device wait gave up: bits 0x1, 0x2, 0x4, 0x10, 0x40) or
 * LMOE_ERR_ARG (a forced expert id out of range or repeated: bit 0x8; routing structures
 * that failed lmoe_validate_routing: bit 0x20); *detail (host, may be NULL) receives the raw
 * word. */
lmoe_status lmoe_check_status(const lmoe_config* cfg, void* workspace, cudaStream_t stream,
                              uint32_t* detail);

/* Byte offsets of the intermediates inside the workspace, for inspection:
 *  xa (router/pooler input rows), logits [T,E] f32, topk_idx [T,k] i32, topk_w [T,k] f32,
 *  counts [E] i32, offsets [E+1] i32, row_of [T,k] i32, tok_of [T*k] i32,
 *  p [T,L] f32, xe [T*k, L] bf16 (expert-contiguous expert inputs), h [T*k, I] bf16,
 *  y [T*k, L] f32 (bf16 with NVFP4 weights), ss_y [T*k, L/128] f32 (sums of squares of the
 *  stored y values), c [T,L] bf16, u [T,D] f32, ss_p / ss_u
 *  [rows, N/128] f32 (row sums of squares per 128 columns), err (u32).
 *  Unused fields are -1. */
typedef struct {
  long long xa, logits, topk_idx, topk_w, counts, offsets, row_of, tok_of, tiles, n_tiles,
      p, ss_p, xe, xe_scale, h, y, ss_y, c, u, ss_u, err, total;
  /* NVFP4 weights only (else -1): xn quantised for the pooler (codes [T, D/2], block scales
   * [T, D/16], row scales [T] f32); row scales of xe [T*k] f32 (xe then holds codes
   * [T*k, L/2] and xe_scale block scales [T*k, L/16]); h block scales [T*k, I/16] (h holds
   * codes [T*k, I/2]); c block scales [T, L/16] and row scales [T] (c holds codes [T, L/2]). */
  long long xq, xq_scale, xq_rowscale, xe_rowscale, h_scale, c_scale, c_rowscale;
  int xa_cols; /* columns of one xa row (2*D: xn_hi | xn_lo, or 3*D for fp32 weights) */
  /* [2] int32: the split-K counts the grouped gate/up and down GEMMs used in the last call
   * (chosen on the device from the live tile count; 1 = unsplit; NVFP4 weights only) */
  long long grouped_splits;
} lmoe_workspace_layout;
lmoe_status lmoe_get_workspace_layout(const lmoe_config* cfg, lmoe_workspace_layout* layout);

/* NVFP4 quantisation of fp32 rows with the activation rule the block applies (one fp32
 * scale per row s = amax/(6*448) when row_scale != 0, else s = 1; one E4M3 scale per 16
 * elements sc = E4M3(amax_16/(6 s)); codes E2M1((v * (1/sc)) * (1/s)); each rounding in fp32,
 * round to nearest even, saturating).  Format: LMSYS post, "NVFP4 as a third MMA type".
 * Device pointers: src [rows, K] f32 (K a multiple of 16, at most 32768); codes [rows, K/2]
 * (even element in the low nibble); scales [rows, K/16] E4M3 codes; s_row [rows] f32 (may
 * be NULL).  Also a way to pack weights: with row_scale = 0 the tensor scale is 1.        */
lmoe_status lmoe_quantize_nvfp4(const float* src, long long rows, int K, int row_scale,
                                uint8_t* codes, uint8_t* scales, float* s_row,
                                cudaStream_t stream);

/* Converts row-major E4M3 block scales [rows, K/16] (device) into the block layout that
 * lmoe_nvfp4_weight.scales uses, with blocks of block_rows = 128 or 64 rows (device,
 * (rows/block_rows) * (K/64) * 512 bytes: rows*K/16 for 128, twice that for 64; may not alias
 * src).  rows must be a multiple of block_rows and K of 64.  Asynchronous on `stream`; a
 * one-time weight preparation.                                                            */
lmoe_status lmoe_nvfp4_block_scales(const uint8_t* src, long long rows, int K, int block_rows,
                                    uint8_t* dst, cudaStream_t stream);

/* Diagnostic of the device wait-timeout path: launches one CTA that waits on an
 * mbarrier nothing ever arrives on, with a budget of `budget_cycles` SM cycles
 * (clamped to 1..4e9).  The wait gives up, sets the workspace error word, and the
 * kernel returns; lmoe_check_status() then reports LMOE_ERR_TIMEOUT.  workspace as for
 * latent_moe_forward (only its error word is touched).                               */
lmoe_status lmoe_wait_selftest(const lmoe_config* cfg, void* workspace, long long budget_cycles,
                               cudaStream_t stream);

/* Token permutation (expert histogram + stable scatter) that allocates nothing, for callers
 * that cannot allocate device memory: code whose memory is planned up front by a framework
 * that cannot hand out one more buffer, plug-ins that may not allocate after start-up, and
 * loops that cannot afford an allocation's implicit synchronisation.  The pages have no
 * counterpart of this entry point; it is a packaging of the block's permutation step.
 * Device pointers:
 *  topk_idx  [T, k] int32   expert id of each (token, slot), every id in [0, E)
 *  offsets   [E + 1] int32  out: first row of each expert in expert-contiguous order;
 *                           offsets[E] = T*k
 *  row_of    [T, k] int32   out: row of pair (t, j); pairs of one expert keep (t, j) order
 *  tok_of    [T*k] int32    out: token of each row
 * The scratch (per-expert counts, M-tile table) is a fixed 64 KiB __device__ array inside
 * the library, held by every GPU that loads the library until the process exits.  Limits:
 * E <= 1024 and T*k <= 65536; larger sizes return LMOE_ERR_UNSUPPORTED before any launch.
 * The four arrays must be 4-byte aligned (else LMOE_ERR_ALIGN) device memory of the current
 * device, and the stream must belong to that device (else LMOE_ERR_ARG), both checked before
 * any launch.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and caches it; make that first call before
 * any stream capture.  Calls after a cudaDeviceReset of the device are not supported (the
 * cached address is then stale).  All calls on a device share the one array and nothing in it
 * needs to start at zero (each call overwrites what it reads), but calls that overlap on the
 * GPU (unordered streams) race on it: order them.  This is the per-expert-scan form of the
 * permutation (each of E CTAs reads every id), whose cost grows as E x T*k: at many pairs it
 * is slower than the chunked permutation the forward call runs from its workspace. */
lmoe_status lmoe_permute_noalloc(const int32_t* topk_idx, int T, int k, int E, int32_t* offsets,
                                 int32_t* row_of, int32_t* tok_of, cudaStream_t stream);

/* Guard bands of the workspace, for memory-safety checks (no counterpart on the pages: a
 * stand-in for a race/bounds sanitiser).  Every sub-buffer of the workspace is followed by
 * LMOE_GUARD_BYTES bytes that no call reads or writes.  Writes *count (host) = the number of
 * bands of a workspace for `cfg` (host_io != 0: the larger host-I/O workspace of
 * lmoe_workspace_size_host_io()) and, when offsets != NULL (host array of `capacity`), the
 * byte offset of each band from the start of the workspace.  A caller (a test) fills the
 * workspace with a known byte pattern, runs the block, and checks that every band still
 * holds it: a changed band is a write past the end of a sub-buffer.                    */
#define LMOE_GUARD_BYTES 256
lmoe_status lmoe_workspace_guards(const lmoe_config* cfg, int host_io, long long* offsets,
                                  int capacity, int* count);

/* Checks the routing structures the last call left in `workspace` (device, as for
 * latent_moe_forward; asynchronous on `stream`) — the structures every later kernel indexes
 * with: expert ids in [0, E); offsets starting at 0, non-decreasing, ending at T*k and
 * equal to the per-expert counts' prefix sums; each (token, slot) pair's row (row_of, the
 * scatter target of the pool norm and the source row of the combine) inside its expert's
 * range, and each row the row of exactly one pair (tok_of); every 128-row and 256-row M tile
 * inside its expert's rows with 1..128 (256) rows, the tiles covering T*k rows, the tile
 * counts within their tables, each expert's first tile a tile of that expert.  Every value is
 * bounds-checked before it is followed.  A violation sets bit 0x20 of the error word
 * (lmoe_check_status then returns LMOE_ERR_ARG).  A library built with
 * -DLMOE_BOUNDS_CHECKS=1 runs this check inside every forward call, right after the
 * permutation, and on a violation also replaces the call's routing by one that the later
 * kernels read in bounds (the output is then meaningless and the status says so).  No
 * counterpart on the pages: a stand-in for a device bounds sanitiser.                   */
lmoe_status lmoe_validate_routing(const lmoe_config* cfg, void* workspace, cudaStream_t stream);

/* Number of kernels this library has launched in this process (all devices, all calls). */
unsigned long long lmoe_kernel_launches(void);

/* Human-readable name of a status code (static string). */
const char* lmoe_status_string(lmoe_status s);

#ifdef __cplusplus
}
#endif
#endif /* LATENT_MOE_H_ */
