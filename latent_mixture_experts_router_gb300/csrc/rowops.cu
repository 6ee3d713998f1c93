// rowops.cu — memory-bound kernels of the latent-MoE block: one row (token) per
// CTA or per warp, 16-byte vector loads and stores, fp32 arithmetic, fixed
// reduction orders (results do not depend on scheduling).
//
// Block structure they implement (LMSYS "SGLang and Miles Add Day-0 Support for
// Muse Spark Open", section "MoE with pooler, unpooler and per-expert
// normalization"; vLLM "Day 0 support for Muse Spark Open", "Sandwich
// normalization"):
//   prenorm            xn = x / sqrt(mean(x^2) + eps) * g_pre, written as a bf16
//                      hi/lo pair so that the router sees xn to ~fp32 accuracy
//   topk               softmax over all experts, top-k (ties -> lower index),
//                      weights renormalised over the k
//   permute            expert-contiguous order of the (token, slot) pairs:
//                      per-expert histogram, exclusive scan, stable scatter (one CTA
//                      per expert, or chunked for many pairs; same order either way)
//   poolnorm_scatter   h0 = p / sqrt(mean(p^2) + eps) * g_pool, copied to the
//                      k expert-contiguous rows of the token
//   combine            c = sum_j w_j * g_expert[e_j] * y_j / sqrt(mean(y_j^2) + eps)
//                      in fp32, slot order (per-expert norm BEFORE weighting)
//   postnorm_residual  out = x + u / sqrt(mean(u^2) + eps) * g_post
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace lmoe {

namespace {

constexpr int kRowThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
  // fixed-order reduction: warp butterfly, then warp 0 over the warp partials
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  if (w == 0) {
    t = (l < (int)(blockDim.x >> 5)) ? red[l] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (l == 0) red[32] = t;
  }
  __syncthreads();
  return red[32];
}

__device__ __forceinline__ int block_sum_int(int v, int* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    int t = (l < (int)(blockDim.x >> 5)) ? red[l] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (l == 0) red[32] = t;
  }
  __syncthreads();
  return red[32];
}

// 8 consecutive elements of a row as fp32
__device__ __forceinline__ void load8(const void* base, bool f32, long long i, float (&v)[8]) {
  if (f32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
    const float4 a = p[0], b = p[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 q = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(h[j]);
      v[2 * j] = f.x;
      v[2 * j + 1] = f.y;
    }
  }
}
__device__ __forceinline__ void load8_bf16(const __nv_bfloat16* p, float (&v)[8]) {
  load8(p, false, 0, v);
}
__device__ __forceinline__ void store8_bf16(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 q;
  q.x = pack_bf16x2(v[0], v[1]);
  q.y = pack_bf16x2(v[2], v[3]);
  q.z = pack_bf16x2(v[4], v[5]);
  q.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = q;
}
__device__ __forceinline__ void load8_f32(const float* p, float (&v)[8]) { load8(p, true, 0, v); }
__device__ __forceinline__ void store8_f32(float* p, const float (&v)[8]) {   // p 16-byte aligned
  float4* q = reinterpret_cast<float4*>(p);
  q[0] = make_float4(v[0], v[1], v[2], v[3]);
  q[1] = make_float4(v[4], v[5], v[6], v[7]);
}

constexpr int kCombineBatch = 4;          // slots per batch of loads at few tokens (8 columns)
constexpr int kCombineBatchMaxT = 512;    // "few": a token per CTA (or per cluster) fills no GPU

// acc[0, NC) += sum over slots j (in slot order) of coef[j] * y[row[j]][i, i+NC) * g[e[j]][i, i+NC)
// (NC = 8 or 16; y fp32, or bf16 when !YF32).  The loads of NB slots are issued together, before their multiply-adds.
// NB > 1 for few tokens, where the combine is a chain of round trips and more loads in
// flight shorten it; NB = 1 for many, where the registers would halve the CTAs an SM holds.
template <int NC, int NB, bool YF32 = true>
__device__ __forceinline__ void combine_cols(const void* __restrict__ y, const float* __restrict__ g_expert,
                                             int L, int i, int k, const int* rows, const int* es,
                                             const float* coef, float (&acc)[NC]) {
  static_assert(NC == 8 || NC == 16, "columns per thread");
  for (int j0 = 0; j0 < k; j0 += NB) {
    float v[NB][NC], gg[NB][NC];
#pragma unroll
    for (int jj = 0; jj < NB; ++jj)
      if (j0 + jj < k) {
#pragma unroll
        for (int h = 0; h < NC / 8; ++h) {
          float a[8], b[8];
          load8(y, YF32, static_cast<long long>(rows[j0 + jj]) * L + i + 8 * h, a);
          load8_f32(g_expert + static_cast<long long>(es[j0 + jj]) * L + i + 8 * h, b);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            v[jj][8 * h + q] = a[q];
            gg[jj][8 * h + q] = b[q];
          }
        }
      }
#pragma unroll
    for (int jj = 0; jj < NB; ++jj)
      if (j0 + jj < k) {
#pragma unroll
        for (int q = 0; q < NC; ++q) acc[q] = fmaf(coef[j0 + jj], v[jj][q] * gg[jj][q], acc[q]);
      }
  }
}

// Sum of the n partials p[0, n) by one warp: lane-strided loads (one round trip for n <= 32),
// then a shuffle tree; lane 0's result, broadcast, so every lane returns the same value and
// the order is the same on every call.
__device__ __forceinline__ float warp_sum_partials(const float* __restrict__ p, int n, int lane) {
  float v = 0.f;
  for (int q = lane; q < n; q += 32) v += p[q];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return __shfl_sync(0xffffffffu, v, 0);
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    float t = (l < (int)(blockDim.x >> 5)) ? red[l] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (l == 0) red[32] = t;
  }
  __syncthreads();
  return red[32];
}

// ------------------------------------------------------------------ row slices
// A row kernel runs C CTAs per token (C = 1, 2, 4 or 8, chosen by the launcher from T so
// that a few tokens still spread over many SMs): CTA blockIdx.x = t * C + c handles the
// columns [c N / C, (c + 1) N / C) of token t.  Kernels that reduce over the row are
// launched as clusters of C CTAs and combine the CTAs' partial sums (maxima) through
// distributed shared memory in rank order, so every CTA of the token gets the same value.
struct RowSlice {
  long long t;
  int c, i0, i1;
};
__device__ __forceinline__ RowSlice row_slice(int N, int C) {
  RowSlice r;
  r.t = blockIdx.x / C;
  r.c = static_cast<int>(blockIdx.x % C);
  const int w = N / C;
  r.i0 = r.c * w;
  r.i1 = r.i0 + w;
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// A float of the shared memory of cluster CTA `rank` (same variable as *p in this CTA)
__device__ __forceinline__ float dsmem_ld(const float* p, int rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
  return v;
}
// Cluster-wide sum (is_max: maximum of non-negative values) of v, which every thread of a
// CTA holds; `slot` is a __shared__ float used by this one reduction only.  Every thread of
// every CTA of the cluster calls it.  A kernel that calls it ends with cluster_sync_all(),
// so that no CTA leaves while another still reads its slot.
__device__ __forceinline__ float cluster_combine(float v, float* slot, int C, bool is_max) {
  if (C == 1) return v;
  if (threadIdx.x == 0) *slot = v;
  cluster_sync_all();
  float r = 0.f;
  for (int q = 0; q < C; ++q) {
    const float o = dsmem_ld(slot, q);
    r = is_max ? fmaxf(r, o) : r + o;
  }
  return r;
}

// ------------------------------------------------------------------ prenorm
// One CTA per token.  xa row = [xn_hi | xn_lo] (or [hi | lo | hi] when xa_cols = 3D,
// to pair with router weights split as [W_hi | W_hi | W_lo]).
__global__ void __launch_bounds__(kRowThreads) prenorm_kernel(const void* __restrict__ x, int x_f32,
                                                              const float* __restrict__ g,
                                                              int D, float eps,
                                                              __nv_bfloat16* __restrict__ xa,
                                                              int xa_cols, unsigned* status2, int C) {
  griddep_enter();
  if (status2 != nullptr && blockIdx.x == 0 && threadIdx.x == 0) status2[0] = status2[1] = 0u;
  __shared__ float red[33];
  __shared__ float slot_ss;
  const RowSlice sl = row_slice(D, C);
  const long long t = sl.t;
  const long long xoff = t * D;
  float ss = 0.f;
  for (int i = sl.i0 + threadIdx.x * 8; i < sl.i1; i += kRowThreads * 8) {
    float v[8];
    load8(x, x_f32, xoff + i, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(v[j], v[j], ss);
  }
  const float rs =
      rsqrtf(cluster_combine(block_sum(ss, red), &slot_ss, C, false) / static_cast<float>(D) + eps);
  __nv_bfloat16* row = xa + t * xa_cols;
  for (int i = sl.i0 + threadIdx.x * 8; i < sl.i1; i += kRowThreads * 8) {
    float v[8], gg[8], hi[8], lo[8];
    load8(x, x_f32, xoff + i, v);
    load8_f32(g + i, gg);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float xn = v[j] * rs * gg[j];
      hi[j] = bf16_round(xn);
      lo[j] = xn - hi[j];
    }
    store8_bf16(row + i, hi);
    store8_bf16(row + D + i, lo);
    if (xa_cols == 3 * D) store8_bf16(row + 2 * D + i, hi);
  }
  if (C > 1) cluster_sync_all();
}

// ------------------------------------------------------------------ top-k + softmax
// One warp per token.  Selection: k rounds of a warp arg-max over (value desc,
// index asc); the (k+1)-th round gives the margin for the near-tie count.
constexpr int kTopkWarps = 4;

// The top-k of one token, computed by one warp: vals[E] (shared memory, overwritten) holds
// the token's logits (+ bias); forced_row, if set, holds its k experts.  Lane 0 writes the
// experts (descending logit) and their softmax weights renormalised over the k.
__device__ __forceinline__ void warp_topk(float* vals, const int32_t* forced_row, int E, int k,
                                          long long t, int lane, int32_t* idx_out, float* w_out,
                                          int32_t* near_tie, int32_t* idx_copy, float* w_copy,
                                          unsigned* err) {
  int sel[16];
  float sval[16];
  if (forced_row != nullptr) {
    for (int j = 0; j < k; ++j) {
      int e = forced_row[j];
      if (e < 0 || e >= E) {  // an id outside [0, E) would index out of bounds downstream
        if (lane == 0) atomicOr(err, kErrBadIndex);
        e = 0;
      }
      // a repeated id breaks the one-row-per-token-and-expert bound the GEMM tiles rely on
      for (int i = 0; i < j; ++i)
        if (sel[i] == e && lane == 0) atomicOr(err, kErrBadIndex);
      sel[j] = e;
      sval[j] = vals[e];
    }
  } else {
    // A NaN logit (a NaN or infinity in the token's input) orders below every number, as -inf;
    // an expert already selected is marked NaN and skipped, so every round picks a valid index
    // distinct from the earlier ones even when all logits are -inf or NaN.
    for (int i = lane; i < E; i += 32)
      if (vals[i] != vals[i]) vals[i] = -INFINITY;
    __syncwarp();
    const int rounds = (k < E) ? k + 1 : k;
    for (int j = 0; j < rounds; ++j) {
      float best = -INFINITY;
      int bi = 0x7fffffff;
      for (int i = lane; i < E; i += 32) {
        const float v = vals[i];
        if (v != v) continue;   // selected in an earlier round
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
        sel[j] = bi;
        sval[j] = best;
        if (lane == 0) vals[bi] = __int_as_float(0x7fc00000);   // NaN: taken
        __syncwarp();
      } else if (lane == 0 && near_tie != nullptr && (sval[k - 1] - best) < 1e-3f) {
        atomicAdd(near_tie, 1);
      }
    }
  }
  if (lane == 0) {
    float m = sval[0];
    for (int j = 1; j < k; ++j) m = fmaxf(m, sval[j]);
    float ex[16], sum = 0.f;
    for (int j = 0; j < k; ++j) {
      ex[j] = expf(sval[j] - m);
      sum += ex[j];
    }
    const float inv = 1.f / sum;
    for (int j = 0; j < k; ++j) {
      idx_out[t * k + j] = sel[j];
      w_out[t * k + j] = ex[j] * inv;
      if (idx_copy) idx_copy[t * k + j] = sel[j];
      if (w_copy) w_copy[t * k + j] = ex[j] * inv;
    }
  }
}

__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(
    const float* __restrict__ logits, int ld, const float* __restrict__ bias,
    const int32_t* __restrict__ forced, int T, int E, int k, int32_t* __restrict__ idx_out,
    float* __restrict__ w_out, int32_t* __restrict__ near_tie, int32_t* __restrict__ idx_copy,
    float* __restrict__ w_copy, unsigned* __restrict__ err) {
  griddep_enter();
  extern __shared__ float vals_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long t = static_cast<long long>(blockIdx.x) * kTopkWarps + warp;
  if (t >= T) return;
  float* vals = vals_all + warp * E;
  for (int i = lane; i < E; i += 32) vals[i] = logits[t * ld + i] + (bias ? bias[i] : 0.f);
  __syncwarp();
  warp_topk(vals, forced ? forced + t * k : nullptr, E, k, t, lane, idx_out, w_out, near_tie,
            idx_copy, w_copy, err);
}

// ------------------------------------------------------------------ permutation
// Pairs (t, j) are numbered i = t*k + j.  Expert e owns rows [off[e], off[e] + cnt[e])
// of the expert-contiguous matrices, in increasing i (stable, so deterministic).
constexpr int kPermThreads = 256;

// Order of the table of 256-row tiles (grouped BF16 GEMMs over many rows).  An expert's tiles
// with more than 128 live rows ("full": MMA-bound, and those of one expert share its weights
// in L2) and its last tile when it holds at most 128 rows ("light": it streams the expert's
// weights for few rows) are interleaved in runs of kMixRun, so that every wave of the
// persistent GEMM mixes tensor-bound and memory-bound tiles instead of alternating between
// phases of each.  Full tile j (in expert order) and light tile i go to these places:
constexpr int kMixRun = 8;
__device__ __forceinline__ int mixed_pos_full(int j, int n_light) {
  return j + min((j / kMixRun) * kMixRun, n_light);
}
__device__ __forceinline__ int mixed_pos_light(int i, int n_full) {
  return i + min((i / kMixRun + 1) * kMixRun, n_full);
}
// (full, light) tile counts of an expert with c rows
__device__ __forceinline__ void tile2_counts(int c, int& full, int& light) {
  const int nt2 = (c + 2 * kBM - 1) / (2 * kBM), rem = c % (2 * kBM);
  light = (rem > 0 && rem <= kBM) ? 1 : 0;
  full = nt2 - light;
}
// writes the 256-row tiles of expert e (c rows from row `off`) given the full and light
// tiles of the experts before it (f0, l0) and the totals (nf, nl)
__device__ __forceinline__ void write_tiles2(Tile* tiles2, int e, int off, int c, int f0, int l0, int nf,
                                             int nl, int first, int step) {
  int full, light;
  tile2_counts(c, full, light);
  for (int m = first; m < full + light; m += step) {
    const int pos = m < full ? mixed_pos_full(f0 + m, nl) : mixed_pos_light(l0, nf);
    tiles2[pos] = Tile{e, off + m * 2 * kBM, min(2 * kBM, c - m * 2 * kBM), 0};
  }
}

__global__ void __launch_bounds__(kPermThreads) expert_count_kernel(const int32_t* __restrict__ idx,
                                                                    int n, int32_t* counts) {
  griddep_enter();
  __shared__ int red[33];
  const int e = blockIdx.x;
  int c = 0;
  for (int i = threadIdx.x; i < n; i += kPermThreads) c += (idx[i] == e);
  const int tot = block_sum_int(c, red);
  if (threadIdx.x == 0) counts[e] = tot;
}

__global__ void __launch_bounds__(kPermThreads) expert_scatter_kernel(
    const int32_t* __restrict__ idx, int n, int k, int E, const int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ row_of, int32_t* __restrict__ tok_of,
    Tile* __restrict__ tiles, int32_t* __restrict__ n_tiles, int32_t* __restrict__ tile_base,
    Tile* __restrict__ tiles2, int32_t* __restrict__ n_tiles2) {
  griddep_enter();
  __shared__ int wsum[kPermThreads / 32];
  __shared__ int red[33];
  const int e = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int my_off = 0, my_t0 = 0, my_f0 = 0, my_l0 = 0, my_nf = 0, my_nl = 0;
  for (int q = threadIdx.x; q < E; q += kPermThreads) {
    int f, l;
    tile2_counts(counts[q], f, l);
    my_nf += f;
    my_nl += l;
    if (q < e) {
      my_off += counts[q];
      my_t0 += (counts[q] + kBM - 1) / kBM;
      my_f0 += f;
      my_l0 += l;
    }
  }
  const int off = block_sum_int(my_off, red);
  const int tile0 = block_sum_int(my_t0, red);
  const int f0 = block_sum_int(my_f0, red), l0 = block_sum_int(my_l0, red);
  const int nf = block_sum_int(my_nf, red), nl = block_sum_int(my_nl, red);
  const int cnt = counts[e];
  if (threadIdx.x == 0) {
    offsets[e] = off;
    if (tile_base != nullptr) tile_base[e] = tile0;   // first M tile of expert e
    if (e == E - 1) {
      offsets[E] = off + cnt;
      *n_tiles = tile0 + (cnt + kBM - 1) / kBM;
      if (n_tiles2 != nullptr) *n_tiles2 = nf + nl;
    }
  }
  const int ntile = (cnt + kBM - 1) / kBM;
  for (int m = threadIdx.x; m < ntile; m += kPermThreads)
    tiles[tile0 + m] = Tile{e, off + m * kBM, min(kBM, cnt - m * kBM), 0};
  if (tiles2 != nullptr) write_tiles2(tiles2, e, off, cnt, f0, l0, nf, nl, threadIdx.x, kPermThreads);
  if (cnt == 0) return;
  // The pairs split into one contiguous segment per warp (a multiple of 128 pairs, so that a
  // lane reads four at a time): a first pass counts the segment's pairs of expert e, a scan
  // over the warps gives each segment its first row, and a second pass ranks the pairs in
  // order (lane-major, four per lane) within each 128-pair chunk; one block barrier in all.
  constexpr int kWarps = kPermThreads / 32;
  const int seg = (n + kWarps * 128 - 1) / (kWarps * 128) * 128;
  const int s0 = warp * seg, s1 = min(n, s0 + seg);
  const bool vec = (reinterpret_cast<uintptr_t>(idx) & 15u) == 0;   // idx may come from a caller
  auto match4 = [&](int c) {   // bit q: pair c + 4 lane + q belongs to expert e
    const int i = c + 4 * lane;
    uint32_t m = 0;
    if (vec && i + 3 < n) {
      const int4 v = *reinterpret_cast<const int4*>(idx + i);
      m = (v.x == e ? 1u : 0u) | (v.y == e ? 2u : 0u) | (v.z == e ? 4u : 0u) | (v.w == e ? 8u : 0u);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (i + q < n && idx[i + q] == e) m |= 1u << q;
    }
    return m;
  };
  int c_w = 0;
  for (int c = s0; c < s1; c += 128) c_w += __popc(match4(c));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c_w += __shfl_xor_sync(0xffffffffu, c_w, o);
  if (lane == 0) wsum[warp] = c_w;
  __syncthreads();
  int r0 = off;
  for (int q = 0; q < warp; ++q) r0 += wsum[q];
  for (int c = s0; c < s1; c += 128) {
    uint32_t m = match4(c);
    const int mine = __popc(m);
    int incl = mine;   // inclusive scan over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int r = r0 + incl - mine;
    while (m) {
      const int q = __ffs(m) - 1;
      m &= m - 1;
      const int i = c + 4 * lane + q;
      row_of[i] = r;
      tok_of[r] = i / k;
      ++r;
    }
    r0 += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// ------------------------------------------------------------------ routing for few tokens
// With few (token, slot) pairs one CTA performs S3 and S4 together, saving two launches on
// the latency-bound chain: each warp selects the top-k of its tokens (warp_topk), then the
// CTA counts the pairs per expert, scans the counts into offsets and first M tiles, writes
// the tile table and gives pair i the row offsets[e] + #{j < i : idx[j] = e} (the stable
// order of the expert_count / expert_scatter path, so both paths give identical results).
constexpr int kRouteThreads = 512;
constexpr int kRouteMaxPairs = 256;

// Exclusive block scan of (a, b) over the threads' values, in thread order; returns the
// totals through *ta, *tb.  Every thread of the block calls it.
__device__ __forceinline__ void block_scan2(int& a, int& b, int* sh, int* ta, int* tb) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ya = __shfl_up_sync(0xffffffffu, ia, o), yb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += ya;
      ib += yb;
    }
  }
  __syncthreads();
  if (lane == 31) {
    sh[warp] = ia;
    sh[32 + warp] = ib;
  }
  __syncthreads();
  int pa = 0, pb = 0, sa = 0, sb = 0;
  for (int q = 0; q < nw; ++q) {
    if (q < warp) {
      pa += sh[q];
      pb += sh[32 + q];
    }
    sa += sh[q];
    sb += sh[32 + q];
  }
  a = pa + ia - a;
  b = pb + ib - b;
  *ta = sa;
  *tb = sb;
}

// logits[t][i] = sum over q in split order of part[q][t][i]; element ti = t * E + i; M logits per
// thread and J splits per round of loads
template <int M, int J>
__device__ __forceinline__ void route_sum_partials(const float* __restrict__ part, int splits, int te, int E,
                                                   float* __restrict__ logits, int ld) {
  for (int g0 = 0; g0 < te; g0 += M * kRouteThreads) {
    float v[M];
#pragma unroll
    for (int m = 0; m < M; ++m) v[m] = 0.f;
    for (int q0 = 0; q0 < splits; q0 += J) {
      float pv[M][J];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const int ti = g0 + m * kRouteThreads + threadIdx.x;
#pragma unroll
        for (int j = 0; j < J; ++j)
          pv[m][j] = (ti < te && q0 + j < splits) ? part[static_cast<long long>(q0 + j) * te + ti] : 0.f;
      }
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int j = 0; j < J; ++j)
          if (q0 + j < splits) v[m] += pv[m][j];
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int ti = g0 + m * kRouteThreads + threadIdx.x;
      if (ti < te) logits[static_cast<long long>(ti / E) * ld + ti % E] = v[m];
    }
  }
}

__global__ void __launch_bounds__(kRouteThreads) route_small_kernel(
    float* __restrict__ logits, int ld, const float* __restrict__ rpart, int rsplits,
    const float* __restrict__ bias,
    const int32_t* __restrict__ forced, int T, int E, int k, int32_t* __restrict__ idx_out,
    float* __restrict__ w_out, int32_t* __restrict__ near_tie, int32_t* __restrict__ idx_copy,
    float* __restrict__ w_copy, unsigned* __restrict__ err, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ row_of, int32_t* __restrict__ tok_of,
    Tile* __restrict__ tiles, int32_t* __restrict__ n_tiles, int32_t* __restrict__ tile_base,
    Tile* __restrict__ tiles2, int32_t* __restrict__ n_tiles2) {
  griddep_enter();
  extern __shared__ float route_sh[];
  constexpr int nw = kRouteThreads / 32;
  float* vals_all = route_sh;                                         // [nw][E]
  int* cnt_s = reinterpret_cast<int*>(route_sh + nw * E);             // [E]
  int* off_s = cnt_s + E;                                             // [E]
  int* idx_s = off_s + E;                                             // [kRouteMaxPairs]
  __shared__ int scan_sh[64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = T * k;
  // S3: a warp per token
  if (rsplits > 1) {
    // the router's split-K partials [rsplits][T][E], summed in split order (as the reduction
    // kernel does) by every thread of the CTA: a chain of dependent L2 round trips, so each
    // thread keeps 32 loads in flight per round (fewer logits per thread, more splits a round)
    const int te = T * E;
    if (te <= kRouteThreads) route_sum_partials<1, 32>(rpart, rsplits, te, E, logits, ld);
    else if (te <= 2 * kRouteThreads) route_sum_partials<2, 16>(rpart, rsplits, te, E, logits, ld);
    else route_sum_partials<4, 8>(rpart, rsplits, te, E, logits, ld);
    __syncthreads();
  }
  for (int t = warp; t < T; t += nw) {
    float* vals = vals_all + warp * E;
    for (int i = lane; i < E; i += 32) vals[i] = logits[static_cast<long long>(t) * ld + i] + (bias ? bias[i] : 0.f);
    __syncwarp();
    warp_topk(vals, forced ? forced + static_cast<long long>(t) * k : nullptr, E, k, t, lane, idx_out, w_out,
              near_tie, idx_copy, w_copy, err);
    __syncwarp();
  }
  for (int e = threadIdx.x; e < E; e += kRouteThreads) cnt_s[e] = 0;
  __syncthreads();   // idx_out of every token written (global, this CTA) and counts zeroed
  for (int i = threadIdx.x; i < n; i += kRouteThreads) {
    const int e = idx_out[i];
    idx_s[i] = e;
    atomicAdd(&cnt_s[e], 1);
  }
  __syncthreads();
  // S4: offsets and first M tiles by an exclusive scan over the experts (thread-contiguous
  // runs of experts, so thread order is expert order)
  const int per = (E + kRouteThreads - 1) / kRouteThreads;
  const int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
  int a = 0, b = 0, f = 0, l = 0;
  for (int e = e0; e < e1; ++e) {
    int fe, le;
    tile2_counts(cnt_s[e], fe, le);
    a += cnt_s[e];
    b += (cnt_s[e] + kBM - 1) / kBM;
    f += fe;
    l += le;
  }
  int ta, tb, nf, nl;
  block_scan2(a, b, scan_sh, &ta, &tb);
  block_scan2(f, l, scan_sh, &nf, &nl);
  for (int e = e0; e < e1; ++e) {
    const int c = cnt_s[e], nt = (c + kBM - 1) / kBM;
    int fe, le;
    tile2_counts(c, fe, le);
    off_s[e] = a;
    counts[e] = c;
    offsets[e] = a;
    if (tile_base != nullptr) tile_base[e] = b;
    for (int m = 0; m < nt; ++m) tiles[b + m] = Tile{e, a + m * kBM, min(kBM, c - m * kBM), 0};
    if (tiles2 != nullptr) write_tiles2(tiles2, e, a, c, f, l, nf, nl, 0, 1);
    a += c;
    b += nt;
    f += fe;
    l += le;
  }
  if (threadIdx.x == 0) {
    offsets[E] = ta;
    *n_tiles = tb;
    if (n_tiles2 != nullptr) *n_tiles2 = nf + nl;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kRouteThreads) {
    const int e = idx_s[i];
    int rank = 0;
    for (int j = 0; j < i; ++j) rank += (idx_s[j] == e);
    const int r = off_s[e] + rank;
    row_of[i] = r;
    tok_of[r] = i / k;
  }
}

// ------------------------------------------------------------------ permutation of many pairs
// With many pairs the per-expert CTAs above all read the whole id array at once.  Instead the
// pairs are cut into chunks of kPermChunk: each chunk CTA histograms its ids in shared memory
// (perm_hist), one CTA turns the chunk histograms into per-chunk bases and the expert offsets
// and tile tables (perm_scan), and each chunk CTA ranks its pairs (perm_rank): warp w of the
// chunk takes 32 consecutive pairs at a time, ranks them among the warp's pairs of the same
// expert by match-any ballots, and adds the counts of the earlier warps, earlier chunks and
// earlier experts.  Same (expert, pair index) order, so the same outputs as the path above.
constexpr int kPermChunk = 2048;           // 8 warps x 8 rounds x 32 pairs
constexpr int kPermScanThreads = 1024;

__global__ void __launch_bounds__(kPermThreads) perm_hist_kernel(const int32_t* __restrict__ idx, int n, int E,
                                                                 int32_t* __restrict__ hist) {
  griddep_enter();
  extern __shared__ int h_sh[];   // [E]
  for (int e = threadIdx.x; e < E; e += kPermThreads) h_sh[e] = 0;
  __syncthreads();
  const long long c0 = static_cast<long long>(blockIdx.x) * kPermChunk;
#pragma unroll
  for (int j = 0; j < kPermChunk / kPermThreads; ++j) {
    const long long i = c0 + j * kPermThreads + threadIdx.x;
    if (i < n) atomicAdd(&h_sh[idx[i]], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kPermThreads) hist[static_cast<long long>(blockIdx.x) * E + e] = h_sh[e];
}

__global__ void __launch_bounds__(kPermScanThreads) perm_scan_kernel(
    const int32_t* __restrict__ hist, int chunks, int E, int32_t* __restrict__ base,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, Tile* __restrict__ tiles,
    int32_t* __restrict__ n_tiles, int32_t* __restrict__ tile_base, Tile* __restrict__ tiles2,
    int32_t* __restrict__ n_tiles2) {
  griddep_enter();
  __shared__ int scan_sh[64];
  // thread-contiguous runs of experts, so that thread order is expert order in the scans
  const int per = (E + kPermScanThreads - 1) / kPermScanThreads;
  const int e0 = min(E, static_cast<int>(threadIdx.x) * per), e1 = min(E, e0 + per);
  int a = 0, b = 0, f = 0, l = 0;
  for (int e = e0; e < e1; ++e) {
    int run = 0;   // chunk bases of expert e: pairs of e in the earlier chunks
    for (int g = 0; g < chunks; ++g) {
      const long long q = static_cast<long long>(g) * E + e;
      const int c = hist[q];
      base[q] = run;
      run += c;
    }
    counts[e] = run;
    int fe, le;
    tile2_counts(run, fe, le);
    a += run;
    b += (run + kBM - 1) / kBM;
    f += fe;
    l += le;
  }
  int ta, tb, nf, nl;
  block_scan2(a, b, scan_sh, &ta, &tb);
  block_scan2(f, l, scan_sh, &nf, &nl);
  for (int e = e0; e < e1; ++e) {
    const int c = counts[e], nt = (c + kBM - 1) / kBM;   // this thread's own store above
    int fe, le;
    tile2_counts(c, fe, le);
    offsets[e] = a;
    if (tile_base != nullptr) tile_base[e] = b;
    for (int m = 0; m < nt; ++m) tiles[b + m] = Tile{e, a + m * kBM, min(kBM, c - m * kBM), 0};
    if (tiles2 != nullptr) write_tiles2(tiles2, e, a, c, f, l, nf, nl, 0, 1);
    a += c;
    b += nt;
    f += fe;
    l += le;
  }
  if (threadIdx.x == 0) {
    offsets[E] = ta;
    *n_tiles = tb;
    if (n_tiles2 != nullptr) *n_tiles2 = nf + nl;
  }
}

__global__ void __launch_bounds__(kPermThreads) perm_rank_kernel(
    const int32_t* __restrict__ idx, int n, int k, int E, const int32_t* __restrict__ base,
    const int32_t* __restrict__ offsets, int32_t* __restrict__ row_of, int32_t* __restrict__ tok_of) {
  griddep_enter();
  extern __shared__ int wc_sh[];   // [8 warps][E]: pairs of each expert the warp has ranked
  constexpr int kWarps = kPermThreads / 32, kRounds = kPermChunk / kPermThreads;
  for (int q = threadIdx.x; q < kWarps * E; q += kPermThreads) wc_sh[q] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long c0 = static_cast<long long>(blockIdx.x) * kPermChunk + warp * (kPermChunk / kWarps);
  int* wc = wc_sh + warp * E;
  int rank[kRounds], ex[kRounds];
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const long long i = c0 + r * 32 + lane;
    const int e = i < n ? idx[i] : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    rank[r] = (e >= 0 ? wc[e] : 0) + __popc(peers & ((1u << lane) - 1u));
    ex[r] = e;
    __syncwarp();   // every lane has read the count before the group's first lane adds to it
    if (e >= 0 && lane == __ffs(peers) - 1) wc[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kPermThreads) {   // exclusive prefix over the warps
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int c = wc_sh[w * E + e];
      wc_sh[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int e = ex[r];
    if (e < 0) continue;
    const long long i = c0 + r * 32 + lane;
    const int row = offsets[e] + base[static_cast<long long>(blockIdx.x) * E + e] + wc[e] + rank[r];
    row_of[i] = row;
    tok_of[row] = static_cast<int32_t>(i / k);
  }
}

// ------------------------------------------------------------------ pool norm + scatter
__global__ void __launch_bounds__(kRowThreads) poolnorm_scatter_kernel(
    const float* __restrict__ p, const float* __restrict__ ss_p, int ld_ss,
    const float* __restrict__ g, const int32_t* __restrict__ row_of, int L, int k, float eps,
    __nv_bfloat16* __restrict__ xe, int C) {
  griddep_enter();
  __shared__ float s_rs;
  __shared__ int s_rows[16];
  const RowSlice sl = row_slice(L, C);
  const long long t = sl.t;
  if (threadIdx.x < 32) {
    const float ss = warp_sum_partials(ss_p + t * ld_ss, ld_ss, threadIdx.x);
    if (threadIdx.x == 0) s_rs = rsqrtf(ss / static_cast<float>(L) + eps);
  }
  if (threadIdx.x < k) s_rows[threadIdx.x] = row_of[t * k + threadIdx.x];
  __syncthreads();
  const float rs = s_rs;
  for (int i = sl.i0 + threadIdx.x * 8; i < sl.i1; i += kRowThreads * 8) {
    float v[8], gg[8];
    load8_f32(p + t * L + i, v);
    load8_f32(g + i, gg);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = v[j] * rs * gg[j];
    for (int j = 0; j < k; ++j) store8_bf16(xe + static_cast<long long>(s_rows[j]) * L + i, v);
  }
}

// ------------------------------------------------------------------ combine
template <int NB>
__global__ void __launch_bounds__(kRowThreads) combine_kernel(
    const float* __restrict__ y, const float* __restrict__ ss_y, int ld_ss,
    const int32_t* __restrict__ row_of, const int32_t* __restrict__ idx,
    const float* __restrict__ w, const float* __restrict__ g_expert, int L, int k, float eps,
    __nv_bfloat16* __restrict__ c, int C) {
  griddep_enter();
  __shared__ float s_coef[16];
  __shared__ int s_row[16], s_e[16];
  const RowSlice sl = row_slice(L, C);
  const long long t = sl.t;
  for (int j = threadIdx.x >> 5; j < k; j += kRowThreads / 32) {   // a warp per slot
    const int lane = threadIdx.x & 31;
    const int row = row_of[t * k + j];
    // (no L2 prefetch of the slot's fp32 row here, unlike the NVFP4 combine: with ~1200
    // resident CTAs the prefetched rows exceed L2, measured 381 -> 410 us at T = 16384)
    const float ss = warp_sum_partials(ss_y + static_cast<long long>(row) * ld_ss, ld_ss, lane);
    if (lane == 0) {
      s_coef[j] = w[t * k + j] * rsqrtf(ss / static_cast<float>(L) + eps);
      s_row[j] = row;
      s_e[j] = idx[t * k + j];
    }
  }
  __syncthreads();
  for (int i = sl.i0 + threadIdx.x * 8; i < sl.i1; i += kRowThreads * 8) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    combine_cols<8, NB>(y, g_expert, L, i, k, s_row, s_e, s_coef, acc);   // slot order
    store8_bf16(c + t * L + i, acc);
  }
}

// ------------------------------------------------------------------ post-norm + residual
__global__ void __launch_bounds__(kRowThreads) postnorm_residual_kernel(
    const void* __restrict__ x, int x_f32, float* __restrict__ u,
    const float* __restrict__ ss_u, int ld_ss, const float* __restrict__ g, int D, float eps,
    void* __restrict__ out, int out_f32, int C, const float* __restrict__ upart, int usplits, int T,
    const float* __restrict__ g_next, void* __restrict__ next_out) {
  griddep_enter();
  __shared__ float s_rs;
  __shared__ float red[33];
  __shared__ float slot_ss, slot_ss2;
  const RowSlice sl = row_slice(D, C);
  const long long t = sl.t;
  float rs;
  if (usplits > 1) {
    // u from the unpooler's split-K partials [usplits][T][D] (split order, as the reduction
    // kernel sums them), written to u; the row's sum of squares over the cluster
    float ss = 0.f;
    for (int i = sl.i0 + threadIdx.x * 8; i < sl.i1; i += kRowThreads * 8) {
      float uv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int q = 0; q < usplits; ++q) {
        float pv[8];
        load8_f32(upart + (static_cast<long long>(q) * T + t) * D + i, pv);
#pragma unroll
        for (int j = 0; j < 8; ++j) uv[j] += pv[j];
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(uv[j], uv[j], ss);
      store8_f32(u + t * D + i, uv);
    }
    rs = rsqrtf(cluster_combine(block_sum(ss, red), &slot_ss, C, false) / static_cast<float>(D) + eps);
  } else {
    if (threadIdx.x < 32) {
      const float ss = warp_sum_partials(ss_u + t * ld_ss, ld_ss, threadIdx.x);
      if (threadIdx.x == 0) s_rs = rsqrtf(ss / static_cast<float>(D) + eps);
    }
    __syncthreads();
    rs = s_rs;
  }
  // out = x + u rs g_post, as stored (bf16 out rounds); with g_next the stored rows also feed
  // the next layer's pre-norm, a second row reduction over the same cluster
  auto out_row = [&](int i, float (&o)[8]) {
    float uv[8], gg[8];
    load8(x, x_f32, t * D + i, o);
    load8_f32(u + t * D + i, uv);   // this thread's own stores when u came from the partials
    load8_f32(g + i, gg);
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = o[j] + uv[j] * rs * gg[j];
    if (!out_f32) {
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] = bf16_round(o[j]);
    }
  };
  float ss2 = 0.f;
  for (int i = sl.i0 + threadIdx.x * 8; i < sl.i1; i += kRowThreads * 8) {
    float o[8];
    out_row(i, o);
    if (out_f32) {
      store8_f32(static_cast<float*>(out) + t * D + i, o);
    } else {
      store8_bf16(static_cast<__nv_bfloat16*>(out) + t * D + i, o);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) ss2 = fmaf(o[j], o[j], ss2);
  }
  if (g_next != nullptr) {
    const float rs2 =
        rsqrtf(cluster_combine(block_sum(ss2, red), &slot_ss2, C, false) / static_cast<float>(D) + eps);
    for (int i = sl.i0 + threadIdx.x * 8; i < sl.i1; i += kRowThreads * 8) {
      float o[8], gg[8];
      out_row(i, o);
      load8_f32(g_next + i, gg);
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] = o[j] * rs2 * gg[j];
      if (out_f32) {
        store8_f32(static_cast<float*>(next_out) + t * D + i, o);
      } else {
        store8_bf16(static_cast<__nv_bfloat16*>(next_out) + t * D + i, o);
      }
    }
  }
  if (C > 1 && (usplits > 1 || g_next != nullptr)) cluster_sync_all();
}

// ------------------------------------------------------------------ fp32 weights -> bf16 hi/lo
// W [rows, K] fp32 -> [rows, parts*K] bf16; part q = W_lo if bit q of lo_mask else W_hi
__global__ void weight_split_kernel(const float* __restrict__ W, long long rows, int K, int parts,
                                    unsigned lo_mask, __nv_bfloat16* __restrict__ dst) {
  griddep_enter();
  const long long chunks = rows * (K / 8);
  for (long long c = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; c < chunks;
       c += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = c / (K / 8);
    const int i = static_cast<int>(c % (K / 8)) * 8;
    float v[8], hi[8], lo[8];
    load8_f32(W + r * K + i, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      hi[j] = bf16_round(v[j]);
      lo[j] = v[j] - hi[j];
    }
    __nv_bfloat16* row = dst + r * parts * K;
    for (int q = 0; q < parts; ++q) store8_bf16(row + static_cast<long long>(q) * K + i, ((lo_mask >> q) & 1) ? lo : hi);
  }
}

// ------------------------------------------------------------------ NVFP4 rows

__device__ __forceinline__ void load_recip(float* recip) {
  for (int i = threadIdx.x; i < 256; i += blockDim.x) recip[i] = g_e4m3_recip.v[i];
}

// Destination row of a quantised row: codes at row `code_row` (pitch K/2 bytes); scales
// row-major at `code_row` (pitch K/16) when blk < 0, else in the block layout at row block
// `blk`, position `m`.
struct QDest {
  long long code_row;
  long long blk;
  int m;
};

// Quantises columns [i0, i1) of a row of K values (buf, shared memory, holds columns i0..)
// with row scale s into `ndst` destination rows.
__device__ __forceinline__ void quantize_row_to(const float* buf, int K, int i0, int i1, float s,
                                                const float* recip, uint8_t* codes, uint8_t* scales,
                                                const QDest* dst, int ndst) {
  const float six_s = __fmul_rn(6.f, s), inv_s = __fdiv_rn(1.f, s);
  for (int b = i0 / 16 + threadIdx.x; b < i1 / 16; b += blockDim.x) {
    float v[16];
    const float4* src = reinterpret_cast<const float4*>(buf + (b * 16 - i0));   // i0 % 16 == 0
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 f = src[i];
      v[4 * i] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
    uint2 q;
    const uint32_t sc = nvfp4_quant16(v, six_s, inv_s, recip, q);
    for (int j = 0; j < ndst; ++j) {
      const QDest d = dst[j];
      *reinterpret_cast<uint2*>(codes + d.code_row * (K / 2) + b * 8) = q;
      const size_t so = d.blk < 0 ? static_cast<size_t>(d.code_row) * (K / 16) + b
                                  : blocked_sf_offset(d.blk, d.m, b, K);
      scales[so] = static_cast<uint8_t>(sc);
    }
  }
}

// Pre-norm that also emits xn in NVFP4 (row scale per token) for the pooler, besides the
// bf16 hi/lo pair the router reads.  Dynamic smem: D + 256 floats.
__global__ void __launch_bounds__(kRowThreads) prenorm_nvfp4_kernel(
    const void* __restrict__ x, int x_f32, const float* __restrict__ g, int D, float eps,
    __nv_bfloat16* __restrict__ xa, int xa_cols, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, float* __restrict__ s_row, unsigned* status2, int C) {
  griddep_enter();
  if (status2 != nullptr && blockIdx.x == 0 && threadIdx.x == 0) status2[0] = status2[1] = 0u;
  extern __shared__ float dyn[];
  const RowSlice sl = row_slice(D, C);
  float* buf = dyn;                  // this CTA's columns
  float* recip = dyn + (sl.i1 - sl.i0);
  __shared__ float red[33];
  __shared__ float slot_ss, slot_amax;
  __shared__ QDest s_d;
  load_recip(recip);
  const long long t = sl.t;
  const long long xoff = t * D;
  float ss = 0.f;
  for (int i = sl.i0 + threadIdx.x * 8; i < sl.i1; i += kRowThreads * 8) {
    float v[8];
    load8(x, x_f32, xoff + i, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(v[j], v[j], ss);
  }
  const float rs =
      rsqrtf(cluster_combine(block_sum(ss, red), &slot_ss, C, false) / static_cast<float>(D) + eps);
  __nv_bfloat16* row = xa + t * xa_cols;
  float amax = 0.f;
  for (int i = sl.i0 + threadIdx.x * 8; i < sl.i1; i += kRowThreads * 8) {
    float v[8], gg[8], hi[8], lo[8];
    load8(x, x_f32, xoff + i, v);
    load8_f32(g + i, gg);
    float xn[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      xn[j] = v[j] * rs * gg[j];
      amax = fmaxf(amax, fabsf(xn[j]));
      hi[j] = bf16_round(xn[j]);
      lo[j] = xn[j] - hi[j];
    }
    store8_f32(buf + (i - sl.i0), xn);
    store8_bf16(row + i, hi);
    store8_bf16(row + D + i, lo);
  }
  const float s = nvfp4_row_scale(cluster_combine(block_max(amax, red), &slot_amax, C, true));
  if (threadIdx.x == 0) {
    if (sl.c == 0) s_row[t] = s;
    s_d = QDest{t, t / kBM, static_cast<int>(t % kBM)};
  }
  __syncthreads();
  quantize_row_to(buf, D, sl.i0, sl.i1, s, recip, codes, scales, &s_d, 1);
  if (C > 1) cluster_sync_all();
}

// Pool norm whose output is quantised once (row scale per token) and written to the token's
// k expert rows.  Dynamic smem: L + 256 floats.
__global__ void __launch_bounds__(kRowThreads) poolnorm_scatter_nvfp4_kernel(
    const float* __restrict__ p, const float* __restrict__ ss_p, int ld_ss, const float* __restrict__ g,
    const int32_t* __restrict__ row_of, const int32_t* __restrict__ idx, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ tile_base, int L, int k, float eps, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, float* __restrict__ s_rows, int C) {
  griddep_enter();
  extern __shared__ float dyn[];
  const RowSlice sl = row_slice(L, C);
  float* buf = dyn;                  // this CTA's columns
  float* recip = dyn + (sl.i1 - sl.i0);
  __shared__ float red[33];
  __shared__ float s_rs, slot_amax;
  __shared__ QDest s_dst[16];
  load_recip(recip);
  const long long t = sl.t;
  if (threadIdx.x < 32) {
    const float ss = warp_sum_partials(ss_p + t * ld_ss, ld_ss, threadIdx.x);
    if (threadIdx.x == 0) s_rs = rsqrtf(ss / static_cast<float>(L) + eps);
  }
  if (threadIdx.x < k) {   // the expert row, and its M tile (the scale block) and place in it
    const int row = row_of[t * k + threadIdx.x];
    const int e = idx[t * k + threadIdx.x];
    const int pos = row - offsets[e];
    s_dst[threadIdx.x] = QDest{row, tile_base[e] + pos / kBM, pos % kBM};
  }
  __syncthreads();
  const float rs = s_rs;
  float amax = 0.f;
  for (int i = sl.i0 + threadIdx.x * 8; i < sl.i1; i += kRowThreads * 8) {
    float v[8], gg[8];
    load8_f32(p + t * L + i, v);
    load8_f32(g + i, gg);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = v[j] * rs * gg[j];
      amax = fmaxf(amax, fabsf(v[j]));
    }
    store8_f32(buf + (i - sl.i0), v);
  }
  const float s = nvfp4_row_scale(cluster_combine(block_max(amax, red), &slot_amax, C, true));
  if (sl.c == 0 && threadIdx.x < k) s_rows[s_dst[threadIdx.x].code_row] = s;
  quantize_row_to(buf, L, sl.i0, sl.i1, s, recip, codes, scales, s_dst, k);
  if (C > 1) cluster_sync_all();
}

// Combine whose output c is quantised (row scale per token) for the unpooler.
// Dynamic smem: L + 256 floats.
template <int NB, bool YF32>
__global__ void __launch_bounds__(kRowThreads) combine_nvfp4_kernel(
    const void* __restrict__ y, const float* __restrict__ ss_y, int ld_ss,
    const int32_t* __restrict__ row_of, const int32_t* __restrict__ idx, const float* __restrict__ w,
    const float* __restrict__ g_expert, int L, int k, float eps, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, float* __restrict__ s_row, int C) {
  griddep_enter();
  extern __shared__ float dyn[];
  const RowSlice sl = row_slice(L, C);
  float* buf = dyn;                  // this CTA's columns
  float* recip = dyn + (sl.i1 - sl.i0);
  __shared__ float red[33];
  __shared__ float s_coef[16], slot_amax;
  __shared__ int s_rowj[16], s_e[16];
  __shared__ QDest s_d;
  load_recip(recip);
  const long long t = sl.t;
  constexpr uint32_t kYBytes = YF32 ? 4u : 2u;
  for (int j = threadIdx.x >> 5; j < k; j += kRowThreads / 32) {   // a warp per slot
    const int lane = threadIdx.x & 31;
    const int row = row_of[t * k + j];
    if (lane == 0)   // the slot's row slice streams into L2 while the norms are computed
      prefetch_l2_bulk(static_cast<const char*>(y) + (static_cast<long long>(row) * L + sl.i0) * kYBytes,
                       static_cast<uint32_t>(sl.i1 - sl.i0) * kYBytes);
    const float ss = warp_sum_partials(ss_y + static_cast<long long>(row) * ld_ss, ld_ss, lane);
    if (lane == 0) {
      s_coef[j] = w[t * k + j] * rsqrtf(ss / static_cast<float>(L) + eps);
      s_rowj[j] = row;
      s_e[j] = idx[t * k + j];
    }
  }
  __syncthreads();
  float amax = 0.f;
  for (int i = sl.i0 + threadIdx.x * 8; i < sl.i1; i += kRowThreads * 8) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    combine_cols<8, NB, YF32>(y, g_expert, L, i, k, s_rowj, s_e, s_coef, acc);   // slot order
#pragma unroll
    for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(acc[q]));
    store8_f32(buf + (i - sl.i0), acc);
  }
  const float s = nvfp4_row_scale(cluster_combine(block_max(amax, red), &slot_amax, C, true));
  if (threadIdx.x == 0) {
    if (sl.c == 0) s_row[t] = s;
    s_d = QDest{t, t / kBM, static_cast<int>(t % kBM)};
  }
  __syncthreads();
  quantize_row_to(buf, L, sl.i0, sl.i1, s, recip, codes, scales, &s_d, 1);
  if (C > 1) cluster_sync_all();
}

// ------------------------------------------------------------------ NVFP4 rows from registers
// The rows are read and written as float4 chunks spread over the CTA (a warp's loads and
// stores are contiguous): thread x of TPB handles, for m < NCH, columns
// i0 + 4 TPB m + 4x .. +3, so the four lanes 4g .. 4g+3 hold one 16-column quantisation block.
// The row is normalised, reduced and quantised from registers (one pass over the inputs, no
// shared-memory staging).  Same rule and per-element arithmetic as the staged kernels above;
// the row reductions run in another order.

// This lane's 4 values of a block held by lanes 4g .. 4g+3 (block positions 4 (lane % 4) ..):
// the block's E4M3 scale code (in every lane of the group, as in nvfp4_quant16) and this
// lane's two code bytes (block bytes 2 (lane % 4), +1), low byte first.
__device__ __forceinline__ uint32_t quant4_group(const float (&v)[4], float six_s, float inv_s, uint32_t& sc) {
  float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  sc = cvt_e4m3(__fdiv_rn(a, six_s));
  const float r = g_e4m3_recip.v[sc];
  const uint32_t b0 = cvt_e2m1x2(__fmul_rn(__fmul_rn(v[1], r), inv_s), __fmul_rn(__fmul_rn(v[0], r), inv_s));
  const uint32_t b1 = cvt_e2m1x2(__fmul_rn(__fmul_rn(v[3], r), inv_s), __fmul_rn(__fmul_rn(v[2], r), inv_s));
  return b0 | (b1 << 8);
}

// Stores block b (this lane's group's) into destination row d: the lane's two code bytes, and
// the scales of the warp's 8 consecutive blocks (lane 0's block a multiple of 8) as two words,
// from lanes 0 and 16 (four adjacent bytes in both scale layouts).
__device__ __forceinline__ void store_group(uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                            const QDest& d, int K, int b, uint32_t bytes2, uint32_t sc, int lane) {
  *reinterpret_cast<uint16_t*>(codes + d.code_row * (K / 2) + b * 8 + 2 * (lane & 3)) = static_cast<uint16_t>(bytes2);
  uint32_t w = 0u;
#pragma unroll
  for (int q = 0; q < 4; ++q) w |= (__shfl_sync(0xffffffffu, sc, (lane & 16) + 4 * q) & 0xffu) << (8 * q);
  if ((lane & 15) == 0) {
    const size_t so = d.blk < 0 ? static_cast<size_t>(d.code_row) * (K / 16) + b : blocked_sf_offset(d.blk, d.m, b, K);
    *reinterpret_cast<uint32_t*>(scales + so) = w;
  }
}

// TPB and NCH for a row slice of n columns: 256 threads with n / 1024 chunks each (1, 2, 4 or
// 8), else one chunk per thread for n = 128, 256 or 512; false when neither fits.
bool qgroup_shape(int n, int& tpb, int& nch) {
  if (n % 1024 == 0 && n / 1024 <= 8 && ((n / 1024) & (n / 1024 - 1)) == 0) {
    tpb = 256;
    nch = n / 1024;
    return true;
  }
  if (n == 128 || n == 256 || n == 512) {
    tpb = n / 4;
    nch = 1;
    return true;
  }
  return false;
}

__device__ __forceinline__ void load4(const void* base, bool f32, long long i, float (&v)[4]) {
  if (f32) {
    const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  } else {
    const uint2 q = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + i);
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.x));
    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.y));
    v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
  }
}

template <int TPB, int NCH>
__global__ void __launch_bounds__(TPB) prenorm_nvfp4_q_kernel(
    const void* __restrict__ x, int x_f32, const float* __restrict__ g, int D, float eps,
    __nv_bfloat16* __restrict__ xa, int xa_cols, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, float* __restrict__ s_row, unsigned* status2, int C) {
  griddep_enter();
  if (status2 != nullptr && blockIdx.x == 0 && threadIdx.x == 0) status2[0] = status2[1] = 0u;
  __shared__ float red[33];
  __shared__ float slot_ss, slot_amax;
  const RowSlice sl = row_slice(D, C);
  const long long t = sl.t;
  const int lane = threadIdx.x & 31;
  float v[NCH][4];
  float ss = 0.f;
#pragma unroll
  for (int m = 0; m < NCH; ++m) load4(x, x_f32, t * D + sl.i0 + 4 * (TPB * m + threadIdx.x), v[m]);
#pragma unroll
  for (int m = 0; m < NCH; ++m)
#pragma unroll
    for (int q = 0; q < 4; ++q) ss = fmaf(v[m][q], v[m][q], ss);
  const float rs =
      rsqrtf(cluster_combine(block_sum(ss, red), &slot_ss, C, false) / static_cast<float>(D) + eps);
  __nv_bfloat16* row = xa + t * xa_cols;
  float amax = 0.f;
#pragma unroll
  for (int m = 0; m < NCH; ++m) {
    const int e = sl.i0 + 4 * (TPB * m + threadIdx.x);
    const float4 gg = *reinterpret_cast<const float4*>(g + e);
    const float gv[4] = {gg.x, gg.y, gg.z, gg.w};
    float hi[4], lo[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v[m][q] = v[m][q] * rs * gv[q];
      amax = fmaxf(amax, fabsf(v[m][q]));
      hi[q] = bf16_round(v[m][q]);
      lo[q] = v[m][q] - hi[q];
    }
    *reinterpret_cast<uint2*>(row + e) = make_uint2(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]));
    *reinterpret_cast<uint2*>(row + D + e) = make_uint2(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]));
  }
  const float s = nvfp4_row_scale(cluster_combine(block_max(amax, red), &slot_amax, C, true));
  if (sl.c == 0 && threadIdx.x == 0) s_row[t] = s;
  const float six_s = __fmul_rn(6.f, s), inv_s = __fdiv_rn(1.f, s);
  const QDest d{t, t / kBM, static_cast<int>(t % kBM)};
#pragma unroll
  for (int m = 0; m < NCH; ++m) {
    uint32_t sc;
    const uint32_t b2 = quant4_group(v[m], six_s, inv_s, sc);
    store_group(codes, scales, d, D, (sl.i0 + 4 * (TPB * m + threadIdx.x)) / 16, b2, sc, lane);
  }
  if (C > 1) cluster_sync_all();
}

// The pool norm writes each quantised row to k destinations, so its stores dominate: here a
// thread owns one whole 16-column block (TPB = columns / 16) and stores its 8 code bytes per
// destination at once; lanes 4i .. 4i+3 hold consecutive blocks, whose scales lane 4i stores as
// one word.
__device__ __forceinline__ void store_qblock(uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                             const QDest& d, int K, int b, uint2 q, uint32_t sc, int lane) {
  *reinterpret_cast<uint2*>(codes + d.code_row * (K / 2) + b * 8) = q;
  uint32_t w = sc & 0xffu;
  w |= (__shfl_down_sync(0xffffffffu, sc, 1) & 0xffu) << 8;
  w |= (__shfl_down_sync(0xffffffffu, sc, 2) & 0xffu) << 16;
  w |= (__shfl_down_sync(0xffffffffu, sc, 3) & 0xffu) << 24;
  if ((lane & 3) == 0) {
    const size_t so = d.blk < 0 ? static_cast<size_t>(d.code_row) * (K / 16) + b : blocked_sf_offset(d.blk, d.m, b, K);
    *reinterpret_cast<uint32_t*>(scales + so) = w;
  }
}

// TPB for a slice of n columns with one block per thread, or 0 when that does not fit.
int qblock_threads(int n) {
  if (n % 16) return 0;
  const int tpb = n / 16;
  return (tpb == 32 || tpb == 64 || tpb == 128 || tpb == 256 || tpb == 512) ? tpb : 0;
}

template <int TPB>
__global__ void __launch_bounds__(TPB) poolnorm_scatter_nvfp4_q_kernel(
    const float* __restrict__ p, const float* __restrict__ ss_p, int ld_ss, const float* __restrict__ g,
    const int32_t* __restrict__ row_of, const int32_t* __restrict__ idx, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ tile_base, int L, int k, float eps, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, float* __restrict__ s_rows, int C) {
  griddep_enter();
  __shared__ float red[33];
  __shared__ float s_rs, slot_amax;
  __shared__ QDest s_dst[16];
  const RowSlice sl = row_slice(L, C);
  const long long t = sl.t;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    const float ss = warp_sum_partials(ss_p + t * ld_ss, ld_ss, lane);
    if (lane == 0) s_rs = rsqrtf(ss / static_cast<float>(L) + eps);
  }
  constexpr int kDstWarp = TPB >= 64 ? 1 : 0;   // the destinations in a second warp when there is one
  if (threadIdx.x >= 32 * kDstWarp && threadIdx.x < 32 * kDstWarp + k) {
    const int j = threadIdx.x - 32 * kDstWarp;
    const int row = row_of[t * k + j];
    const int e = idx[t * k + j];
    const int pos = row - offsets[e];
    s_dst[j] = QDest{row, tile_base[e] + pos / kBM, pos % kBM};
  }
  const int i = sl.i0 + threadIdx.x * 16;
  float v[16], gg[16];
  {
    float a[8], b[8];
    load8_f32(p + t * L + i, a);
    load8_f32(p + t * L + i + 8, b);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = a[j];
      v[8 + j] = b[j];
    }
    load8_f32(g + i, a);
    load8_f32(g + i + 8, b);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      gg[j] = a[j];
      gg[8 + j] = b[j];
    }
  }
  __syncthreads();
  const float rs = s_rs;
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    v[j] = v[j] * rs * gg[j];
    amax = fmaxf(amax, fabsf(v[j]));
  }
  const float s = nvfp4_row_scale(cluster_combine(block_max(amax, red), &slot_amax, C, true));
  if (sl.c == 0 && threadIdx.x < k) s_rows[s_dst[threadIdx.x].code_row] = s;
  uint2 q;
  const uint32_t sc = nvfp4_quant16(v, __fmul_rn(6.f, s), __fdiv_rn(1.f, s), g_e4m3_recip.v, q);
  for (int j = 0; j < k; ++j) store_qblock(codes, scales, s_dst[j], L, i / 16, q, sc, lane);
  if (C > 1) cluster_sync_all();
}

template <int TPB, int NCH, int NB, bool YF32>
__global__ void __launch_bounds__(TPB) combine_nvfp4_q_kernel(
    const void* __restrict__ y, const float* __restrict__ ss_y, int ld_ss,
    const int32_t* __restrict__ row_of, const int32_t* __restrict__ idx, const float* __restrict__ w,
    const float* __restrict__ g_expert, int L, int k, float eps, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, float* __restrict__ s_row, int C) {
  griddep_enter();
  __shared__ float red[33];
  __shared__ float s_coef[16], slot_amax;
  __shared__ int s_rowj[16], s_e[16];
  const RowSlice sl = row_slice(L, C);
  const long long t = sl.t;
  const int lane = threadIdx.x & 31;
  constexpr uint32_t kYBytes = YF32 ? 4u : 2u;
  for (int j = threadIdx.x >> 5; j < k; j += TPB / 32) {   // a warp per slot
    const int row = row_of[t * k + j];
    // the slot's row slice starts streaming into L2 now; the weighted sum then reads it from
    // there (measured without: long-scoreboard stalls bound this kernel at 0.48 of HBM)
    if (lane == 0)
      prefetch_l2_bulk(static_cast<const char*>(y) + (static_cast<long long>(row) * L + sl.i0) * kYBytes,
                       static_cast<uint32_t>(sl.i1 - sl.i0) * kYBytes);
    const float ss = warp_sum_partials(ss_y + static_cast<long long>(row) * ld_ss, ld_ss, lane);
    if (lane == 0) {
      s_coef[j] = w[t * k + j] * rsqrtf(ss / static_cast<float>(L) + eps);
      s_rowj[j] = row;
      s_e[j] = idx[t * k + j];
    }
  }
  __syncthreads();
  float acc[NCH][4];
#pragma unroll
  for (int m = 0; m < NCH; ++m)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[m][q] = 0.f;
  for (int j0 = 0; j0 < k; j0 += NB) {   // slot order; the loads of NB slots issued together
    float yv[NB][NCH][4], gv[NB][NCH][4];
#pragma unroll
    for (int jj = 0; jj < NB; ++jj)
      if (j0 + jj < k) {
#pragma unroll
        for (int m = 0; m < NCH; ++m) {
          const int e = sl.i0 + 4 * (TPB * m + threadIdx.x);
          load4(y, YF32, static_cast<long long>(s_rowj[j0 + jj]) * L + e, yv[jj][m]);
          load4(g_expert, true, static_cast<long long>(s_e[j0 + jj]) * L + e, gv[jj][m]);
        }
      }
#pragma unroll
    for (int jj = 0; jj < NB; ++jj)
      if (j0 + jj < k) {
#pragma unroll
        for (int m = 0; m < NCH; ++m)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[m][q] = fmaf(s_coef[j0 + jj], yv[jj][m][q] * gv[jj][m][q], acc[m][q]);
      }
  }
  float amax = 0.f;
#pragma unroll
  for (int m = 0; m < NCH; ++m)
#pragma unroll
    for (int q = 0; q < 4; ++q) amax = fmaxf(amax, fabsf(acc[m][q]));
  const float s = nvfp4_row_scale(cluster_combine(block_max(amax, red), &slot_amax, C, true));
  if (sl.c == 0 && threadIdx.x == 0) s_row[t] = s;
  const float six_s = __fmul_rn(6.f, s), inv_s = __fdiv_rn(1.f, s);
  const QDest d{t, t / kBM, static_cast<int>(t % kBM)};
#pragma unroll
  for (int m = 0; m < NCH; ++m) {
    uint32_t sc;
    const uint32_t b2 = quant4_group(acc[m], six_s, inv_s, sc);
    store_group(codes, scales, d, L, (sl.i0 + 4 * (TPB * m + threadIdx.x)) / 16, b2, sc, lane);
  }
  if (C > 1) cluster_sync_all();
}

// Stand-alone quantiser: one CTA per row of src [rows, K] fp32.
__global__ void __launch_bounds__(kRowThreads) quantize_nvfp4_kernel(
    const float* __restrict__ src, int K, int row_scale, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, float* __restrict__ s_row) {
  griddep_enter();
  extern __shared__ float dyn[];
  float* buf = dyn;
  float* recip = dyn + K;
  __shared__ float red[33];
  __shared__ QDest s_d;
  load_recip(recip);
  const long long t = blockIdx.x;
  float amax = 0.f;
  for (int i = threadIdx.x; i < K; i += kRowThreads) {
    const float v = src[t * K + i];
    buf[i] = v;
    amax = fmaxf(amax, fabsf(v));
  }
  amax = block_max(amax, red);
  const float s = row_scale ? nvfp4_row_scale(amax) : 1.f;
  if (threadIdx.x == 0) {
    if (s_row) s_row[t] = s;
    s_d = QDest{t, -1, 0};   // row-major scales
  }
  __syncthreads();
  quantize_row_to(buf, K, 0, K, s, recip, codes, scales, &s_d, 1);
}

// Row-major E4M3 scales [rows, K/16] -> block layout with blocks of block_rows rows (128, or
// 64: then a line's last two words stay unused): one thread moves the 4 scale bytes of one
// (row, 64-wide K step) as one word.
__global__ void nvfp4_block_scales_kernel(const uint8_t* __restrict__ src, long long rows, int K,
                                          int block_rows, uint8_t* __restrict__ dst) {
  griddep_enter();
  const long long words = rows * (K / 64);
  for (long long w = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; w < words;
       w += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = w / (K / 64);
    const int k64 = static_cast<int>(w % (K / 64));
    const uint8_t* p = src + r * (K / 16) + k64 * 4;
    const uint32_t v = static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8) |
                       (static_cast<uint32_t>(p[2]) << 16) | (static_cast<uint32_t>(p[3]) << 24);
    *reinterpret_cast<uint32_t*>(dst + blocked_sf_offset(r / block_rows, static_cast<int>(r % block_rows), k64 * 4, K)) = v;
  }
}

// ------------------------------------------------------------------ split-K reduction
// One CTA of `group` threads per (row, column group): sums the partials in split order (the
// result does not depend on scheduling) and writes the group's sum of squares.
__global__ void splitk_reduce_kernel(const float* __restrict__ partial, int splits, int rows, int N,
                                     void* __restrict__ out, long long ldo, float* __restrict__ ss,
                                     int ld_ss, const int* __restrict__ splits_dev, int out_bf16) {
  griddep_enter();
  if (splits_dev != nullptr) {
    splits = *splits_dev;
    if (splits <= 1) return;   // the GEMM wrote out and ss itself
  }
  __shared__ float red[33];
  const int r = blockIdx.x, grp = blockIdx.y;
  const int col = grp * blockDim.x + threadIdx.x;
  float v = 0.f;
  if (col < N) {
    for (int q = 0; q < splits; ++q) v += partial[(static_cast<long long>(q) * rows + r) * N + col];
    if (out_bf16) {   // stored rounded; the sum of squares is that of the stored value
      const __nv_bfloat16 b = __float2bfloat16_rn(v);
      static_cast<__nv_bfloat16*>(out)[static_cast<long long>(r) * ldo + col] = b;
      v = __bfloat162float(b);
    } else {
      static_cast<float*>(out)[static_cast<long long>(r) * ldo + col] = v;
    }
  }
  if (ss != nullptr) {
    const float t = block_sum(col < N ? v * v : 0.f, red);
    if (threadIdx.x == 0) ss[static_cast<long long>(r) * ld_ss + grp] = t;
  }
}

// One CTA per (M tile, 4096 columns); a thread owns one 16-column block of h and walks the
// tile's rows: sums the gate and up partials in split order, applies SwiGLU and quantises the
// block (scale 1) exactly as the unsplit GEMM epilogue does.
__global__ void __launch_bounds__(256) swiglu_reduce_nvfp4_kernel(
    const float* __restrict__ partial, const int* __restrict__ splits_dev, int rows, int N,
    const Tile* __restrict__ tiles, const int* __restrict__ n_tiles, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales) {
  griddep_enter();
  __shared__ float recip[256];
  const int splits = *splits_dev;
  const int mt = blockIdx.x;
  if (splits <= 1 || mt >= *n_tiles) return;
  for (int i = threadIdx.x; i < 256; i += blockDim.x) recip[i] = g_e4m3_recip.v[i];
  __syncthreads();
  const Tile t = tiles[mt];
  const int cb = blockIdx.y * blockDim.x + threadIdx.x;   // 16-column block of h
  if (cb * 16 >= N) return;
  const long long plane = static_cast<long long>(rows) * 2 * N;   // one split's partials
  for (int r = 0; r < t.nrows; ++r) {
    const long long grow = static_cast<long long>(t.row0) + r;
    const float* pg = partial + grow * 2 * N + cb * 16;
    float g[16], u[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) g[i] = u[i] = 0.f;
    for (int q = 0; q < splits; ++q) {
      const float4* g4 = reinterpret_cast<const float4*>(pg + q * plane);
      const float4* u4 = reinterpret_cast<const float4*>(pg + q * plane + N);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 a = g4[i], b = u4[i];
        g[4 * i] += a.x; g[4 * i + 1] += a.y; g[4 * i + 2] += a.z; g[4 * i + 3] += a.w;
        u[4 * i] += b.x; u[4 * i + 1] += b.y; u[4 * i + 2] += b.z; u[4 * i + 3] += b.w;
      }
    }
    float h[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) h[i] = __fdividef(g[i], 1.f + __expf(-g[i])) * u[i];
    uint2 q;
    const uint32_t sc = nvfp4_quant16(h, 6.f, 1.f, recip, q);
    *reinterpret_cast<uint2*>(codes + grow * (N / 2) + cb * 8) = q;
    scales[blocked_sf_offset(mt, r, cb, N)] = static_cast<uint8_t>(sc);
  }
}

// ------------------------------------------------------------------ routing validation
// One CTA.  Every read of a value under test is bounds-checked first, so corrupted structures
// are reported, never followed.
constexpr int kValidateThreads = 1024;

__device__ __forceinline__ bool tile_ok(const Tile& t, int E, const int32_t* offsets, int max_rows) {
  if (t.expert < 0 || t.expert >= E || t.nrows < 1 || t.nrows > max_rows) return false;
  return t.row0 >= offsets[t.expert] && t.row0 + t.nrows <= offsets[t.expert + 1];
}

__global__ void __launch_bounds__(kValidateThreads) validate_routing_kernel(
    int32_t* __restrict__ idx, int T, int k, int E, const int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ row_of, const int32_t* __restrict__ tok_of,
    const Tile* __restrict__ tiles, int32_t* __restrict__ n_tiles, int max_tiles,
    int32_t* __restrict__ tile_base, const Tile* __restrict__ tiles2, int32_t* __restrict__ n_tiles2,
    int max_tiles2, unsigned* __restrict__ err, int sanitize) {
  griddep_enter();
  __shared__ int bad, offsets_ok;
  __shared__ int red[33];
  const long long R = static_cast<long long>(T) * k;
  if (threadIdx.x == 0) {
    bad = 0;
    offsets_ok = offsets[0] == 0 && offsets[E] == R;
  }
  __syncthreads();
  // offsets and counts
  for (int e = threadIdx.x; e < E; e += kValidateThreads)
    if (offsets[e + 1] < offsets[e] || counts[e] != offsets[e + 1] - offsets[e]) offsets_ok = 0;
  __syncthreads();
  if (!offsets_ok) {
    bad = 1;
  } else {
    // every pair: its expert, its row inside the expert's range, the row's token
    for (long long i = threadIdx.x; i < R; i += kValidateThreads) {
      const int e = idx[i], r = row_of[i];
      if (e < 0 || e >= E || r < offsets[e] || r >= offsets[e + 1] || tok_of[r] != static_cast<int>(i / k))
        bad = 1;
    }
    // every row is the row of one of its token's pairs (with the above: a bijection)
    for (long long r = threadIdx.x; r < R; r += kValidateThreads) {
      const int t = tok_of[r];
      bool found = false;
      if (t >= 0 && t < T)
        for (int j = 0; j < k; ++j) found = found || row_of[static_cast<long long>(t) * k + j] == r;
      if (!found) bad = 1;
    }
    // the tile tables
    const int nt = *n_tiles;
    if (nt < 0 || nt > max_tiles) bad = 1;
    int rows = 0;
    for (int m = threadIdx.x; m < min(max(nt, 0), max_tiles); m += kValidateThreads) {
      const Tile t = tiles[m];
      if (!tile_ok(t, E, offsets, kBM)) bad = 1;
      else rows += t.nrows;
    }
    if (block_sum_int(rows, red) != R) bad = 1;
    if (tiles2 != nullptr) {
      const int nt2 = *n_tiles2;
      if (nt2 < 0 || nt2 > max_tiles2) bad = 1;
      int rows2 = 0;
      for (int m = threadIdx.x; m < min(max(nt2, 0), max_tiles2); m += kValidateThreads) {
        const Tile t = tiles2[m];
        if (!tile_ok(t, E, offsets, 2 * kBM)) bad = 1;
        else rows2 += t.nrows;
      }
      if (block_sum_int(rows2, red) != R) bad = 1;
    }
    if (tile_base != nullptr)
      for (int e = threadIdx.x; e < E; e += kValidateThreads)
        if (counts[e] > 0) {
          const int b = tile_base[e];
          if (b < 0 || b >= min(max(nt, 0), max_tiles) || tiles[b].expert != e || tiles[b].row0 != offsets[e])
            bad = 1;
        }
  }
  __syncthreads();
  if (!bad) return;
  if (threadIdx.x == 0) atomicOr(err, kErrBounds);
  if (!sanitize) return;
  // a routing every later kernel of the call reads in bounds: no tiles (the grouped GEMMs do
  // nothing), every pair to expert 0 and row 0, every expert starting at row 0 and tile 0
  for (long long i = threadIdx.x; i < R; i += kValidateThreads) {
    idx[i] = 0;
    row_of[i] = 0;
  }
  for (int e = threadIdx.x; e <= E; e += kValidateThreads) {
    offsets[e] = 0;
    if (tile_base != nullptr && e < E) tile_base[e] = 0;
  }
  if (threadIdx.x == 0) {
    *n_tiles = 0;
    if (n_tiles2 != nullptr) *n_tiles2 = 0;
  }
}

// ------------------------------------------------------------------ wait self-test
// One thread waits on a barrier that is initialised for one arrival that never comes.
__global__ void wait_selftest_kernel(long long budget, unsigned* err) {
  griddep_enter();
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, budget)) atomicOr(err, kErrWaitEpilogue);
  }
}

}  // namespace

// ------------------------------------------------------------------ launchers
// CTAs per token of the row kernels: a few tokens are spread over about 128 CTAs or more
// (at most 8 per token, each taking a multiple of 128 columns).
int row_split(int T, int N) {
  int C = 1;
  while (C < 8 && static_cast<long long>(T) * C < 128 && N % (2 * C * 128) == 0) C *= 2;
  return C;
}

cudaError_t launch_prenorm_nvfp4(const void* x, bool x_f32, const float* g_pre, int T, int D,
                                 float eps, __nv_bfloat16* xa, int xa_cols, uint8_t* codes,
                                 uint8_t* scales, float* s_row, unsigned* status2, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int C = row_split(T, D);
  int tpb = 0, nch = 0;
  if (qgroup_shape(D / C, tpb, nch)) {   // rows from registers, coalesced chunks
#define LMOE_Q(TPB, NCH)                                                                                \
  if (tpb == TPB && nch == NCH)                                                                         \
    return launch_pdl_cluster(prenorm_nvfp4_q_kernel<TPB, NCH>, dim3(T * C), dim3(TPB), 0, s, C, x,     \
                              x_f32 ? 1 : 0, g_pre, D, eps, xa, xa_cols, codes, scales, s_row, status2, C);
    LMOE_Q(256, 1) LMOE_Q(256, 2) LMOE_Q(256, 4) LMOE_Q(256, 8) LMOE_Q(128, 1) LMOE_Q(64, 1) LMOE_Q(32, 1)
#undef LMOE_Q
  }
  const size_t smem = (static_cast<size_t>(D / C) + 256) * sizeof(float);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(prenorm_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl_cluster(prenorm_nvfp4_kernel, dim3(T * C), dim3(kRowThreads), smem, s, C, x,
                            x_f32 ? 1 : 0, g_pre, D, eps, xa, xa_cols, codes, scales, s_row, status2, C);
}

cudaError_t launch_poolnorm_scatter_nvfp4(const float* p, const float* ss_p, int ld_ss,
                                          const float* g_pool, const int32_t* row_of,
                                          const int32_t* idx, const int32_t* offsets,
                                          const int32_t* tile_base, int T, int L, int k, float eps,
                                          uint8_t* codes, uint8_t* scales, float* s_rows,
                                          cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int C = row_split(T, L);
  switch (qblock_threads(L / C)) {   // one quantisation block per thread, from registers
#define LMOE_Q(TPB)                                                                                     \
  case TPB:                                                                                             \
    return launch_pdl_cluster(poolnorm_scatter_nvfp4_q_kernel<TPB>, dim3(T * C), dim3(TPB), 0, s, C, p, \
                              ss_p, ld_ss, g_pool, row_of, idx, offsets, tile_base, L, k, eps, codes,   \
                              scales, s_rows, C);
    LMOE_Q(32) LMOE_Q(64) LMOE_Q(128) LMOE_Q(256) LMOE_Q(512)
#undef LMOE_Q
    default: break;
  }
  const size_t smem = (static_cast<size_t>(L / C) + 256) * sizeof(float);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(poolnorm_scatter_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl_cluster(poolnorm_scatter_nvfp4_kernel, dim3(T * C), dim3(kRowThreads), smem, s, C,
                            p, ss_p, ld_ss, g_pool, row_of, idx, offsets, tile_base, L, k, eps, codes,
                            scales, s_rows, C);
}

cudaError_t launch_combine_nvfp4(const void* y, bool y_bf16, const float* ss_y, int ld_ss,
                                 const int32_t* row_of, const int32_t* idx, const float* w,
                                 const float* g_expert, int T, int L, int k, float eps, uint8_t* codes,
                                 uint8_t* scales, float* s_row, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int C = row_split(T, L);
  const bool few = T <= kCombineBatchMaxT;
  int tpb = 0, nch = 0;
  if (qgroup_shape(L / C, tpb, nch)) {   // rows from registers, coalesced chunks
#define LMOE_Q(TPB, NCH)                                                                                \
  if (tpb == TPB && nch == NCH) {                                                                       \
    auto kern = few ? (y_bf16 ? combine_nvfp4_q_kernel<TPB, NCH, 2, false> : combine_nvfp4_q_kernel<TPB, NCH, 2, true>) \
                    : (y_bf16 ? combine_nvfp4_q_kernel<TPB, NCH, 1, false> : combine_nvfp4_q_kernel<TPB, NCH, 1, true>); \
    return launch_pdl_cluster(kern, dim3(T * C), dim3(TPB), 0, s, C, y, ss_y, ld_ss, row_of, idx, w,    \
                              g_expert, L, k, eps, codes, scales, s_row, C);                             \
  }
    LMOE_Q(256, 1) LMOE_Q(256, 2) LMOE_Q(256, 4) LMOE_Q(256, 8) LMOE_Q(128, 1) LMOE_Q(64, 1) LMOE_Q(32, 1)
#undef LMOE_Q
  }
  const size_t smem = (static_cast<size_t>(L / C) + 256) * sizeof(float);
  static bool attr = false;
  if (!attr) {
    for (auto kern : {combine_nvfp4_kernel<1, true>, combine_nvfp4_kernel<kCombineBatch, true>,
                      combine_nvfp4_kernel<1, false>, combine_nvfp4_kernel<kCombineBatch, false>}) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
      if (e != cudaSuccess) return e;
    }
    attr = true;
  }
  auto kern = few ? (y_bf16 ? combine_nvfp4_kernel<kCombineBatch, false> : combine_nvfp4_kernel<kCombineBatch, true>)
                  : (y_bf16 ? combine_nvfp4_kernel<1, false> : combine_nvfp4_kernel<1, true>);
  return launch_pdl_cluster(kern, dim3(T * C), dim3(kRowThreads), smem, s, C, y, ss_y, ld_ss, row_of, idx, w,
                            g_expert, L, k, eps, codes, scales, s_row, C);
}

cudaError_t launch_quantize_nvfp4(const float* src, long long rows, int K, bool row_scale,
                                  uint8_t* codes, uint8_t* scales, float* s_row, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const size_t smem = (static_cast<size_t>(K) + 256) * sizeof(float);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(quantize_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(quantize_nvfp4_kernel, dim3(static_cast<unsigned>(rows)), dim3(kRowThreads),
                    smem, s, src, K, row_scale ? 1 : 0, codes, scales, s_row);
}

cudaError_t launch_nvfp4_block_scales(const uint8_t* src, long long rows, int K, int block_rows,
                                      uint8_t* dst, cudaStream_t s) {
  const long long words = rows * (K / 64);
  if (words == 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<long long>((words + 255) / 256, 152 * 32));
  return launch_pdl(nvfp4_block_scales_kernel, dim3(blocks), dim3(256), 0, s, src, rows, K,
                    block_rows, dst);
}

cudaError_t launch_splitk_reduce(const float* partial, int splits, int rows, int N, void* out,
                                 long long ldo, float* ss, int ld_ss, int group, cudaStream_t s,
                                 const int* splits_dev, bool out_bf16) {
  if (rows == 0) return cudaSuccess;
  dim3 grid(rows, (N + group - 1) / group);
  return launch_pdl(splitk_reduce_kernel, dim3(grid), dim3(group), 0, s, partial, splits, rows, N,
                    out, ldo, ss, ld_ss, splits_dev, out_bf16 ? 1 : 0);
}

cudaError_t launch_swiglu_reduce_nvfp4(const float* partial, const int* splits_dev, int rows, int N,
                                       const Tile* tiles, const int* n_tiles, int max_tiles,
                                       uint8_t* codes, uint8_t* scales, cudaStream_t s) {
  if (rows == 0 || max_tiles == 0) return cudaSuccess;
  dim3 grid(max_tiles, (N / 16 + 255) / 256);
  return launch_pdl(swiglu_reduce_nvfp4_kernel, grid, dim3(256), 0, s, partial, splits_dev, rows, N,
                    tiles, n_tiles, codes, scales);
}

cudaError_t launch_validate_routing(int32_t* idx, int T, int k, int E, const int32_t* counts, int32_t* offsets,
                                    int32_t* row_of, const int32_t* tok_of, const Tile* tiles, int32_t* n_tiles,
                                    int max_tiles, int32_t* tile_base, const Tile* tiles2, int32_t* n_tiles2,
                                    int max_tiles2, unsigned* err, bool sanitize, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(validate_routing_kernel, dim3(1), dim3(kValidateThreads), 0, s, idx, T, k, E, counts,
                    offsets, row_of, tok_of, tiles, n_tiles, max_tiles, tile_base, tiles2, n_tiles2,
                    max_tiles2, err, sanitize ? 1 : 0);
}

cudaError_t launch_wait_selftest(long long budget, unsigned* err, cudaStream_t s) {
  return launch_pdl(wait_selftest_kernel, dim3(1), dim3(32), 0, s, budget, err);
}

cudaError_t launch_prenorm(const void* x, bool x_f32, const float* g_pre, int T, int D, float eps,
                           __nv_bfloat16* xa, int xa_cols, unsigned* status2, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int C = row_split(T, D);
  return launch_pdl_cluster(prenorm_kernel, dim3(T * C), dim3(kRowThreads), 0, s, C, x, x_f32 ? 1 : 0,
                            g_pre, D, eps, xa, xa_cols, status2, C);
}

cudaError_t launch_topk(const float* logits, int ld, const float* bias, const int32_t* forced,
                        int T, int E, int k, int32_t* idx, float* w, int32_t* near_tie,
                        int32_t* idx_copy, float* w_copy, unsigned* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kTopkWarps - 1) / kTopkWarps;
  const size_t smem = static_cast<size_t>(kTopkWarps) * E * sizeof(float);
  return launch_pdl(topk_kernel, dim3(blocks), dim3(kTopkWarps * 32), smem, s, logits, ld, bias,
                    forced, T, E, k, idx, w, near_tie, idx_copy, w_copy, err);
}

bool route_small_fits(int T, int k, int E) {
  return T * k <= kRouteMaxPairs && E <= 1024;
}

cudaError_t launch_route_small(float* logits, int ld, const float* rpart, int rsplits, const float* bias,
                               const int32_t* forced,
                               int T, int E, int k, int32_t* idx, float* w, int32_t* near_tie,
                               int32_t* idx_copy, float* w_copy, unsigned* err, int32_t* counts,
                               int32_t* offsets, int32_t* row_of, int32_t* tok_of, Tile* tiles,
                               int32_t* n_tiles, int32_t* tile_base, Tile* tiles2, int32_t* n_tiles2,
                               cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const size_t smem = (static_cast<size_t>(kRouteThreads / 32) * E + 2 * E + kRouteMaxPairs) * 4;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>((kRouteThreads / 32 * 1024 + 2 * 1024 + kRouteMaxPairs) * 4));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(route_small_kernel, dim3(1), dim3(kRouteThreads), smem, s, logits, ld, rpart, rsplits,
                    bias, forced, T, E,
                    k, idx, w, near_tie, idx_copy, w_copy, err, counts, offsets, row_of, tok_of, tiles,
                    n_tiles, tile_base, tiles2, n_tiles2);
}

int perm_chunks(long long pairs) { return static_cast<int>((pairs + kPermChunk - 1) / kPermChunk); }

cudaError_t launch_permute(const int32_t* idx, int T, int k, int E, int32_t* counts,
                           int32_t* offsets, int32_t* row_of, int32_t* tok_of, Tile* tiles,
                           int32_t* n_tiles, cudaStream_t s, int32_t* tile_base, Tile* tiles2,
                           int32_t* n_tiles2, int32_t* chunk_hist, int32_t* chunk_base) {
  const int n = T * k;
  if (chunk_hist != nullptr && chunk_base != nullptr && n >= kPermChunkedMinPairs) {
    const int chunks = perm_chunks(n);
    const size_t smem_h = static_cast<size_t>(E) * 4, smem_r = static_cast<size_t>(kPermThreads / 32) * E * 4;
    cudaError_t e = launch_pdl(perm_hist_kernel, dim3(chunks), dim3(kPermThreads), smem_h, s, idx, n, E,
                               chunk_hist);
    if (e != cudaSuccess) return e;
    e = launch_pdl(perm_scan_kernel, dim3(1), dim3(kPermScanThreads), 0, s, chunk_hist, chunks, E,
                   chunk_base, counts, offsets, tiles, n_tiles, tile_base, tiles2, n_tiles2);
    if (e != cudaSuccess) return e;
    return launch_pdl(perm_rank_kernel, dim3(chunks), dim3(kPermThreads), smem_r, s, idx, n, k, E,
                      chunk_base, offsets, row_of, tok_of);
  }
  cudaError_t e = launch_pdl(expert_count_kernel, dim3(E), dim3(kPermThreads), 0, s, idx, n,
                             counts);
  if (e != cudaSuccess) return e;
  return launch_pdl(expert_scatter_kernel, dim3(E), dim3(kPermThreads), 0, s, idx, n, k, E, counts,
                    offsets, row_of, tok_of, tiles, n_tiles, tile_base, tiles2, n_tiles2);
}

cudaError_t launch_poolnorm_scatter(const float* p, const float* ss_p, int ld_ss,
                                    const float* g_pool, const int32_t* row_of, int T, int L,
                                    int k, float eps, __nv_bfloat16* xe, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int C = row_split(T, L);
  return launch_pdl(poolnorm_scatter_kernel, dim3(T * C), dim3(kRowThreads), 0, s, p, ss_p, ld_ss,
                    g_pool, row_of, L, k, eps, xe, C);
}

cudaError_t launch_combine(const float* y, const float* ss_y, int ld_ss,
                           const int32_t* row_of, const int32_t* idx, const float* w,
                           const float* g_expert, int T, int L, int k, float eps,
                           __nv_bfloat16* c, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int C = row_split(T, L);
  return launch_pdl(T <= kCombineBatchMaxT ? combine_kernel<kCombineBatch> : combine_kernel<1>, dim3(T * C),
                    dim3(kRowThreads), 0, s, y, ss_y, ld_ss, row_of, idx, w, g_expert, L, k, eps, c, C);
}

cudaError_t launch_postnorm_residual(const void* x, bool x_f32, float* u,
                                     const float* ss_u, int ld_ss, const float* g_post, int T,
                                     int D, float eps, void* out, bool out_f32, cudaStream_t s,
                                     const float* upart, int usplits, const float* g_next,
                                     void* next_out) {
  if (T == 0) return cudaSuccess;
  const int C = row_split(T, D);
  if (usplits > 1 || g_next != nullptr)   // row sums of squares combined over a cluster of C CTAs
    return launch_pdl_cluster(postnorm_residual_kernel, dim3(T * C), dim3(kRowThreads), 0, s, C, x,
                              x_f32 ? 1 : 0, u, ss_u, ld_ss, g_post, D, eps, out, out_f32 ? 1 : 0, C, upart,
                              usplits, T, g_next, next_out);
  return launch_pdl(postnorm_residual_kernel, dim3(T * C), dim3(kRowThreads), 0, s, x, x_f32 ? 1 : 0,
                    u, ss_u, ld_ss, g_post, D, eps, out, out_f32 ? 1 : 0, C, upart, usplits, T, g_next,
                    next_out);
}

cudaError_t launch_weight_split(const float* W, long long rows, int K, int parts,
                                unsigned lo_mask, __nv_bfloat16* dst, cudaStream_t s) {
  const long long chunks = rows * (K / 8);
  if (chunks == 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<long long>((chunks + 255) / 256, 152 * 16));
  return launch_pdl(weight_split_kernel, dim3(blocks), dim3(256), 0, s, W, rows, K, parts, lo_mask,
                    dst);
}

}  // namespace lmoe
