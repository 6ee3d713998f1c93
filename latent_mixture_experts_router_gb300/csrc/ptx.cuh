// ptx.cuh — thin inline-PTX wrappers for the Blackwell (sm_103a) features the
// kernels use: mbarriers, TMA tensor copies, and the 5th-generation tensor
// core (tcgen05.mma with accumulators in tensor memory).  Every wait here is
// bounded by a clock64 budget: a wait that runs out returns false and the
// caller records an error word and leaves its loop, so no kernel can spin
// forever.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define LMOE_DEV __device__ __forceinline__

namespace lmoe {

LMOE_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
LMOE_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
LMOE_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
LMOE_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
LMOE_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
LMOE_DEV bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same with a suspend-time hint: a waiting thread may sleep up to `ns` nanoseconds and
// resumes as soon as the phase completes, so waiting warps issue few instructions.
LMOE_DEV bool mbar_try_wait_sleep(uint32_t addr, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
constexpr uint32_t kWaitSleepNs = 20000;
// Waits for the phase of parity `parity` to complete; false once `budget` cycles pass.
LMOE_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, long long budget) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(a, parity, kWaitSleepNs)) {
    if (clock64() - t0 > budget) return false;
  }
  return true;
}

// ------------------------------------------------------------------ TMA
LMOE_DEV void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// 2-D tiled copy global -> shared; completion is signalled on `bar` as transaction bytes.
// c0 is the innermost (contiguous) coordinate in elements, c1 the row.
LMOE_DEV void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
// Same, with an L2 cache-policy hint (createpolicy value).
LMOE_DEV void tma_load_2d_hint(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1,
                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}
// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
LMOE_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
LMOE_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
LMOE_DEV uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
LMOE_DEV uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------ tcgen05
// Tensor-memory allocation: executed by one whole warp; the base address lands in smem.
LMOE_DEV void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
LMOE_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
LMOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
LMOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
LMOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with
// 128-byte swizzle: rows of 64 bf16 (128 B), 8-row groups 1024 B apart.
// Fields: start address >> 4 [0,14), leading byte offset >> 4 [16,30) (unused for
// swizzled K-major), stride byte offset >> 4 [32,46), version 1 [46,48),
// base offset 0 [49,52), layout type [61,64) = 2 (128-byte swizzle).
LMOE_DEV uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A/B, fp32 accumulator,
// both operands K-major: D format [4,6)=1 (f32), A format [7,10)=1 (bf16),
// B format [10,13)=1 (bf16), N>>3 at [17,23), M>>4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, one 128xNx16 step, issued by a single thread.
LMOE_DEV void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when every tcgen05 operation issued so far by this thread completes.
LMOE_DEV void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Warp-collective load of 32 consecutive fp32 columns of the warp's 32 TMEM lanes:
// lane i of the warp receives row (lane base + i), columns col..col+31.
LMOE_DEV void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
LMOE_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ epilogue stores
// One thread's 32 consecutive fp32 values (a row segment, 16-byte aligned), as 8 vector stores.
LMOE_DEV void store_row32_f32(float* g, const uint32_t (&v)[32]) {
  float4* o = reinterpret_cast<float4*>(g);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    o[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                       __uint_as_float(v[4 * i + 3]));
}
// A warp's 32 x 32 fp32 block, read from tensor memory with one row per thread (thread i
// holds row i's 32 columns in v).  Stored straight from those registers, every store
// instruction would touch 32 rows, 16 bytes each; instead the block passes through this warp's
// padded shared tile (32 x 33 floats: the odd pitch keeps the row writes and the column reads
// free of bank conflicts) and each store instruction writes four whole 128-byte row segments.
// Rows [0, nvalid) are stored at g + row * ld (g and ld * 4 bytes 16-byte aligned).
LMOE_DEV void warp_store_32x32_f32(float* xp, const uint32_t (&v)[32], float* g, long long ld,
                                   int nvalid, int lane) {
#pragma unroll
  for (int c = 0; c < 32; ++c) xp[lane * 33 + c] = __uint_as_float(v[c]);
  __syncwarp();
  const int sub = lane >> 3, c4 = (lane & 7) * 4;
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    const int r = 4 * st + sub;
    if (r < nvalid) {
      const float* q = xp + r * 33 + c4;
      *reinterpret_cast<float4*>(g + r * ld + c4) = make_float4(q[0], q[1], q[2], q[3]);
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ programmatic dependent launch
// Every kernel of the library is launched with programmatic stream serialisation: its CTAs
// may become resident while the previous kernel of the stream is still finishing, and they
// block in griddep_wait() until that kernel has completed and its writes are visible.  Each
// kernel calls griddep_wait() before touching anything an earlier kernel wrote, then lets
// its own dependents launch (they wait likewise, so the trigger point only affects overlap).
LMOE_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
LMOE_DEV void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
LMOE_DEV void griddep_enter() {
  griddep_wait();
  griddep_launch_dependents();
}

// L2 prefetch of one tensor-map box (no shared memory, no barrier) and of a contiguous range
// (16-byte aligned address and size).  Used for operands no earlier kernel writes (weights),
// ahead of griddep_wait().
LMOE_DEV void prefetch_l2_tile_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
               :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y) : "memory");
}
LMOE_DEV void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
               :: "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ tile order
// Grouped rasterisation of a 1-D grid over (M tile, N tile): groups of `group` consecutive M
// tiles; inside a group the M index runs fastest, so the CTAs resident at one time share
// each B (weight) tile while the group's A tiles stay in L2.  Returns false for ids past the
// live tile count (it is read on the device for grouped GEMMs).
LMOE_DEV bool grouped_tile(int id, int total_m, int nt, int group, int& m, int& n) {
  const int gsz = group * nt;
  const int g = id / gsz;
  const int first = g * group;
  const int gm = min(group, total_m - first);
  if (gm <= 0) return false;
  const int local = id - g * gsz;
  if (local >= gm * nt) return false;
  m = first + local % gm;
  n = local / gm;
  return true;
}
constexpr int kRasterGroup = 16;

// ------------------------------------------------------------------ misc
LMOE_DEV float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

LMOE_DEV uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x = a (low half), .y = b
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace lmoe
