// noalloc.cu — the token permutation with its scratch in a fixed device array, for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code whose device memory is planned up front by a
// host framework or runtime and that has no way to ask it for one more buffer, plug-ins
// loaded into a process that forbids allocation after start-up, and latency-critical loops
// where the implicit synchronisation of an allocation is not acceptable.  For them,
// lmoe_permute_noalloc runs the same histogram + stable-scatter kernels as the block's
// permutation step, with their scratch (per-expert counts, the M-tile table and its length)
// placed in g_noalloc_scratch below instead of in a caller-provided workspace.
//
// The array is a file-scope __device__ object: every GPU that loads this library holds its
// 64 KiB until the process exits.  Host code cannot use the symbol as a device address, so
// the first call on each device looks the address up with cudaGetSymbolAddress (that
// device current) and caches it; later calls reuse it.  A cudaDeviceReset unloads the module
// and leaves the cached address stale: calls after a reset of the device are not supported.
//
// This is the per-expert-scan form of the permutation (one CTA per expert, each reading every
// id twice), so its cost grows as E x T*k; the block's own forward switches to a chunked
// histogram/scan/rank form from 16384 pairs, whose per-chunk tables need workspace.
#include <mutex>

#include "../../include/latent_moe.h"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 64 * 1024;
constexpr int kNoAllocMaxExperts = 1024;
constexpr long long kNoAllocMaxPairs = 65536;  // T * k
constexpr size_t kCountsOffset = 0;            // int32 [E]
constexpr size_t kNTilesOffset = 4096;         // int32
constexpr size_t kTilesOffset = 4352;          // Tile [ceil(T*k/128) + min(E, T*k)]

static_assert(kCountsOffset + kNoAllocMaxExperts * sizeof(int32_t) <= kNTilesOffset, "layout");
static_assert(kTilesOffset + (kNoAllocMaxPairs / lmoe::kBM + kNoAllocMaxExperts) * sizeof(lmoe::Tile) <=
                  kNoAllocScratchBytes,
              "layout");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// True when `p` is device (or managed) memory that device `dev` can use as its own.
bool on_device(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();   // an unknown pointer must not leave an error behind
    return false;
  }
  if (a.type == cudaMemoryTypeManaged) return true;
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

}  // namespace

extern "C" lmoe_status lmoe_permute_noalloc(const int32_t* topk_idx, int T, int k, int E,
                                            int32_t* offsets, int32_t* row_of, int32_t* tok_of,
                                            cudaStream_t stream) {
  if (T < 0 || k < 1 || k > 16 || E < 1 || k > E) return LMOE_ERR_ARG;
  if (E > kNoAllocMaxExperts || static_cast<long long>(T) * k > kNoAllocMaxPairs)
    return LMOE_ERR_UNSUPPORTED;  // beyond the fixed scratch array
  if (offsets == nullptr || (T > 0 && (topk_idx == nullptr || row_of == nullptr || tok_of == nullptr)))
    return LMOE_ERR_ARG;
  // the kernels do plain int32 loads and stores on these arrays
  if (!aligned4(offsets) || (T > 0 && (!aligned4(topk_idx) || !aligned4(row_of) || !aligned4(tok_of))))
    return LMOE_ERR_ALIGN;
  // The scratch address is looked up for the current device and the kernels run on the
  // stream's device: they must be the same device, and so must the arrays' device.
  int dev = 0, sdev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaStreamGetDevice(stream, &sdev) != cudaSuccess)
    return LMOE_ERR_CUDA;
  if (sdev != dev) return LMOE_ERR_ARG;
  if (!on_device(offsets, dev) ||
      (T > 0 && (!on_device(topk_idx, dev) || !on_device(row_of, dev) || !on_device(tok_of, dev))))
    return LMOE_ERR_ARG;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return LMOE_ERR_CUDA;
  unsigned char* s = static_cast<unsigned char*>(base);
  // Nothing here must start at zero: the count kernel overwrites counts[e] for every e, the
  // scatter overwrites every tile it reports and the tile count, and offsets/row_of/tok_of
  // are outputs.  So no clearing pass is needed between calls.
  if (lmoe::launch_permute(topk_idx, T, k, E, reinterpret_cast<int32_t*>(s + kCountsOffset), offsets,
                           row_of, tok_of, reinterpret_cast<lmoe::Tile*>(s + kTilesOffset),
                           reinterpret_cast<int32_t*>(s + kNTilesOffset), stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}
