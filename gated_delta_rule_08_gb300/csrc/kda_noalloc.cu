// kda_chunk_fwd_noalloc: chunked prefill for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point where
// they run the prefill: code running under a foreign allocator that owns all device
// memory, plugin hosts that forbid allocation on their execution path, or runtimes
// that have already fixed their memory footprint.  kda_chunk_fwd needs a scratch
// workspace from its caller; this variant instead uses one fixed scratch array that
// the library owns, declared below as a file-scope __device__ array.  Loading the
// library on a device reserves that array on the device until the process exits.
//
// The kernels, arguments and results are exactly those of kda_chunk_fwd; only the
// origin of the scratch differs.  Host code cannot use the array's name as a device
// address (it names a host-side stand-in), so the device address is looked up with
// cudaGetSymbolAddress, once per device, on that device's first call.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kda.h"

#define KDA_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kScratchBytes = (size_t)64 << 20;  // 64 MiB per device
constexpr int kMaxDevices = 64;

// The library-owned scratch.  Shared by every call on the device: calls whose GPU
// work overlaps in time (different streams without ordering) race on it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on first use).
kda_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return KDA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KDA_OK;
}

}  // namespace

KDA_API size_t kda_noalloc_scratch_bytes(void) { return kScratchBytes; }

KDA_API kda_status kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                         const float* beta, const float* h0, const int32_t* cu_seqlens,
                                         void* out, float* hT, int B, int64_t T, int H, int dk, int dv, int C,
                                         kda_dtype dtype, kda_dtype out_dtype, const kda_epilogue* epi,
                                         void* stream) {
  const size_t need = kda_chunk_fwd_workspace_size(B, T, H, dk, dv, C, dtype);
  if (need == 0) {
    // Same argument classification as kda_chunk_fwd (it rejects these before any launch).
    return kda_chunk_fwd(q, k, v, g, beta, h0, cu_seqlens, out, hT, B, T, H, dk, dv, C, dtype, out_dtype, epi,
                         nullptr, 0, stream);
  }
  if (need > kScratchBytes) return KDA_ERR_WORKSPACE;  // problem larger than the built-in scratch
  void* scratch = nullptr;
  const kda_status st = scratch_address(&scratch);
  if (st != KDA_OK) return st;
  return kda_chunk_fwd(q, k, v, g, beta, h0, cu_seqlens, out, hT, B, T, H, dk, dv, C, dtype, out_dtype, epi,
                       scratch, kScratchBytes, stream);
}
