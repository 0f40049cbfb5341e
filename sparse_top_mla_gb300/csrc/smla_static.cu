// smla_decode_static: the split-K decode schedule with its scratch in a fixed device array
// owned by the library, for callers that cannot allocate device memory themselves.
//
// Who needs it: callers that hold no allocator to hand the library a workspace — a plugin
// behind a fixed C interface that passes only the problem tensors, or a runtime whose device
// memory is entirely owned by its own pool and which forbids allocations outside it. For
// them this entry point takes the same smla_params and ignores `workspace`.
//
// The scratch is the file-scope array below (kStaticScratchBytes, 32 MiB). Every GPU that
// loads libsmla holds it until the process exits. Host code may not pass the array's name
// to a kernel (on the host it is only a stand-in for the symbol), so the device address is
// looked up with cudaGetSymbolAddress once per device, with that device current, the first
// time this entry point runs on it; make that first call before any stream capture.
#include <cuda_runtime.h>

#include <atomic>

#include "smla.h"
#include "smla_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

// Split-K partial outputs and log-sum-exps of the most recent call. Shared by every call on
// the device: two calls that overlap on the GPU (different streams, no ordering) race on it.
// Nothing in it needs to start at zero: each call writes every partial it later reads.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of g_static_scratch on the current device (set-up on first use).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    smla::note_cuda_error(e, "cudaGetDevice (smla_decode_static)");
    return e;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    smla::note_cuda_error(cudaErrorInvalidDevice, "device index beyond the static scratch table");
    return cudaErrorInvalidDevice;
  }
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) {
      smla::note_cuda_error(e, "cudaGetSymbolAddress(g_static_scratch)");
      return e;
    }
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" {

smla_status smla_decode_static(const smla_params* p, smla_stream_t stream) {
  if (p == nullptr) return SMLA_ERR_INVALID;
  const size_t need = smla_workspace_size(p);  // 0 for a malformed problem or one needing no split
  if (need > kStaticScratchBytes) return SMLA_ERR_WORKSPACE;
  smla_params q = *p;
  q.workspace = nullptr;
  q.workspace_bytes = 0;
  if (need > 0) {
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return SMLA_ERR_CUDA;
    q.workspace = scratch;
    q.workspace_bytes = kStaticScratchBytes;
  }
  return smla_decode(&q, stream);  // validates everything else exactly as the allocating entry point
}

}  // extern "C"
