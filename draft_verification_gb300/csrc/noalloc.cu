// spec_verify_chain_noalloc: chain verification without a caller workspace.
//
// Some callers cannot hand the library a workspace: code that must not call
// cudaMalloc at all (an inference loop whose memory is budgeted up front, a
// plugin running inside a host framework that owns every allocation, or a
// process that is not allowed to allocate device memory while serving).  For
// them the scratch lives in one fixed array in this file, reserved when the
// library is loaded, and this entry point allocates nothing.
//
// The array is shared by every call on a device and keeps whatever the last
// call left in it; calls that overlap on the GPU (two streams, or two host
// threads) race on it and must be serialised by the caller.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "spec_verify.h"

namespace {

// Held by every GPU that loads the library until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of the array on the current device.  The host-side name of
// a __device__ array is only a stand-in: a kernel must be given the address
// this query returns, never the symbol itself.  Done once per device, with
// that device current (the first call on the device does it).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return e;
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" spec_status spec_verify_chain_noalloc(const spec_chain_args* args, cudaStream_t stream) {
  sv::NvtxRange nvtx_range("spec_verify_chain_noalloc");
  if (args == nullptr) return SPEC_EINVAL;
  // Refuse calls whose scratch would not fit before touching the device.
  if (args->B < 1 || args->B > 65535 || args->gamma < 0 || args->gamma > 32 || args->V < 1) return SPEC_EINVAL;
  if (spec_chain_workspace_size(args->B, args->gamma, args->V) > SPEC_NOALLOC_SCRATCH_BYTES)
    return SPEC_EWORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return SPEC_ECUDA;
  // The scratch holds only the statistics partials, which a call writes
  // before it reads them (the consulted-only mode uses none), so nothing a
  // previous call left behind is ever read and nothing needs clearing.
  spec_chain_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = SPEC_NOALLOC_SCRATCH_BYTES;
  return sv::verify_chain(&a, stream, false);  // no library streams or events
}
