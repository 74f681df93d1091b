// fox_fwd_noalloc: the forward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) where they
// run this library: a plugin inside a host application that owns all device
// memory and does not let its plugins allocate, or a latency-bound loop that
// cannot afford an allocation's implicit synchronisation. fox_fwd needs a
// caller-provided workspace for the gate terms (and, when it has room, an fp16
// copy of V); this entry point instead uses
// a fixed scratch array compiled into the library (kStaticScratchBytes, held
// by every GPU that loads the library until the process exits). The caller
// still passes inputs and outputs.
//
// Host code sees the array's name only as a host-side stand-in, so the device
// address is looked up with cudaGetSymbolAddress once per device, with that
// device current, on the first call made on it; that first call should come
// before any stream capture. Every call shares the one array: the scratch is
// fully rewritten by each call (its error word is cleared by the first kernel),
// and calls whose work overlaps on the GPU race on it. fox_noalloc_check_error
// reads the array's error word. The cached address lives as long as the process:
// after a cudaDeviceReset the array is gone with the context, and this entry
// point must not be used on that device again.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fox.h"
#include "fox_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_fox_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_fox_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t fox_noalloc_scratch_bytes(void) { return kStaticScratchBytes; }

// The scratch array's error word, read and cleared like any workspace's.
fox_status fox_noalloc_check_error(void* stream) {
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return FOX_ERR_CUDA;
  return fox_check_error(scratch, stream);
}

fox_status fox_fwd_noalloc(const fox_params* p, const void* q, const void* k, const void* v, const float* z, void* o,
                           float* lse, void* stream) {
  if (!p) return FOX_ERR_INVALID_ARG;
  // The gate terms must fit; the fp16 copy of V is used when it fits too (fox_fwd decides by size).
  const size_t need = fox_fwd_min_workspace_bytes(p);
  if (need == 0) return fox_fwd(p, q, k, v, z, o, lse, nullptr, 0, stream);  // reports the parameter error
  if (need > kStaticScratchBytes) return FOX_ERR_WORKSPACE;                  // larger than the fixed scratch
  if (p->B == 0 || p->H == 0 || p->N == 0) return FOX_OK;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return FOX_ERR_CUDA;
  return fox_fwd(p, q, k, v, z, o, lse, scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
