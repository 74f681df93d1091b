// fox_selftest_wait_timeout: a self-test of the device-side error path.
//
// Every wait in the attention kernels is bounded: a wait that runs out raises the
// CTA's shared abort flag (which releases the CTA's other waits at once), ORs a bit
// into the workspace's error word and returns, so the kernel ends and the context
// stays usable; fox_check_error reports the bit. In normal operation no wait ever
// runs out, so this kernel makes one run out on purpose, with the same wait code:
//   warp 0 waits on an mbarrier that nothing arrives at, for limit_ns;
//   warp 1 waits on a second such mbarrier with a 16x longer limit, and must be
//   released by warp 0's abort flag rather than by its own limit.
// The error word then holds warp 0's code only (DEV_ERR_TIMEOUT_SYNC); the words
// after it record what each wait returned. Nothing is copied, no tensor memory is
// allocated, and both waits end within 16 * limit_ns in the worst case.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/fox.h"
#include "fox_internal.h"
#include "fox_ptx.cuh"

namespace fox {
namespace {

__global__ void __launch_bounds__(64) selftest_wait_kernel(uint32_t* header, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    header[1] = 0xFFFFFFFFu;
    header[2] = 0xFFFFFFFFu;
    fence_mbar_init();
  }
  __syncthreads();
  if (lane == 0) {
    // Phase 0 of a fresh barrier completes only when its one expected arrival comes.
    if (warp == 0)
      header[1] = mbar_wait_for(&bars[0], 0, abort_flag, header, DEV_ERR_TIMEOUT_SYNC, limit_ns) ? 1u : 0u;
    else
      header[2] = mbar_wait_for(&bars[1], 0, abort_flag, header, DEV_ERR_TIMEOUT_MMA, 16 * limit_ns) ? 1u : 0u;
  }
  __syncthreads();
}

}  // namespace
}  // namespace fox

extern "C" fox_status fox_selftest_wait_timeout(unsigned limit_us, void* workspace, size_t workspace_bytes,
                                                void* stream) {
  if (limit_us < 1 || limit_us > 100000) return FOX_ERR_INVALID_ARG;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 || workspace_bytes < fox::kErrWordBytes)
    return FOX_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* header = static_cast<uint32_t*>(workspace);
  if (cudaMemsetAsync(header, 0, sizeof(uint32_t), s) != cudaSuccess) return FOX_ERR_CUDA;
  fox::selftest_wait_kernel<<<1, 64, 0, s>>>(header, static_cast<uint64_t>(limit_us) * 1000ull);
  return cudaGetLastError() == cudaSuccess ? FOX_OK : FOX_ERR_CUDA;
}
