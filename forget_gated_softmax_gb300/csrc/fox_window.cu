// Epsilon-effective window of every query row (foxwindow README, "The window
// is a first-passage time"): with X_t = -log g_t, row i's window is
//   N_i(eps) = inf{ n >= 1 : X_i + ... + X_{i-n+1} > L },  L = ln(1/eps),
// one more than the largest distance whose decay prod g_t is still >= eps; -1
// when the whole prefix does not pass L. The walk's partial sums are
// c_{i-n} - c_i with c the prefix sums of log g, non-increasing, so the first
// passage is a binary search on c. Both kernels work in fp64 so that the
// integer result is decided in the same precision as a double-precision
// statement of the definition.
#include <cuda_runtime.h>

#include "fox_internal.h"

namespace fox {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kPerThread = 8;

__device__ __forceinline__ double log_sigmoid64(float zf) {
  const double z = (double)zf;
  return fmin(z, 0.0) - log1p(exp(-fabs(z)));  // 0 at z = +inf
}

// One CTA per (b, h): c64[bh][t] = sum_{l<=t} log sigmoid(z_l), fp64.
__global__ void __launch_bounds__(kScanThreads) window_scan64_kernel(const float* __restrict__ z, int N, int H,
                                                                    int Npad, double* __restrict__ c64) {
  __shared__ double wsum[kScanThreads / 32];
  const int bh = blockIdx.x, b = bh / H, h = bh % H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  double carry = 0.0;
  for (int t0 = 0; t0 < N; t0 += kScanThreads * kPerThread) {
    double loc[kPerThread];
    double run = 0.0;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int t = t0 + tid * kPerThread + e;
      run += t < N ? log_sigmoid64(z[((size_t)b * N + t) * H + h]) : 0.0;
      loc[e] = run;
    }
    double x = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      double w = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      wsum[lane] = w;
    }
    __syncthreads();
    const double excl = carry + (warp > 0 ? wsum[warp - 1] : 0.0) + (x - run);
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int t = t0 + tid * kPerThread + e;
      if (t < N) c64[(size_t)bh * Npad + t] = excl + loc[e];
    }
    carry += wsum[kScanThreads / 32 - 1];
    __syncthreads();
  }
}

// One thread per (b, i, h), in output order.
__global__ void __launch_bounds__(256) window_search_kernel(const double* __restrict__ c64, int B, int N, int H,
                                                           int Npad, double L, int* __restrict__ out) {
  const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= (long long)B * N * H) return;
  const int h = (int)(row % H);
  const long long bi = row / H;
  const int i = (int)(bi % N), b = (int)(bi / N);
  const double* c = c64 + ((size_t)b * H + h) * Npad;
  const double ci = c[i];
  int result = -1;
  if (-ci > L) {  // c_{-1} - c_i = -c_i: the whole prefix passes L
    // largest j in [-1, i-1] with c_j - c_i > L (true at j = -1, false at j = i)
    int lo = -1, hi = i;
    while (hi - lo > 1) {
      const int mid = lo + ((hi - lo) >> 1);
      if (c[mid] - ci > L)
        lo = mid;
      else
        hi = mid;
    }
    result = i - lo;
  }
  out[row] = result;
}

}  // namespace

cudaError_t launch_window(const float* z, int B, int N, int H, double eps, int* out, void* ws, cudaStream_t s) {
  const int Npad = ((N + kTile - 1) / kTile) * kTile;
  double* c64 = reinterpret_cast<double*>(static_cast<char*>(ws) + kErrWordBytes);
  {
    TraceScope trace("window_scan64", s);
    window_scan64_kernel<<<B * H, kScanThreads, 0, s>>>(z, N, H, Npad, c64);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long rows = (long long)B * N * H;
  {
    TraceScope trace("window_search", s);
    window_search_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(c64, B, N, H, Npad, log(1.0 / eps), out);
  }
  return cudaGetLastError();
}

size_t window_workspace_bytes(int B, int N, int H) {
  const size_t Npad = ((size_t)N + kTile - 1) / kTile * kTile;
  return kErrWordBytes + sizeof(double) * (size_t)B * H * Npad;
}

}  // namespace fox
