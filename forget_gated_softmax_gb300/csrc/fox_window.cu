// Epsilon-effective window of every query row (foxwindow README, "The window
// is a first-passage time"): with X_t = -log g_t, row i's window is
//   N_i(eps) = inf{ n >= 1 : X_i + ... + X_{i-n+1} > L },  L = ln(1/eps),
// one more than the largest distance whose decay prod g_t is still >= eps; -1
// when the whole prefix does not pass L. The walk's partial sums are
// c_{i-n} - c_i with c the prefix sums of log g, non-increasing, so the first
// passage is a binary search on c. The prefix sums (chunk-local scans plus
// chunk bases) and the comparison are fp64, so the integer result is decided
// in the same precision as a double-precision statement of the definition.
#include <cuda_runtime.h>

#include "fox_internal.h"

namespace fox {
namespace {

constexpr int kChunk = 1024;  // tokens per local scan
constexpr int kChunkThreads = 256;

__device__ __forceinline__ double log_sigmoid64(float zf) {
  const double z = (double)zf;
  return fmin(z, 0.0) - log1p(exp(-fabs(z)));  // 0 at z = +inf
}

// CTA per (b*H + h, chunk of 1024 tokens), flattened: local inclusive fp64 sums of
// log sigmoid(z) and the chunk total. Spread over all SMs: fp64 exp / log1p
// are the bulk of the work.
__global__ void __launch_bounds__(kChunkThreads) window_local_kernel(const float* __restrict__ z, int N, int H,
                                                                    int Npad, int nChunks, double* __restrict__ loc64,
                                                                    double* __restrict__ tot64) {
  __shared__ double wsum[kChunkThreads / 32];
  const int chunk = static_cast<int>(blockIdx.x % nChunks), bh = static_cast<int>(blockIdx.x / nChunks);
  const int b = bh / H, h = bh % H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kPer = kChunk / kChunkThreads;
  double v[kPer];
  double run = 0.0;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int t = chunk * kChunk + tid * kPer + e;
    run += t < N ? log_sigmoid64(z[((size_t)b * N + t) * H + h]) : 0.0;
    v[e] = run;
  }
  double x = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  double before = 0.0;
  for (int w = 0; w < warp; ++w) before += wsum[w];
  const double excl = before + (x - run);
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int t = chunk * kChunk + tid * kPer + e;
    if (t < N) loc64[(size_t)bh * Npad + t] = excl + v[e];
  }
  if (tid == kChunkThreads - 1) tot64[(size_t)bh * nChunks + chunk] = excl + run;
}

// One warp per (b, h): exclusive fp64 scan of the chunk totals -> chunk bases (in place).
__global__ void __launch_bounds__(256) window_base_kernel(int BH, int nChunks, double* __restrict__ tot64) {
  const int bh = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (bh >= BH) return;
  double carry = 0.0;
  for (int c0 = 0; c0 < nChunks; c0 += 32) {
    const int c = c0 + lane;
    const double v = c < nChunks ? tot64[(size_t)bh * nChunks + c] : 0.0;
    double incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (c < nChunks) tot64[(size_t)bh * nChunks + c] = carry + incl - v;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// One thread per (b, i, h), in output order.
__global__ void __launch_bounds__(256) window_search_kernel(const double* __restrict__ loc64,
                                                           const double* __restrict__ base64, int B, int N, int H,
                                                           int Npad, int nChunks, double L, int* __restrict__ out) {
  const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= (long long)B * N * H) return;
  const int h = (int)(row % H);
  const long long bi = row / H;
  const int i = (int)(bi % N), b = (int)(bi / N);
  const size_t bh = (size_t)b * H + h;
  const double* lc = loc64 + bh * Npad;
  const double* bs = base64 + bh * nChunks;
  auto c = [&](int t) { return bs[t / kChunk] + lc[t]; };  // prefix sum of log sigmoid(z) up to t
  const double ci = c(i);
  int result = -1;
  if (-ci > L) {  // c_{-1} - c_i = -c_i: the whole prefix passes L
    // largest j in [-1, i-1] with c_j - c_i > L (true at j = -1, false at j = i)
    int lo = -1, hi = i;
    while (hi - lo > 1) {
      const int mid = lo + ((hi - lo) >> 1);
      if (c(mid) - ci > L)
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
  const int nChunks = (N + kChunk - 1) / kChunk;
  double* loc64 = reinterpret_cast<double*>(static_cast<char*>(ws) + kErrWordBytes);
  double* tot64 = loc64 + (size_t)B * H * Npad;
  {
    TraceScope trace("window_local", s);
    const long long blocks = (long long)nChunks * B * H;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    window_local_kernel<<<(unsigned)blocks, kChunkThreads, 0, s>>>(z, N, H, Npad, nChunks, loc64, tot64);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    TraceScope trace("window_base", s);
    window_base_kernel<<<(B * H + 7) / 8, 256, 0, s>>>(B * H, nChunks, tot64);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long rows = (long long)B * N * H;
  {
    TraceScope trace("window_search", s);
    window_search_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(loc64, tot64, B, N, H, Npad, nChunks,
                                                                        log(1.0 / eps), out);
  }
  return cudaGetLastError();
}

size_t window_workspace_bytes(int B, int N, int H) {
  const size_t Npad = ((size_t)N + kTile - 1) / kTile * kTile;
  const size_t nChunks = ((size_t)N + kChunk - 1) / kChunk;
  return kErrWordBytes + sizeof(double) * (size_t)B * H * (Npad + nChunks);
}

}  // namespace fox
