// Decay-aware tile skipping for the causal attention kernels.
//
// Every log f_t < 0, so the forget bias falls monotonically with the distance
// i - j (foxwindow README, "The window is a first-passage time"). For query
// tile I and an earlier key tile J, in log2 units, with i0 the first row of I
// and j1 the last key of J (Cauchy-Schwarz on q_i.k_j and on q_i.k_i):
//   x_ij - max_j' x_ij'  <=  x_ij - x_ii
//                        <=  scale log2e qmax_I (kmax_J + kmax_I) + colterm(i0) - colterm(j1)  =: U(I, J)
// where qmax_T, kmax_T are the largest row norms of q, k in tile T and
// colterm(t) = base_T + kappa_t is the gate scan's column term. When
// U < -150 every weight of the pair is below 2^-150 of its row's largest, and
// the flushing exp2 of the attention kernels returns exactly 0 for all of
// them: skipping the pair leaves every output bit unchanged.
//
// kmax_J is replaced by its running maximum over tiles 0..J, which keeps the
// bound valid and makes it non-increasing as J moves back, so the skipped key
// tiles of query tile I are J < jraw(I). The start is then made non-decreasing
// in I (jmin(I) = min over I' >= I of jraw(I'); keeping more pairs is always
// exact), so that every key tile J serves the contiguous query tiles
// J..imax(J), which is what the backward kernel (one CTA per key tile) needs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fox_internal.h"

namespace fox {
namespace {

constexpr double kSkipLog2 = 150.0;  // skip below 2^-150 of the row's largest weight
constexpr int kSpanThreads = 512;

// CTA per (tile T, b*H + h): largest row norms of q and k over the tile's
// rows t < N (fp32 sum of the exact bf16 squares, then sqrtf). Each warp takes 16 rows:
// all their q and k loads are issued first (rows past N read as zero), each lane forms its
// partial sums of squares, and one reduce-scatter across the warp (halving rounds) leaves
// lane l with the full sum of q row l (l < 16) or k row l - 16; the row maxima follow.
template <int D>
__global__ void __launch_bounds__(256) tile_norm_kernel(const __nv_bfloat16* __restrict__ q,
                                                        const __nv_bfloat16* __restrict__ k, int N, int H, int nT,
                                                        float* __restrict__ qmax, float* __restrict__ kmax) {
  constexpr int E = D / 32;  // bf16 per lane: 4 (D = 128) or 2 (D = 64)
  constexpr int kRowsPerWarp = kTile / 8;  // 16
  __shared__ float red[2][8];
  const int T = static_cast<int>(blockIdx.x % nT);
  const int bh = static_cast<int>(blockIdx.x / nT);
  const int b = bh / H, h = bh % H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t qa[kRowsPerWarp][E / 2], ka[kRowsPerWarp][E / 2];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int t = T * kTile + warp * kRowsPerWarp + rr;
    const size_t base = (((size_t)b * N + t) * H + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E / 2; ++e) {
      qa[rr][e] = t < N ? reinterpret_cast<const uint32_t*>(q + base)[e] : 0u;
      ka[rr][e] = t < N ? reinterpret_cast<const uint32_t*>(k + base)[e] : 0u;
    }
  }
  float v[2 * kRowsPerWarp];  // [0, 16): q rows, [16, 32): k rows (this lane's partial sums)
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int e = 0; e < E / 2; ++e) {
      const float a0 = __uint_as_float(qa[rr][e] << 16), a1 = __uint_as_float(qa[rr][e] & 0xffff0000u);
      const float c0 = __uint_as_float(ka[rr][e] << 16), c1 = __uint_as_float(ka[rr][e] & 0xffff0000u);
      sq = fmaf(a0, a0, fmaf(a1, a1, sq));
      sk = fmaf(c0, c0, fmaf(c1, c1, sk));
    }
    v[rr] = sq;
    v[kRowsPerWarp + rr] = sk;
  }
  // Reduce-scatter: after the round of width w, lane l holds the partial sums of values
  // l mod 2w .. for the half it keeps; after five rounds, the full sum of value l.
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, half);
    }
  }
  // lane l now holds the sum of value l: q row l (l < 16) or k row l - 16; maxima per half
  float m = v[0];
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[0][warp] = m;
  if (lane == 16) red[1][warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f, c = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      a = fmaxf(a, red[0][w]);
      c = fmaxf(c, red[1][w]);
    }
    qmax[(size_t)bh * nT + T] = sqrtf(a);
    kmax[(size_t)bh * nT + T] = sqrtf(c);
  }
}

// Warp 0 of the CTA: running maximum from the front (kMax) or running minimum
// from the back of x[0..n), in place.
template <typename T, bool kMax>
__device__ void warp_running_extreme(T* x, int n, int lane, T identity) {
  auto op = [](T a, T b) { return kMax ? (a > b ? a : b) : (a < b ? a : b); };
  T carry = identity;
  for (int c0 = 0; c0 < n; c0 += 32) {
    const bool in = c0 + lane < n;
    const int i = kMax ? c0 + lane : n - 1 - (c0 + lane);
    T v = in ? x[i] : identity;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v = op(v, y);
    }
    v = op(v, carry);
    if (in) x[i] = v;
    carry = __shfl_sync(0xffffffffu, v, 31);
  }
}

// CTA per b*H + h: kpre (running max of kmax), jmin and imax.
__global__ void __launch_bounds__(kSpanThreads) tile_span_kernel(int nT, double s2, const float* __restrict__ colrec,
                                                                 const float* __restrict__ qmax,
                                                                 const float* __restrict__ kmax,
                                                                 float* __restrict__ kpre, int* __restrict__ jmin,
                                                                 int* __restrict__ imax) {
  const int bh = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const float* rec = colrec + (size_t)bh * nT * kColRec;
  const float* qm = qmax + (size_t)bh * nT;
  const float* km = kmax + (size_t)bh * nT;
  float* kp = kpre + (size_t)bh * nT;
  int* jm = jmin + (size_t)bh * nT;
  int* im = imax + (size_t)bh * nT;
  for (int T = threadIdx.x; T < nT; T += blockDim.x) kp[T] = km[T];
  __syncthreads();
  if (threadIdx.x < 32) warp_running_extreme<float, true>(kp, nT, lane, 0.f);
  __syncthreads();
  // colterm(t) = base_T + kappa_t (log2 units), base as hi + lo
  auto colterm = [&](int T, int r) -> double {
    const float* R = rec + (size_t)T * kColRec;
    return ((double)R[kTile] + (double)R[kTile + 1]) + (double)R[r];
  };
  for (int I = threadIdx.x; I < nT; I += blockDim.x) {
    const double ci0 = colterm(I, 0);
    const double qI = qm[I], kI = km[I];
    auto negligible = [&](int J) {  // U(I, J) < -threshold, J < I
      return s2 * qI * ((double)kp[J] + kI) + (ci0 - colterm(J, kTile - 1)) < -kSkipLog2;
    };
    // largest J < I that is negligible (the negligible ones form a prefix 0..J)
    int lo = -1, hi = I;  // negligible(lo) holds (lo = -1: none), negligible(hi) fails (hi = I: the diagonal)
    while (hi - lo > 1) {
      const int mid = lo + ((hi - lo) >> 1);
      if (negligible(mid))
        lo = mid;
      else
        hi = mid;
    }
    jm[I] = lo + 1;
  }
  __syncthreads();
  // jmin(I) = min over I' >= I of jraw(I')
  if (threadIdx.x < 32) warp_running_extreme<int, false>(jm, nT, lane, 0x7fffffff);
  __syncthreads();
  // imax(J) = largest I >= J with jmin(I) <= J (jmin is non-decreasing, jmin(J) <= J)
  for (int J = threadIdx.x; J < nT; J += blockDim.x) {
    int lo = J, hi = nT;  // jmin(lo) <= J holds; hi = nT is past the end
    while (hi - lo > 1) {
      const int mid = lo + ((hi - lo) >> 1);
      if (jm[mid] <= J)
        lo = mid;
      else
        hi = mid;
    }
    im[J] = lo;
  }
}

}  // namespace

cudaError_t launch_tile_span(const void* q, const void* k, int B, int N, int H, int d, float scale,
                             const GateLayout& g, void* ws, cudaStream_t s) {
  char* base = static_cast<char*>(ws);
  float* qmax = reinterpret_cast<float*>(base + g.qmax);
  float* kmax = reinterpret_cast<float*>(base + g.kmax);
  float* kpre = reinterpret_cast<float*>(base + g.kpre);
  int* jmin = reinterpret_cast<int*>(base + g.jmin);
  int* imax = reinterpret_cast<int*>(base + g.imax);
  const float* colrec = reinterpret_cast<const float*>(base + g.colrec);
  const long long blocks = (long long)g.nT * g.BH;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  {
    TraceScope trace("tile_norm", s);
    const auto* qb = static_cast<const __nv_bfloat16*>(q);
    const auto* kb = static_cast<const __nv_bfloat16*>(k);
    if (d == 128)
      tile_norm_kernel<128><<<(unsigned)blocks, 256, 0, s>>>(qb, kb, N, H, g.nT, qmax, kmax);
    else if (d == 64)
      tile_norm_kernel<64><<<(unsigned)blocks, 256, 0, s>>>(qb, kb, N, H, g.nT, qmax, kmax);
    else
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    TraceScope trace("tile_span", s);
    tile_span_kernel<<<g.BH, kSpanThreads, 0, s>>>(g.nT, (double)scale * (double)kLog2e, colrec, qmax, kmax, kpre,
                                                   jmin, imax);
  }
  return cudaGetLastError();
}

}  // namespace fox
