// Gate kernels: log-sigmoid of the forget-gate logits and the per-head prefix
// scan of log f ("Forgetting Transformer (FoX) Attention" module source,
// ForgettingAttention.forward: sigmoid of the gate projection, log, cumsum
// along the sequence), stored two-level so that the attention kernels can
// form D_ij = c_i - c_j to fp32 accuracy at any sequence length:
// tile-local fp32 sums (warp-shuffle scan over 128 tokens) plus per-tile
// bases from an fp64 scan over tile totals.
#include <cuda_runtime.h>

#include "fox_internal.h"

namespace fox {
namespace {

constexpr int kHeadsPerPass = 32;

// log sigmoid(z) = min(z, 0) - log1p(exp(-|z|)); exactly 0 at z = +inf.
__device__ __forceinline__ float log_sigmoid(float z) { return fminf(z, 0.f) - log1pf(expf(-fabsf(z))); }

__device__ __forceinline__ float warp_inclusive_scan(float x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// One CTA per (tile T, batch b); all heads of that tile. z rows of one token
// are contiguous over heads, so the load is coalesced; each warp then scans
// one head's 128 tokens (4 per lane, serial, then a shuffle scan).
__global__ void __launch_bounds__(256) gate_tile_scan_kernel(const float* __restrict__ z, int B, int N, int H,
                                                             int nT, int Npad, int bias_from_j,
                                                             float* __restrict__ rowloc, float* __restrict__ colrec,
                                                             float* __restrict__ tiletot, uint32_t* err) {
  __shared__ float zs[kTile][kHeadsPerPass + 1];
  const int T = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (T == 0 && b == 0 && threadIdx.x == 0 && err) *err = 0u;  // each call starts with a clean error word
  const int t0 = T * kTile;
  for (int h0 = 0; h0 < H; h0 += kHeadsPerPass) {
    const int nh = min(kHeadsPerPass, H - h0);
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * kHeadsPerPass; e += blockDim.x) {
      const int r = e / kHeadsPerPass, c = e % kHeadsPerPass;
      const int t = t0 + r;
      float a = 0.f;  // tokens past the end contribute log f = 0
      if (t < N && c < nh) a = log_sigmoid(z[((size_t)b * N + t) * H + h0 + c]) * kLog2e;
      zs[r][c] = a;
    }
    __syncthreads();
    for (int c = warp; c < nh; c += blockDim.x / 32) {
      const int h = h0 + c;
      const size_t bh = (size_t)b * H + h;
      float a[4], incl[4];
      float run = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        a[e] = zs[lane * 4 + e][c];
        run += a[e];
        incl[e] = run;
      }
      const float lane_incl = warp_inclusive_scan(run, lane);
      const float excl_lane = lane_incl - run;
#pragma unroll
      for (int e = 0; e < 4; ++e) incl[e] += excl_lane;
      float4 rl = make_float4(incl[0], incl[1], incl[2], incl[3]);
      *reinterpret_cast<float4*>(rowloc + bh * Npad + t0 + lane * 4) = rl;
      float4 cl = bias_from_j ? make_float4(incl[0] - a[0], incl[1] - a[1], incl[2] - a[2], incl[3] - a[3]) : rl;
      // keys past the sequence end get an infinite column term: x = ... - kappa = -inf, p = 0
      const int tl = t0 + lane * 4;
      if (tl + 0 >= N) cl.x = INFINITY;
      if (tl + 1 >= N) cl.y = INFINITY;
      if (tl + 2 >= N) cl.z = INFINITY;
      if (tl + 3 >= N) cl.w = INFINITY;
      *reinterpret_cast<float4*>(colrec + (bh * nT + T) * kColRec + lane * 4) = cl;
      if (lane == 31) tiletot[bh * nT + T] = incl[3];
    }
  }
}

// One warp per (b, h): exclusive fp64 scan of the tile totals -> base_T,
// stored as an fp32 hi/lo pair in each column record.
__global__ void __launch_bounds__(256) gate_base_scan_kernel(int BH, int nT, const float* __restrict__ tiletot,
                                                             float* __restrict__ colrec) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= BH) return;
  double carry = 0.0;
  for (int T0 = 0; T0 < nT; T0 += 32) {
    const int T = T0 + lane;
    const double v = T < nT ? (double)tiletot[(size_t)warp * nT + T] : 0.0;
    double incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const double base = carry + incl - v;
    if (T < nT) {
      float* rec = colrec + ((size_t)warp * nT + T) * kColRec;
      const float hi = (float)base;
      const float lo = (float)(base - (double)hi);
      *reinterpret_cast<float4*>(rec + kTile) = make_float4(hi, lo, 0.f, 0.f);
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
}

}  // namespace

cudaError_t launch_gate_scan(const float* z, int B, int N, int H, int bias_from_j, void* ws, const GateLayout& g,
                             cudaStream_t s) {
  char* base = static_cast<char*>(ws);
  float* rowloc = reinterpret_cast<float*>(base + g.rowloc);
  float* colrec = reinterpret_cast<float*>(base + g.colrec);
  float* tiletot = reinterpret_cast<float*>(base + g.tiletot);
  uint32_t* err = reinterpret_cast<uint32_t*>(base);
  dim3 grid(g.nT, B);
  {
    TraceScope trace("gate_tile_scan", s);
    gate_tile_scan_kernel<<<grid, 256, 0, s>>>(z, B, N, H, g.nT, g.Npad, bias_from_j, rowloc, colrec, tiletot, err);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int warps_per_block = 8;
  {
    TraceScope trace("gate_base_scan", s);
    gate_base_scan_kernel<<<(g.BH + warps_per_block - 1) / warps_per_block, 256, 0, s>>>(g.BH, g.nT, tiletot, colrec);
  }
  return cudaGetLastError();
}

}  // namespace fox
