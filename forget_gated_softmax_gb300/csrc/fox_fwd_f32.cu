// fp32 forward of forget-gated causal attention on CUDA cores (SIMT), for
// inputs held in fp32 where the bf16 tensor-core path would not meet an fp32
// tolerance. Same math as the bf16 kernel ("Forgetting Transformer (FoX)
// Attention" module source, ForgettingAttention.forward): one warp per query
// row, lanes split the head dimension, online softmax over keys j <= i in
// log2 units with the two-level gate terms.
#include <cuda_runtime.h>

#include "fox_internal.h"

namespace fox {
namespace {

constexpr int kRowsPerBlock = 8;

template <int D>
__global__ void __launch_bounds__(32 * kRowsPerBlock) fox_attn_fwd_f32_kernel(
    int B, int N, int H, int nT, int Npad, float scale2, const float* __restrict__ q, const float* __restrict__ k,
    const float* __restrict__ v, const float* __restrict__ rowloc, const float* __restrict__ colrec,
    float* __restrict__ o, float* __restrict__ lse) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * kRowsPerBlock + warp;
  const int bh = blockIdx.y;
  if (i >= N) return;
  const int b = bh / H, h = bh % H;
  const size_t row_stride = (size_t)H * D;
  const float* qi = q + (((size_t)b * N + i) * H + h) * D;
  const float* kb = k + ((size_t)b * N * H + h) * D;
  const float* vb = v + ((size_t)b * N * H + h) * D;
  float qr[E], acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    qr[e] = qi[e * 32 + lane];
    acc[e] = 0.f;
  }
  const int I = i / kTile;
  const float* rec = colrec + (size_t)bh * nT * kColRec;
  const float baseI_hi = rec[(size_t)I * kColRec + kTile], baseI_lo = rec[(size_t)I * kColRec + kTile + 1];
  float m = -INFINITY, l = 0.f, beta = 0.f;
  for (int j = 0; j <= i; ++j) {
    const int J = j / kTile, jj = j % kTile;
    if (jj == 0 || j == 0) {
      const float* rJ = rec + (size_t)J * kColRec;
      beta = (baseI_hi - rJ[kTile]) + (baseI_lo - rJ[kTile + 1]);
    }
    const float* kj = kb + (size_t)j * row_stride;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) dot = fmaf(qr[e], kj[e * 32 + lane], dot);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const float y = fmaf(dot, scale2, -rec[(size_t)J * kColRec + jj]) + beta;
    const float m_new = fmaxf(m, y);
    const float corr = exp2f(m - m_new);
    const float pj = exp2f(y - m_new);
    l = l * corr + pj;
    const float* vj = vb + (size_t)j * row_stride;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(pj, vj[e * 32 + lane], acc[e] * corr);
    m = m_new;
  }
  const float inv = 1.f / l;
  float* oi = o + (((size_t)b * N + i) * H + h) * D;
#pragma unroll
  for (int e = 0; e < E; ++e) oi[e * 32 + lane] = acc[e] * inv;
  if (lane == 0) lse[((size_t)b * N + i) * H + h] = (m + log2f(l) + rowloc[(size_t)bh * Npad + i]) * kLn2;
}

}  // namespace

cudaError_t launch_attn_fwd_f32(const AttnFwdArgs& a, int nT, int Npad, cudaStream_t s) {
  const int BH = a.B * a.H;
  if (BH > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid((a.N + kRowsPerBlock - 1) / kRowsPerBlock, BH);
  const float scale2 = a.scale * kLog2e;
  const float* q = static_cast<const float*>(a.q);
  const float* k = static_cast<const float*>(a.k);
  const float* v = static_cast<const float*>(a.v);
  float* o = static_cast<float*>(a.o);
  TraceScope trace("attn_fwd_f32", s);
  if (a.d == 64)
    fox_attn_fwd_f32_kernel<64><<<grid, 32 * kRowsPerBlock, 0, s>>>(a.B, a.N, a.H, nT, Npad, scale2, q, k, v,
                                                                      a.rowloc, a.colrec, o, a.lse);
  else if (a.d == 128)
    fox_attn_fwd_f32_kernel<128><<<grid, 32 * kRowsPerBlock, 0, s>>>(a.B, a.N, a.H, nT, Npad, scale2, q, k, v,
                                                                       a.rowloc, a.colrec, o, a.lse);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace fox
