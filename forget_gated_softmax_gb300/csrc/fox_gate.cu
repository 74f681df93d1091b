// Gate kernels: log-sigmoid of the forget-gate logits and the per-head prefix
// scan of log f ("Forgetting Transformer (FoX) Attention" module source,
// ForgettingAttention.forward: sigmoid of the gate projection, log, cumsum
// along the sequence), stored two-level so that the attention kernels can
// form D_ij = c_i - c_j to fp32 accuracy at any sequence length:
// tile-local fp32 sums (warp-shuffle scan over 128 tokens) plus per-tile
// bases from a double-float (about 48-bit) scan over tile totals.
#include <cuda_runtime.h>

#include "fox_internal.h"
#include "fox_ptx.cuh"

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

// One warp scans one head's 128 tokens of tile T (4 per lane, serial, then a
// shuffle scan) from column c of the staged log-gate values zs[token][c]
// (log2 units, 0 past the sequence end), and writes the tile-local row terms,
// the column record's 128 column terms and the tile total.
__device__ __forceinline__ void scan_head_column(const float (*zs)[kHeadsPerPass + 1], int c, int lane, size_t bh,
                                                 int T, int N, int nT, int Npad, int bias_from_j,
                                                 float* __restrict__ rowloc, float* __restrict__ colrec,
                                                 float* __restrict__ tiletot) {
  const int t0 = T * kTile;
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

// One CTA per (tile T, batch b, group of kTileScanHeads heads). Each thread loads its
// z values first (a warp reads 2 tokens x 16 heads, whole 32-byte sectors), then takes
// the log-sigmoids; each warp then scans one or two heads' 128 tokens.
constexpr int kTileScanHeads = 16;

__global__ void __launch_bounds__(256) gate_tile_scan_kernel(const float* __restrict__ z, int B, int N, int H,
                                                             int nT, int Npad, int bias_from_j,
                                                             float* __restrict__ rowloc, float* __restrict__ colrec,
                                                             float* __restrict__ tiletot, uint32_t* err) {
  __shared__ float zs[kTile][kHeadsPerPass + 1];
  const int T = blockIdx.x, b = blockIdx.y, h0 = blockIdx.z * kTileScanHeads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_trigger();  // the base scan may start launching (it waits for this kernel's results)
  if (T == 0 && b == 0 && h0 == 0 && threadIdx.x == 0 && err) *err = 0u;  // each call starts with a clean error word
  const int t0 = T * kTile;
  const int nh = min(kTileScanHeads, H - h0);
  constexpr int kPer = kTile * kTileScanHeads / 256;  // values per thread
  float v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = threadIdx.x + u * 256, r = e / kTileScanHeads, c = e % kTileScanHeads;
    const int t = t0 + r;
    v[u] = (t < N && c < nh) ? z[((size_t)b * N + t) * H + h0 + c] : INFINITY;  // log f = 0 past the end
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = threadIdx.x + u * 256;
    zs[e / kTileScanHeads][e % kTileScanHeads] = log_sigmoid(v[u]) * kLog2e;
  }
  __syncthreads();
  for (int c = warp; c < nh; c += 8)
    scan_head_column(zs, c, lane, (size_t)b * H + h0 + c, T, N, nT, Npad, bias_from_j, rowloc, colrec, tiletot);
}

// ---------------------------------------------------------------- fused gate projection
// z = x W_f^T + b_f ("Forgetting Transformer (FoX) Attention" module source:
// f_proj = Linear(hidden_size, num_heads, bias=True), f = sigmoid(f_proj(x)))
// fused with the tile scan above. CTA per (tile T, batch b): the tensor core
// forms the 128 x H block of z for the tile's tokens (M = 128 tokens, N = H
// padded to 16, K = hidden in chunks of 64 staged by TMA), and the epilogue
// adds the bias, writes z, and scans it exactly as gate_tile_scan_kernel does.
//   warp 0   TMA producer (x chunk 128 x 64, W chunk Hpad x 64; kProjStages stages)
//   warp 1   TMEM allocator and MMA issuer
//   warps 2-5 epilogue (thread = token = TMEM lane), then one head per warp in the scan
constexpr int kProjThreads = 192;
constexpr int kProjStages = 4;

struct ProjParams {
  int B, N, H, Hpad, hidden, nT, Npad, bias_from_j;
  const float* bias;
  float* z;  // [B, N, H] or null
  float* rowloc;
  float* colrec;
  float* tiletot;
  uint32_t* err;
};

__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

__global__ void __launch_bounds__(kProjThreads, 1)
    gate_proj_scan_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                          const ProjParams p) {
  grid_dep_trigger();  // the base scan may start launching (it waits for this kernel's results)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t xb = kTile * 64 * 2;            // x chunk bytes (16 KB)
  const uint32_t wb = (uint32_t)p.Hpad * 64 * 2;  // W chunk bytes (multiple of 2 KB)
  uint8_t* sx = sm;
  uint8_t* sw = sm + kProjStages * xb;
  float(*zs)[kHeadsPerPass + 1] = reinterpret_cast<float(*)[kHeadsPerPass + 1]>(sw + kProjStages * wb);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sw + kProjStages * wb + kTile * (kHeadsPerPass + 1) * 4);
  // bars: FULL[kProjStages], EMPTY[kProjStages], DONE
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kProjStages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int T = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nK = (p.hidden + 63) / 64;
  uint32_t tcols = 32;
  while (tcols < (uint32_t)p.Hpad) tcols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kProjStages; ++s) {
      mbar_init(&bars[s], 1);
      mbar_init(&bars[kProjStages + s], 1);
    }
    mbar_init(&bars[2 * kProjStages], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmap_x);
      tma_prefetch_desc(&tmap_w);
      int issued = 0;
      for (int kc = 0; kc < nK; ++kc) {
        const int st = kc % kProjStages, n = kc / kProjStages;
        if (n > 0 && !mbar_wait(&bars[kProjStages + st], (n - 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC))
          break;
        mbar_arrive_expect_tx(&bars[st], xb + wb);
        tma_load_3d(sx + st * xb, &tmap_x, &bars[st], kc * 64, T * kTile, b);
        tma_load_2d(sw + st * wb, &tmap_w, &bars[st], kc * 64, 0);
        ++issued;
      }
      // every copy issued must land before shared memory is released
      for (int kc = issued - kProjStages < 0 ? 0 : issued - kProjStages; kc < issued; ++kc)
        mbar_wait_drain(&bars[kc % kProjStages], (kc / kProjStages) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kTile, p.Hpad, false, false);
      bool ok = true;
      for (int kc = 0; kc < nK && ok; ++kc) {
        const int st = kc % kProjStages;
        ok = mbar_wait(&bars[st], (kc / kProjStages) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ax = smem_u32(sx + st * xb), aw = smem_u32(sw + st * wb);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_ss(tbase, sdesc_sw128(ax + ks * 32, 16, 1024), sdesc_sw128(aw + ks * 32, 16, 1024), idesc,
                  (kc > 0 || ks > 0) ? 1u : 0u);
        umma_commit(&bars[kProjStages + st]);
      }
      // DONE also follows the retirement of every MMA issued, so TMEM can be freed after it.
      umma_commit(&bars[2 * kProjStages]);
      if (!ok) mbar_wait_drain(&bars[2 * kProjStages], 0);
    }
    __syncwarp();
  } else {
    const int wq = warp & 3;  // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;
    const int t = T * kTile + r;
    const int ew = warp - 2;  // 0..3 within the epilogue warps
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    bool ok = mbar_wait(&bars[2 * kProjStages], 0, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA) && !*abort_flag;
    ok = __all_sync(0xffffffffu, ok);
    if (ok) tc_fence_after();
    for (int h0 = 0; h0 < p.H; h0 += kHeadsPerPass) {
      const int nh = min(kHeadsPerPass, p.H - h0);
      uint32_t acc[32];
      if (ok) {
        if (p.Hpad - h0 >= 32) {
          tmem_ld32(tbase + lane_off + h0, acc);
        } else {
          tmem_ld16(tbase + lane_off + h0, acc);
#pragma unroll
          for (int c = 16; c < 32; ++c) acc[c] = 0u;
        }
        tmem_ld_wait();
      }
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float a = 0.f;  // tokens past the end contribute log f = 0
        if (ok && c < nh && t < p.N) {
          const float zv = __uint_as_float(acc[c]) + p.bias[h0 + c];
          if (p.z) p.z[((size_t)b * p.N + t) * p.H + h0 + c] = zv;
          a = log_sigmoid(zv) * kLog2e;
        }
        zs[r][c] = a;
      }
      named_bar(1, 128);
      if (ok)
        for (int c = ew; c < nh; c += 4)
          scan_head_column(zs, c, lane, (size_t)b * p.H + h0 + c, T, p.N, p.nT, p.Npad, p.bias_from_j, p.rowloc,
                           p.colrec, p.tiletot);
      named_bar(1, 128);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, tcols);
  }
}

// Double-float arithmetic (a value is hi + lo, two fp32 numbers; Knuth's TwoSum and
// Dekker's FastTwoSum): about 48 significant bits from fp32 additions only.
struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF df_add(DF a, DF b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float e = (a.hi - (s - bb)) + (b.hi - bb) + (a.lo + b.lo);
  const float hi = s + e;
  return DF{hi, e - (hi - s)};
}

// One warp, one (b, h): exclusive scan of the tile totals -> base_T, in double-float,
// stored as the hi/lo pair in each column record. The totals of up to 128 tiles are
// loaded before the scan (4 per lane), so the loads overlap.
__device__ __forceinline__ void base_scan_warp(size_t bh, int nT, int lane, const float* __restrict__ tiletot,
                                               float* __restrict__ colrec) {
  DF carry{0.f, 0.f};
  for (int T0 = 0; T0 < nT; T0 += 128) {
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int T = T0 + 32 * q + lane;
      v[q] = T < nT ? tiletot[(size_t)bh * nT + T] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int T = T0 + 32 * q + lane;
      DF incl{v[q], 0.f};
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const DF y{__shfl_up_sync(0xffffffffu, incl.hi, o), __shfl_up_sync(0xffffffffu, incl.lo, o)};
        if (lane >= o) incl = df_add(incl, y);
      }
      // exclusive prefix = carry + (inclusive - own value): the lane below's inclusive sum
      DF below{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
      if (lane == 0) below = DF{0.f, 0.f};
      const DF base = df_add(carry, below);
      if (T < nT) {
        float* rec = colrec + ((size_t)bh * nT + T) * kColRec;
        *reinterpret_cast<float4*>(rec + kTile) = make_float4(base.hi, base.lo, 0.f, 0.f);
      }
      carry = df_add(carry, DF{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)});
    }
  }
}

__global__ void __launch_bounds__(256) gate_base_scan_kernel(int BH, int nT, const float* __restrict__ tiletot,
                                                             float* __restrict__ colrec) {
  grid_dep_trigger();  // the attention kernel may start its prologue
  grid_dep_wait();     // the tile totals of the tile scan
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp < BH) base_scan_warp((size_t)warp, nT, lane, tiletot, colrec);
}

// The forward's fp16 copy of V (the P V operand type) and the base scan in one kernel, run
// as a programmatic dependent of the tile scan: V is converted while the tile scan runs; then
// every warp waits for the tile scan and takes its share of the (b, h) base scans. V (bf16
// bits) goes to fp16 in 16-byte pieces, a grid-stride loop with four loads in flight per
// thread. Every bf16 value of magnitude 2^-14 .. 65280 is exactly an fp16 value; smaller ones
// round to the nearest multiple of 2^-24 (cvt.rn); 65536 and above (infinities included) are
// outside fp16 and set DEV_ERR_RANGE, after the wait (the tile scan, or the memset before the
// fused projection, clears the error word first).
constexpr int kV16Threads = 256;
constexpr int kV16Unroll = 4;

__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 w, uint32_t& vmax) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    out[q] = pack_f16x2(__uint_as_float(in[q] << 16), __uint_as_float(in[q] & 0xFFFF0000u));
    asm("max.u16x2 %0, %0, %1;" : "+r"(vmax) : "r"(in[q] & 0x7FFF7FFFu));
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

__global__ void __launch_bounds__(kV16Threads) gate_base_scan_v16_kernel(int BH, int nT, const float* __restrict__ tiletot,
                                                                          float* __restrict__ colrec,
                                                                          const uint4* __restrict__ v,
                                                                          uint4* __restrict__ v16, size_t pieces,
                                                                          uint32_t* err) {
  grid_dep_trigger();  // the attention kernel may start launching (it waits for this one)
  uint32_t vmax = 0u;
  const size_t stride = (size_t)gridDim.x * kV16Threads;
  size_t i = (size_t)blockIdx.x * kV16Threads + threadIdx.x;
  for (; i + (kV16Unroll - 1) * stride < pieces; i += kV16Unroll * stride) {
    uint4 w[kV16Unroll];
#pragma unroll
    for (int u = 0; u < kV16Unroll; ++u) w[u] = __ldcs(v + i + u * stride);
#pragma unroll
    for (int u = 0; u < kV16Unroll; ++u) v16[i + u * stride] = bf16x8_to_f16x8(w[u], vmax);
  }
  for (; i < pieces; i += stride) v16[i] = bf16x8_to_f16x8(__ldcs(v + i), vmax);
  const bool over = (vmax & 0xFFFFu) >= 0x4780u || (vmax >> 16) >= 0x4780u;
  grid_dep_wait();  // the tile scan's totals and its clearing of the error word
  const int lane = threadIdx.x & 31;
  if (__any_sync(0xffffffffu, over) && lane == 0) atomicOr(err, DEV_ERR_RANGE);
  const int warps = gridDim.x * (kV16Threads / 32);
  for (int w = (int)((blockIdx.x * kV16Threads + threadIdx.x) >> 5); w < BH; w += warps)
    base_scan_warp((size_t)w, nT, lane, tiletot, colrec);
}

// Launches the base scan after a tile-scan kernel: alone, or with the V conversion.
cudaError_t launch_base_scan(const GateLayout& g, const float* tiletot, float* colrec, uint32_t* err,
                             const V16Job* v16, cudaStream_t s) {
  cudaError_t e;
  if (!v16) {
    TraceScope trace("gate_base_scan", s);
    e = launch_dependent(gate_base_scan_kernel, dim3((g.BH + 7) / 8), dim3(256), 0, s, g.BH, g.nT, tiletot, colrec);
  } else {
    const size_t pieces = v16->n / 8;
    size_t blocks = (pieces + kV16Threads * kV16Unroll - 1) / (kV16Threads * kV16Unroll);
    const size_t scan_blocks = ((size_t)g.BH + 7) / 8;
    if (blocks < scan_blocks) blocks = scan_blocks;
    if (blocks > 4096) blocks = 4096;  // grid-stride loops cover the rest
    TraceScope trace("gate_base_scan_v16", s);
    e = launch_dependent(gate_base_scan_v16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kV16Threads), 0, s,
                         g.BH, g.nT, tiletot, colrec, static_cast<const uint4*>(v16->v), static_cast<uint4*>(v16->v16),
                         pieces, err);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

size_t gate_proj_smem_bytes(int H) {
  const int Hpad = (H + 15) / 16 * 16;
  return 1024 + kProjStages * (size_t)(kTile * 64 * 2 + Hpad * 64 * 2) + kTile * (kHeadsPerPass + 1) * 4 +
         (2 * kProjStages + 1) * 8 + 16;
}

cudaError_t launch_gate_proj_scan(const CUtensorMap* maps /* x, W */, const float* bias, int hidden, float* z_out,
                                  int B, int N, int H, int bias_from_j, void* ws, const GateLayout& g,
                                  cudaStream_t s, const V16Job* v16) {
  char* base = static_cast<char*>(ws);
  uint32_t* err = reinterpret_cast<uint32_t*>(base);
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(uint32_t), s);  // each call starts with a clean error word
  if (e != cudaSuccess) return e;
  ProjParams p;
  p.B = B;
  p.N = N;
  p.H = H;
  p.Hpad = (H + 15) / 16 * 16;
  p.hidden = hidden;
  p.nT = g.nT;
  p.Npad = g.Npad;
  p.bias_from_j = bias_from_j;
  p.bias = bias;
  p.z = z_out;
  p.rowloc = reinterpret_cast<float*>(base + g.rowloc);
  p.colrec = reinterpret_cast<float*>(base + g.colrec);
  p.tiletot = reinterpret_cast<float*>(base + g.tiletot);
  p.err = err;
  const size_t smem = gate_proj_smem_bytes(H);
  e = cudaFuncSetAttribute(gate_proj_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  {
    TraceScope trace("gate_proj_scan", s);
    gate_proj_scan_kernel<<<dim3(g.nT, B), kProjThreads, smem, s>>>(maps[0], maps[1], p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_base_scan(g, p.tiletot, p.colrec, err, v16, s);
}

namespace {
// c[b,t,h] = (base_T + local_t) / log2 e, thread per (b, t, h): the output is coalesced over heads.
__global__ void __launch_bounds__(256) gate_cumulative_kernel(int B, int N, int H, int nT, int Npad,
                                                              const float* __restrict__ rowloc,
                                                              const float* __restrict__ colrec, float* __restrict__ c) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)B * N * H) return;
  const int h = (int)(idx % H);
  const long long bt = idx / H;
  const int t = (int)(bt % N), b = (int)(bt / N);
  const size_t bh = (size_t)b * H + h;
  const float* rec = colrec + (bh * nT + t / kTile) * kColRec;
  const double v = (double)rec[kTile] + (double)rec[kTile + 1] + (double)rowloc[bh * Npad + t];
  c[idx] = (float)(v / (double)kLog2e);
}
}  // namespace

cudaError_t launch_gate_cumulative(const void* ws, const GateLayout& g, int B, int N, int H, float* c, cudaStream_t s) {
  const char* base = static_cast<const char*>(ws);
  const float* rowloc = reinterpret_cast<const float*>(base + g.rowloc);
  const float* colrec = reinterpret_cast<const float*>(base + g.colrec);
  const long long n = (long long)B * N * H;
  if (n == 0) return cudaSuccess;
  {
    TraceScope trace("gate_cumulative", s);
    gate_cumulative_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(B, N, H, g.nT, g.Npad, rowloc, colrec, c);
  }
  return cudaGetLastError();
}

cudaError_t launch_gate_scan(const float* z, int B, int N, int H, int bias_from_j, void* ws, const GateLayout& g,
                             cudaStream_t s, const V16Job* v16) {
  char* base = static_cast<char*>(ws);
  float* rowloc = reinterpret_cast<float*>(base + g.rowloc);
  float* colrec = reinterpret_cast<float*>(base + g.colrec);
  float* tiletot = reinterpret_cast<float*>(base + g.tiletot);
  uint32_t* err = reinterpret_cast<uint32_t*>(base);
  dim3 grid(g.nT, B, (H + kTileScanHeads - 1) / kTileScanHeads);
  {
    TraceScope trace("gate_tile_scan", s);
    gate_tile_scan_kernel<<<grid, 256, 0, s>>>(z, B, N, H, g.nT, g.Npad, bias_from_j, rowloc, colrec, tiletot, err);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_base_scan(g, tiletot, colrec, err, v16, s);
}

}  // namespace fox
