// Backward of forget-gated causal attention for sm_103a (bf16 in, fp32
// accumulate). The pages give only the forward ("Forgetting Transformer (FoX)
// Attention" module source, ForgettingAttention.forward); this is the chain
// rule through it:
//   P_ij = exp(x_ij - LSE_i)        (recomputed from the saved LSE)
//   dP_ij = dO_i . v_j,  Delta_i = dO_i . O_i,  dS_ij = P_ij (dP_ij - Delta_i)
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j
//   gate: R_i = sum_j dS_ij and C_j = sum_i dS_ij (row and column sums), then
//   d a_t = sum_{s>=t} (R_s - C_s) under the j+1 convention (+ C_t under j), and
//   dz_t = d a_t * sigmoid(-z_t). R_i is 0 in exact arithmetic, but Delta_i is
//   formed from the bf16-rounded O, so the computed dS has small row sums;
//   including them makes d a_t the sum of the computed dS over the entries that
//   contain a_t, instead of accumulating those row errors along the sequence.
//
// Kernels, in launch order (the gate scan of the forward runs first):
//   (memset)      the dQ accumulator cleared
//   bwd_rows      Delta_i, the row offset rho_i = LSE_i log2 e - l_i; clears the row sums
//   bwd_main      one CTA per (b, h, 128-key tile J) over the query tiles I >= J
//                 (all I when not causal), pipelined over 64-query half-tiles:
//                 S^T = K Q^T, dP^T = V dO^T, dV += P^T dO, dK += dS^T Q and
//                 dQ^T = K^T dS^T on the tensor core (tcgen05, TMEM, two issuing warps),
//                 dQ reduced into an fp32 accumulator; the row sums R_i and column sums
//                 C_j of dS (added into global accumulators)
//   bwd_dq        dQ = scale * accumulator -> bf16
//   bwd_gate      reverse prefix scan of (R - C) (one pass, decoupled look-back) and the sigmoid
//                 chain rule -> dz
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fox_internal.h"
#include "fox_ptx.cuh"

namespace fox {
namespace {


// The fp32 dQ accumulator is blocked so that the 32 queries x 32 channels that one readout
// warp adds at a time form one contiguous 4 KB block: [bh][Npad / 32][D / 32][32][32]
// (query i, channel e of (b, h) at block (bh (Npad / 32) + i / 32) (D / 32) + e / 32,
// float (i % 32) 32 + e % 32 within it).

// ------------------------------------------------------------------ rows
// Delta_i = dO_i . O_i, the row offset rho_i and a cleared row sum for every row (b, i, h)
// with i < N, taken in the [B, N, H] order of O, dO and LSE so that their loads are contiguous:
// a warp takes 8 consecutive rows, D / 8 lanes per row, each lane one 16-byte piece of O and
// of dO per row, all issued before the arithmetic. The padding rows N <= i < Npad of every
// (b, h) get Delta = 0, rho = +inf and R = 0 from a grid-stride loop over the same threads, which
// also clears the gate gradient's status records and ticket counter. (The dQ accumulator is
// zeroed by a memset before this kernel.)
template <int D>
__global__ void __launch_bounds__(256) bwd_rows_kernel(int B, int N, int H, int Npad, const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dO, const float* __restrict__ lse,
                                                      const float* __restrict__ rowloc, float* __restrict__ delta,
                                                      float* __restrict__ rho, float* __restrict__ rowsum,
                                                      int delta_ready, uint4* __restrict__ gstat, size_t gstat16,
                                                      unsigned* __restrict__ ticket) {
  grid_dep_trigger();  // the attention kernel may start its prologue and its K, V loads
  constexpr int LPR = D / 8;          // lanes per row
  constexpr int RPI = 32 / LPR;       // rows per load instruction
  constexpr int LOADS = 8 / RPI;      // loads per lane per tensor
  const int lane = threadIdx.x & 31, sub = lane % LPR, grp = lane / LPR;
  const long long rows = (long long)B * N * H;
  const long long octet = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const long long row0 = octet * 8;
  if (row0 < rows) {
    uint4 ov[LOADS], gv[LOADS];
#pragma unroll
    for (int k = 0; k < LOADS; ++k) {
      const long long row = row0 + k * RPI + grp;
      ov[k] = make_uint4(0u, 0u, 0u, 0u);
      gv[k] = make_uint4(0u, 0u, 0u, 0u);
      if (row < rows) {
        ov[k] = *reinterpret_cast<const uint4*>(o + row * D + sub * 8);
        gv[k] = *reinterpret_cast<const uint4*>(dO + row * D + sub * 8);
      }
    }
    float acc[LOADS];
#pragma unroll
    for (int k = 0; k < LOADS; ++k) {
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov[k]);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv[k]);
      float sum = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(o2[e]), y = __bfloat1622float2(g2[e]);
        sum = fmaf(x.x, y.x, fmaf(x.y, y.y, sum));
      }
      acc[k] = sum;
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1)
#pragma unroll
      for (int k = 0; k < LOADS; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], off);
    // Lane m < 8 finishes row row0 + m: its sum sits in lane (m % RPI) * LPR, slot m / RPI.
    // (B * N * H < 2^31, so the row index and its decode fit 32-bit arithmetic.)
    const int m = lane & 7;
    float dsum = 0.f;
#pragma unroll
    for (int k = 0; k < LOADS; ++k) {
      const float v = __shfl_sync(0xffffffffu, acc[k], (m % RPI) * LPR);
      if (k == m / RPI) dsum = v;
    }
    const long long rowm = row0 + m;
    if (lane < 8 && rowm < rows) {
      const uint32_t row = static_cast<uint32_t>(rowm);
      const uint32_t h = row % (uint32_t)H, t = row / (uint32_t)H;
      const uint32_t i = t % (uint32_t)N, b = t / (uint32_t)N;
      const size_t r = ((size_t)b * H + h) * Npad + i;
      rowsum[r] = 0.f;
      if (!delta_ready) delta[r] = dsum;
      rho[r] = lse[row] * kLog2e - rowloc[r];
    }
  }
  // the gate gradient's look-back status records and ticket counter start at zero
  for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < gstat16; q += (size_t)gridDim.x * blockDim.x)
    gstat[q] = make_uint4(0u, 0u, 0u, 0u);
  if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0u;
  const long long pads = (long long)B * H * (Npad - N);
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < pads; q += (long long)gridDim.x * blockDim.x) {
    const long long bh = q / (Npad - N);
    const size_t r = (size_t)bh * Npad + N + (size_t)(q % (Npad - N));
    rowsum[r] = 0.f;
    delta[r] = 0.f;
    rho[r] = __int_as_float(0x7f800000);
  }
}

// ------------------------------------------------------------------ main
// One CTA per (b, h, 128-key tile J). The query tiles I >= J (every I when not
// causal) are processed as half-tiles g = 0, 1, ... of 64 queries, pipelined
// over two tensor-memory buffers x = g % 2 of 128 columns each:
//   [0, 64)    S^T_g (fp32), then P^T_g and dS^T_g packed bf16: queries 32h .. 32h + 31
//              (h = 0, 1) of P^T in [32h, 32h + 16), of dS^T in [32h + 16, 32h + 32)
//   [64, 128)  dP^T_g (fp32), then dQ^T_g (fp32)
// and the dK, dV accumulators in [256, 256 + 2D). Warp roles (512 threads; warp 15
// has no role and in the causal variant gives its registers to the elementwise warps):
//   warp 13       S^T_g = K Q_g^T once dK / dV of g-2 have read P^T / dS^T out of the
//                 buffer, dP^T_g = V dO_g^T once dQ^T_g-2 has been read out.
//   warp 14       dV += P^T_g dO_g, dK += dS^T_g Q_g, then dQ^T_g = K^T dS^T_g (dS^T from
//                 shared memory) once the elementwise warps are done with g.
//                 (Two issuers measured faster than one: each group of MMAs waits on a
//                 different part of the pipeline.)
//   8 elementwise P^T, dS^T of g (thread = key row x 32 queries); dS^T also goes to a
//     warps        swizzled shared-memory buffer, the B operand of dQ^T.
//   4 readout     copy dQ^T_g out of tensor memory (releasing its columns), the row sums
//     warps       R_g of dS (see below), then add dQ into the fp32 accumulator: 4 KB
//                 blocks staged in shared memory, added in L2 by the bulk-copy engine.
//   1 producer    K_J, V_J once; Q, dO, Delta, rho half-tiles through 3 stages.
// CTAs are scheduled in groups of kHeadGroup heads (see the kernel).
// The gate gradient needs R_i = sum_j dS_ij and C_j = sum_i dS_ij from the same
// values (so that the suffix sums of R - C telescope over one matrix). Causal
// (kExactSums = false): both come from the bf16 dS values; the elementwise warps
// keep C in registers and the readout warps sum the columns of the dS^T buffer in
// shared memory for R, off the elementwise warps' path. Non-causal (kExactSums =
// true): the gate gradient is a small difference of large sums there, so the
// elementwise warps sum the fp32 values: C in registers, R by a shuffle
// reduce-scatter across the warp's 32 keys.
struct BwdKParams {
  int B, N, H, nT, Npad;
  int non_causal;
  float scale2;  // scale * log2 e
  float scale;
  const float* colrec;
  const float* delta;
  const float* rho;
  float* colsum;
  float* rowsum;
  float* dqacc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  uint32_t* err;
  const int* imax;  // tile skipping: last query tile of each key tile ([bh][nT]), or null
};

constexpr int kHalf = 64;        // queries per half-tile
// First tensor-memory column of K step ks (16 queries, 8 packed columns) of P^T in a buffer;
// dS^T's is 16 columns further. Queries 32h .. 32h + 31 sit in [32h, 32h + 32).
__host__ __device__ constexpr uint32_t pds_col(int ks) { return (uint32_t)((ks >> 1) * 32 + (ks & 1) * 8); }
constexpr int kStages = 3;       // Q / dO / Delta / rho stages
constexpr int kBwdThreads = 512; // 16 warps = 4 warpgroups (warp 15 only donates registers)
constexpr int kHeadGroup = 8;    // heads whose key tiles are scheduled together

template <int D>
struct BwdLayoutSmem {
  static constexpr int kTileBytes = kTile * D * 2;  // K or V tile (128 keys)
  static constexpr int kHalfBytes = kHalf * D * 2;  // Q or dO half-tile (64 queries)
  static constexpr int kK = 0;
  static constexpr int kV = kTileBytes;
  static constexpr int kQ = 2 * kTileBytes;                    // kStages stages
  static constexpr int kDO = kQ + kStages * kHalfBytes;        // kStages stages
  static constexpr int kDS = kDO + kStages * kHalfBytes;       // 2 buffers of dS^T: 128 keys x 64 queries bf16
  static constexpr int kZeros = kDS + 2 * 16384;               // 64-wide zero chunk (padding operand, D = 64)
  static constexpr int kZeroBytes = D == 64 ? 16384 : 0;
  static constexpr int kDQ = kZeros + kZeroBytes;              // dQ staging: 4 readout warps x 4 KB
  static constexpr int kDR = kDQ + 16384;                      // kStages x (Delta 256 B, rho 256 B)
  static constexpr int kRec = kDR + kStages * 512;             // column record of tile J (528 B)
  static constexpr int kRsum = kRec + 1024;                    // [3 slots][4 lane quarters][64] row-sum partials
  static constexpr int kCs = kRsum + 3 * 4 * kHalf * 4;        // column-sum exchange, 128 floats
  static constexpr int kBars = kCs + 512;
  static constexpr int kNumBars = 27;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = (kBytes + 1024) > 118784 ? (kBytes + 1024) : 118784;
};

enum BwdBar {
  BB_KV = 0,
  BB_FULL = 1,    // +stage (3): Q, dO, Delta, rho of a half-tile landed
  BB_EMPTY = 4,   // +stage (3): the MMAs reading that stage retired
  BB_SDP = 7,     // +buffer (2): S^T and dP^T in tensor memory
  BB_PDS = 9,     // +buffer (2): P^T, dS^T written (one arrival per elementwise warp)
  BB_DQ = 11,     // +buffer (2): dQ^T in tensor memory
  BB_DQFREE = 13, // +buffer (2): dQ^T read out of tensor memory (one arrival per readout warp)
  BB_FINAL = 15,  // every MMA of warp 14 retired (the last dK / dV included)
  BB_BDONE = 16,  // every MMA of warp 13 retired
  BB_KVD = 17,    // +buffer (2): dV, dK of the buffer's half-tile retired (P^T, dS^T read)
  BB_DSFREE = 19, // +4 buffer + lane quarter (8): that quarter's rows of the dS^T smem buffer
                  // have been summed, and the dQ block staged over them read by the bulk engine
};

__device__ __forceinline__ void sts_f32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
// c + the low (even column) or high bf16 half of a packed word, widened exactly to fp32
// (one mixed-precision add: the same result as widening first and adding in fp32).
__device__ __forceinline__ float add_bf_lo(float c, uint32_t w) {
  float d;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.bf16 %0, l, %2;\n\t}" : "=f"(d) : "r"(w), "f"(c));
  return d;
}
__device__ __forceinline__ float add_bf_hi(float c, uint32_t w) {
  float d;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.bf16 %0, h, %2;\n\t}" : "=f"(d) : "r"(w), "f"(c));
  return d;
}

// P^T and dS^T for 32 queries of this thread's key row (columns c0 .. c0+31 of
// the half-tile). S^T / dP^T values come from tensor memory columns [c0, c0+32)
// and [64+c0, 64+c0+32); packed bf16 P^T goes to [c0, c0+16) and dS^T to
// [c0+16, c0+32) (over the S^T values just loaded), and the packed dS^T words are left in dd for the caller to
// store into the swizzled smem buffer. The column sum (csum) is accumulated from the
// bf16 values, or from the fp32 ones with kExactSums, which also leaves this lane
// quarter's row-sum partials in rsum.
template <bool kDiag, bool kExactSums>
__device__ __forceinline__ void pds32(uint32_t tX, int c0, int qoff, int jr, float scale2, float cj, const float* dlt,
                                      const float* rh, const uint32_t* rs, const uint32_t* rp, float* rsum,
                                      float& csum, uint32_t* dd) {
  uint32_t pp[16];
  float v[32];  // fp32 dS of this row's 32 queries
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    const float4 r4 = lds_f4(rh + c0 + 4 * e4);
    const float4 d4 = lds_f4(dlt + c0 + 4 * e4);
    const float rr[4] = {r4.x, r4.y, r4.z, r4.w};
    const float dl[4] = {d4.x, d4.y, d4.z, d4.w};
    float pv[4];
#pragma unroll
    for (int e = 0; e < 4; e += 2) {  // element pairs in packed fp32
      const int c = 4 * e4 + e;
      float2 x = fsub2(ffma2(make_float2(__uint_as_float(rs[c]), __uint_as_float(rs[c + 1])),
                             make_float2(scale2, scale2), make_float2(cj, cj)),
                       make_float2(rr[e], rr[e + 1]));
      if (kDiag && qoff + c0 + c < jr) x.x = -INFINITY;  // query before key: masked
      if (kDiag && qoff + c0 + c + 1 < jr) x.y = -INFINITY;
      pv[e] = ex2_approx(x.x);
      pv[e + 1] = ex2_approx(x.y);
      const float2 t = fmul2(make_float2(pv[e], pv[e + 1]),
                             fsub2(make_float2(__uint_as_float(rp[c]), __uint_as_float(rp[c + 1])),
                                   make_float2(dl[e], dl[e + 1])));
      v[c] = t.x;
      v[c + 1] = t.y;
      if (kExactSums) {
        csum += v[c];
        csum += v[c + 1];
      }
    }
    pp[2 * e4] = pack_bf16x2(pv[0], pv[1]);
    pp[2 * e4 + 1] = pack_bf16x2(pv[2], pv[3]);
    dd[2 * e4] = pack_bf16x2(v[4 * e4], v[4 * e4 + 1]);
    dd[2 * e4 + 1] = pack_bf16x2(v[4 * e4 + 2], v[4 * e4 + 3]);
    if (!kExactSums)  // the column sum of the bf16 values the readout's row sums also use
      csum = add_bf_hi(add_bf_lo(add_bf_hi(add_bf_lo(csum, dd[2 * e4]), dd[2 * e4]), dd[2 * e4 + 1]), dd[2 * e4 + 1]);
  }
  tmem_st16(tX + c0, pp);
  tmem_st16(tX + c0 + 16, dd);
  if (kExactSums) {
    // Row sums over this warp's 32 keys: reduce-scatter across the lanes (five halving
    // rounds), after which lane l holds query c0 + l's sum.
    const int lane = jr & 31;
#pragma unroll
    for (int half = 16; half >= 1; half >>= 1) {
      const bool upper = (lane & half) != 0;
#pragma unroll
      for (int k = 0; k < half; ++k) {
        const float send = upper ? v[k] : v[k + half];
        const float keep = upper ? v[k + half] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, half);
      }
    }
    rsum[c0 + lane] = v[0];  // this lane quarter's partial; the readout adds the four quarters
  }
}

// Work order: groups of kHeadGroup heads, and within a group the key tiles from J = 0
// (the most query tiles) down, the group's heads interleaved. The CTAs resident at once
// then share few heads, whose Q / dO streams stay in L2.
__device__ __forceinline__ void bwd_work_item(int idx, int BH, int nT, int& J, int& bh) {
  const int full = (BH / kHeadGroup) * kHeadGroup * nT;  // CTAs in complete groups
  const int gsize = idx < full ? kHeadGroup : BH % kHeadGroup;
  const int gbase = idx < full ? (idx / (kHeadGroup * nT)) * kHeadGroup : BH - BH % kHeadGroup;
  const int r = idx < full ? idx % (kHeadGroup * nT) : idx - full;
  J = r / gsize;
  bh = gbase + r % gsize;
}

template <int D, bool kExactSums>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fox_attn_bwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                        const __grid_constant__ CUtensorMap tmap_dk, const __grid_constant__ CUtensorMap tmap_dv,
                        const BwdKParams p) {
  using L = BwdLayoutSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  int J, bh;
  bwd_work_item(static_cast<int>(blockIdx.x), BH, p.nT, J, bh);
  const int b = bh / p.H, h = bh % p.H;
  // Half-tiles of 64 queries: causal, query tiles I = J .. nT-1 (.. imax(J) with tile
  // skipping); non-causal, all of them.
  const bool causal = !p.non_causal;
  const int I_first = causal ? J : 0;
  const int I_last = p.imax ? p.imax[(size_t)bh * p.nT + J] : p.nT - 1;
  const int G = 2 * (I_last - I_first + 1);
  // The elementwise and readout warps read the half-tile count from shared memory at
  // each iteration instead of holding it in a register (their register budget is full).
  volatile int* G_shared = reinterpret_cast<volatile int*>(sm + L::kMisc + 8);

  // The producer thread initialises the barriers and starts the K and V loads (the caller's
  // inputs) at once, so that they overlap the set-up below.
  if (warp == 12 && lane == 0) {
    mbar_init(&bars[BB_KV], 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[BB_FULL + s], 1);
      mbar_init(&bars[BB_EMPTY + s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars[BB_SDP + x], 1);
      mbar_init(&bars[BB_PDS + x], 8);
      mbar_init(&bars[BB_DQ + x], 1);
      mbar_init(&bars[BB_DQFREE + x], 4);
      mbar_init(&bars[BB_KVD + x], 1);
      for (int w = 0; w < 4; ++w) mbar_init(&bars[BB_DSFREE + x * 4 + w], 1);
    }
    mbar_init(&bars[BB_FINAL], 1);
    mbar_init(&bars[BB_BDONE], 1);
    *abort_flag = 0;
    *G_shared = G;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
    tma_prefetch_desc(&tmap_do);
    mbar_arrive_expect_tx(&bars[BB_KV], 2 * L::kTileBytes + kColRec * 4);
    for (int x = 0; x < D / 64; ++x) {
      tma_load_4d(sm + L::kK + x * 16384, &tmap_k, &bars[BB_KV], x * 64, h, J * kTile, b);
      tma_load_4d(sm + L::kV + x * 16384, &tmap_v, &bars[BB_KV], x * 64, h, J * kTile, b);
    }
  }
  if (warp == 13) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (D == 64) {
    // Constant operand: a 64-wide chunk of zeros, the upper M half of K^T when D = 64.
    uint32_t* zw = reinterpret_cast<uint32_t*>(sm + L::kZeros);
    for (int e = threadIdx.x; e < 16384 / 4; e += blockDim.x) zw[e] = 0u;
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // Registers per warpgroup (launched at 128 each, 65536 in total): the producer and MMA
  // warpgroup needs few, the readout warpgroup fewer than 128, and the elementwise
  // warpgroups take the rest (256 x 144 + 128 x 112 + 128 x 112 = 65536).
  // (The non-causal variant, with the fp32 row-sum shuffles in the elementwise warps,
  // measured faster without the rebalancing.)
  if (!kExactSums) {
    if (warp >= 12)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 112;" ::: "memory");
    else if (warp >= 8)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 112;" ::: "memory");
    else
      asm volatile("setmaxnreg.inc.sync.aligned.u32 144;" ::: "memory");
  }

  // This kernel may start while the row kernel before it still runs (launch_dependent): the K and
  // V tiles are the caller's input and load at once (above); everything the earlier kernels wrote
  // (the column record, Delta, rho, the cleared row sums) is read only after grid_dep_wait().
  grid_dep_wait();
  grid_dep_trigger();  // the dQ conversion may start launching (it waits for this kernel's results)

  if (warp == 12) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      constexpr uint32_t hb = L::kHalfBytes;
      bulk_load(sm + L::kRec, p.colrec + ((size_t)bh * p.nT + J) * kColRec, kColRec * 4, &bars[BB_KV]);
      int fills[kStages] = {};
      for (int g = 0; g < G; ++g) {
        const int st = g % kStages;
        const int q0 = I_first * kTile + g * kHalf;
        if (g >= kStages &&
            !mbar_wait(&bars[BB_EMPTY + st], ((g / kStages) - 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC))
          break;
        mbar_arrive_expect_tx(&bars[BB_FULL + st], 2 * hb + 512);
        for (int x = 0; x < D / 64; ++x) {
          tma_load_4d(sm + L::kQ + st * hb + x * 8192, &tmap_q, &bars[BB_FULL + st], x * 64, h, q0, b);
          tma_load_4d(sm + L::kDO + st * hb + x * 8192, &tmap_do, &bars[BB_FULL + st], x * 64, h, q0, b);
        }
        const size_t roff = (size_t)bh * p.Npad + q0;
        bulk_load(sm + L::kDR + st * 512, p.delta + roff, 256, &bars[BB_FULL + st]);
        bulk_load(sm + L::kDR + st * 512 + 256, p.rho + roff, 256, &bars[BB_FULL + st]);
        ++fills[st];
      }
      mbar_wait_drain(&bars[BB_KV], 0);
      for (int st = 0; st < kStages; ++st)
        if (fills[st] > 0) mbar_wait_drain(&bars[BB_FULL + st], (fills[st] - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 13 || warp == 14) {
    // ----------------------------------------------------------- MMA issuers
    if (lane == 0) {
      constexpr uint32_t hb = L::kHalfBytes;
      constexpr uint32_t idSP = idesc_bf16(128, kHalf, false, false);  // S^T, dP^T: M keys, N queries
      constexpr uint32_t idKV = idesc_bf16(128, D, false, true);       // dV, dK: A from TMEM, B MN-major
      constexpr uint32_t idQ = idesc_bf16(128, kHalf, true, true);     // dQ^T: A = K^T (MN-major), B = dS (MN-major)
      const uint32_t sK = smem_u32(sm + L::kK), sQ = smem_u32(sm + L::kQ), sdO = smem_u32(sm + L::kDO);
      bool ok = mbar_wait(&bars[BB_KV], 0, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
      // Operand descriptors: the key-tile operands (K, V, K^T) are computed once; those of a
      // half-tile stage or dS^T buffer are its base descriptor plus offset / 16, formed before
      // each group so that the group's MMAs issue back to back. (Shared-memory addresses stay
      // below 2^18, so the 14-bit start-address field of base + offset never carries.)
      if (warp == 13) {
        const uint32_t sV = smem_u32(sm + L::kV);
        uint64_t aK[D / 16], aV[D / 16];
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t koff = (ks >> 2) * 16384 + (ks & 3) * 32;  // K / V tile: 128-row chunks
          aK[ks] = sdesc_sw128(sK + koff, 16, 1024);
          aV[ks] = sdesc_sw128(sV + koff, 16, 1024);
        }
        const uint64_t bQ0 = sdesc_sw128(sQ, 16, 1024), bdO0 = sdesc_sw128(sdO, 16, 1024);
        for (int g = 0; g < G && ok; ++g) {
          const int x = g & 1, st = g % kStages;
          const uint32_t tX = tbase + 128 * x;
          uint64_t bQ[D / 16], bdO[D / 16];
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t qoff = st * hb + (ks >> 2) * 8192 + (ks & 3) * 32;  // Q / dO half-tile: 64-row chunks
            bQ[ks] = desc_plus(bQ0, qoff);
            bdO[ks] = desc_plus(bdO0, qoff);
          }
          ok = mbar_wait(&bars[BB_FULL + st], (g / kStages) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
          // S^T_g overwrites P^T / dS^T of g-2, read by warp 14's dV / dK of g-2. (For g < 2 the
          // parity is 1: the phase before a fresh barrier's first counts as complete, so the
          // wait returns at once and the issue path has no branch on g.)
          if (ok) ok = mbar_wait(&bars[BB_KVD + x], ((g - 2) >> 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) umma_ss(tX, aK[ks], bQ[ks], idSP, ks > 0);
          // dP^T_g overwrites dQ^T of g-2, which the readout warps must have copied out
          ok = mbar_wait(&bars[BB_DQFREE + x], ((g - 2) >> 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) umma_ss(tX + 64, aV[ks], bdO[ks], idSP, ks > 0);
          umma_commit(&bars[BB_SDP + x]);
        }
      } else {
        const uint32_t tdK = tbase + 256, tdV = tbase + 256 + D;
        const uint32_t sdS = smem_u32(sm + L::kDS), sZeros = smem_u32(sm + L::kZeros);
        // A = K^T: M = d channels (MN-major 64-wide chunks 16 KB apart; D = 64 pads the upper half with zeros)
        const uint32_t kt_lbo = D == 128 ? 16384u : sZeros - sK;
        uint64_t aKt[kTile / 16];
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) aKt[ks] = sdesc_sw128(sK + ks * 2048, kt_lbo, 1024);
        const uint64_t bdO0 = sdesc_sw128(sdO, 8192, 1024), bQ0 = sdesc_sw128(sQ, 8192, 1024);
        const uint64_t bdS0 = sdesc_sw128(sdS, 16384, 1024);
        for (int g = 0; g < G && ok; ++g) {
          const int x = g & 1, st = g % kStages;
          const uint32_t tX = tbase + 128 * x;
          uint64_t bdO[kHalf / 16], bQ[kHalf / 16], bdS[kTile / 16];
#pragma unroll
          for (int ks = 0; ks < kHalf / 16; ++ks) {
            bdO[ks] = desc_plus(bdO0, st * hb + ks * 2048);
            bQ[ks] = desc_plus(bQ0, st * hb + ks * 2048);
          }
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks) bdS[ks] = desc_plus(bdS0, x * 16384 + ks * 2048);
          ok = mbar_wait(&bars[BB_PDS + x], (g >> 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < kHalf / 16; ++ks)  // dV += P^T dO (K = 64 queries)
            umma_ts(tdV, tX + pds_col(ks), bdO[ks], idKV, (g > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
          for (int ks = 0; ks < kHalf / 16; ++ks)  // dK += dS^T Q
            umma_ts(tdK, tX + pds_col(ks) + 16, bQ[ks], idKV, (g > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&bars[BB_KVD + x]);
          umma_commit(&bars[BB_EMPTY + st]);
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)  // dQ^T = K^T dS^T (K = 128 keys) over [64,128)
            umma_ss(tX + 64, aKt[ks], bdS[ks], idQ, ks > 0);
          umma_commit(&bars[BB_DQ + x]);
        }
      }
      // Every MMA this thread issued must retire before tensor memory is freed; for warp 14
      // this is also the end of the dK / dV accumulation.
      uint64_t* done = &bars[warp == 14 ? BB_FINAL : BB_BDONE];
      umma_commit(done);
      mbar_wait_drain(done, 0);
    }
    __syncwarp();
  } else if (warp == 15) {
    // no role
  } else if (warp >= 8) {
    // ------------------------------------------- R, C, dQ^T readout
    const int wq = warp & 3;
    const int ln = wq * 32 + lane;  // TMEM lane: output channel of dQ^T; key row of C
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    float* rpart = reinterpret_cast<float*>(sm + L::kRsum);  // [2][4][64] (causal) or [3][4][64] partials
    const uint32_t stage = smem_u32(sm + L::kDQ) + (uint32_t)wq * 4096u;
    float* dq_bh = p.dqacc + (size_t)bh * p.Npad * D;  // this (b, h)'s slab of the blocked accumulator
    bool ok = true, staged = false;
    for (int g = 0; g < *G_shared && ok; ++g) {
      const int x = g & 1;
      const uint32_t tX = tbase + 128 * x + lane_off;
      const int q0 = I_first * kTile + g * kHalf;
      // The first dQ block of g - 1 went over this warp's rows of the dS^T buffer of g - 1. Once
      // the bulk engine has read it (by now it normally has), the elementwise warps of this lane
      // quarter may write those rows for g + 1. (Waiting for the read right after issuing it
      // stalled them.)
      if (staged && lane == 0) {
        bulk_wait_read<1>();
        mbar_arrive(&bars[BB_DSFREE + (x ^ 1) * 4 + wq]);
      }
      staged = false;
      ok = mbar_wait(&bars[BB_PDS + x], (g >> 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC);
      // dQ^T first, so that dP^T of g + 2 can follow as early as possible; the row sums below
      // read the dS^T buffer, which the elementwise warps overwrite only after DSFREE.
      ok = ok && mbar_wait(&bars[BB_DQ + x], (g >> 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      uint32_t r0[32], r1[32], rv = 0;
      if (ok) {  // a failed wait still reaches the readout barrier below, where all four warps stop
        tmem_ld32(tX + 64, r0);
        tmem_ld32(tX + 96, r1);
        tmem_ld_wait();
      }
      if (kExactSums && wq < 2) {  // R of the half-tile's 64 queries: the four lane quarters' partials (slot g % 3)
        const float* rs = rpart + (g % 3) * 4 * kHalf + ln;
        rv = __float_as_uint((rs[0] + rs[kHalf]) + (rs[2 * kHalf] + rs[3 * kHalf]));
      }
      tc_fence_before();
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&bars[BB_DQFREE + x]);  // the warp's dQ^T is in registers
      // At d = 64 each readout warp adds its own key quarter's row sums (four times the atomics,
      // no meeting of the four warps per half-tile: 0.176 -> 0.167 ms at B4 H16 N2048); at
      // d = 128 one warp adds the four quarters' partials after the meeting (the other way
      // measured 2 % slower there).
      constexpr bool kOwnRowSums = D == 64 && !kExactSums;
      if (kOwnRowSums && !ok) break;
      float r_lo = 0.f, r_hi = 0.f;  // causal: R of queries 2 lane, 2 lane + 1 over this warp's 32 keys
      if (!kExactSums && ok) {
        const uint32_t sdx = smem_u32(sm + L::kDS + x * 16384);
        // R: queries 2 lane and 2 lane + 1 (piece lane / 4, word lane % 4) over keys 32 wq .. 32 wq + 31
        const uint32_t wofs = (uint32_t)(lane & 3) * 4u;
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
          const int jr = wq * 32 + k;
          const uint32_t w = lds_u32(sdx + (uint32_t)jr * 128u + (uint32_t)(((lane >> 2) ^ (jr & 7)) << 4) + wofs);
          r_lo = add_bf_lo(r_lo, w);
          r_hi = add_bf_hi(r_hi, w);
        }
        if (kOwnRowSums) {
          atomicAdd(p.rowsum + (size_t)bh * p.Npad + q0 + 2 * lane, r_lo);
          atomicAdd(p.rowsum + (size_t)bh * p.Npad + q0 + 2 * lane + 1, r_hi);
          __syncwarp();  // every lane's loads of these rows come before the block staged over them
        } else {
          reinterpret_cast<float2*>(rpart + ((g & 1) * 4 + wq) * kHalf)[lane] = make_float2(r_lo, r_hi);
        }
      }
      // The four readout warps meet once per half-tile (and agree whether to stop).
      if (!kOwnRowSums && named_bar_any(6, 128, !ok)) {
        ok = false;
        break;
      }
      if (!kExactSums && !kOwnRowSums && wq == 0) {  // R of the half-tile's 64 queries: the four key quarters
        const float2* rp2 = reinterpret_cast<const float2*>(rpart + (g & 1) * 4 * kHalf);
        const float2 a = rp2[lane], bq = rp2[kHalf / 2 + lane], c = rp2[kHalf + lane], d2 = rp2[3 * kHalf / 2 + lane];
        atomicAdd(p.rowsum + (size_t)bh * p.Npad + q0 + 2 * lane, (a.x + bq.x) + (c.x + d2.x));
        atomicAdd(p.rowsum + (size_t)bh * p.Npad + q0 + 2 * lane + 1, (a.y + bq.y) + (c.y + d2.y));
      }
      if (kExactSums && wq < 2) atomicAdd(p.rowsum + (size_t)bh * p.Npad + q0 + ln, __uint_as_float(rv));
      if (wq * 32 < D) {
        // dQ[q0 + i][32 wq + lane] += dQ^T[32 wq + lane][i], as two blocks of 32 queries x 32
        // channels staged in shared memory and added into the accumulator by the bulk-copy
        // engine. The first block goes over this warp's own rows of the dS^T buffer x (the
        // dQ^T MMA and this warp's row sums are done with them), the second into the warp's
        // staging block once the block staged there for g - 1 has been read.
        const uint32_t stage_a = smem_u32(sm + L::kDS + x * 16384) + (uint32_t)wq * 4096u;
        float* blk = dq_bh + ((size_t)(q0 >> 5) * (D / 32) + wq) * 1024;
#pragma unroll
        for (int i = 0; i < 32; ++i) sts_f32(stage_a + (uint32_t)(i * 32 + lane) * 4u, r0[i]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          bulk_reduce_add_f32(blk, stage_a, 4096);
          bulk_commit_group();
          bulk_wait_read<1>();
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 32; ++i) sts_f32(stage + (uint32_t)(i * 32 + lane) * 4u, r1[i]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          bulk_reduce_add_f32(blk + (D / 32) * 1024, stage, 4096);
          bulk_commit_group();
        }
      }
      staged = true;
    }
    // The bulk engine must have read every staged block before shared memory is released;
    // the additions themselves complete before the kernel does.
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  } else {
    // ------------------------------------------------------ P^T, dS^T, epilogue
    const int wq = warp & 3, ch = warp >> 2;
    const int jr = wq * 32 + lane;  // TMEM lane = key row of S^T, dP^T, dK, dV
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float* rec = reinterpret_cast<const float*>(sm + L::kRec);
    const float* recs = p.colrec + (size_t)bh * p.nT * kColRec;
    float csum = 0.f;  // C_j for key j = jr over this warp's queries of every half-tile
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[BB_KV], 0, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA));
    const float kap = ok ? rec[jr] : 0.f;
    const float baseJ_hi = ok ? rec[kTile] : 0.f, baseJ_lo = ok ? rec[kTile + 1] : 0.f;
    for (int g = 0; g < *G_shared && ok; ++g) {
      const int x = g & 1, st = g % kStages;
      const int I = I_first + (g >> 1), half = g & 1;
      const uint32_t tX = tbase + 128 * x + lane_off;
      const uint32_t sds_row = smem_u32(sm + L::kDS + x * 16384) + (uint32_t)jr * 128u;
      const float* dlt = reinterpret_cast<const float*>(sm + L::kDR + st * 512);
      const float* rh = dlt + kHalf;
      float* rsum = reinterpret_cast<float*>(sm + L::kRsum) + ((g % 3) * 4 + wq) * kHalf;
      const float baseI_hi = recs[(size_t)I * kColRec + kTile], baseI_lo = recs[(size_t)I * kColRec + kTile + 1];
      ok = mbar_wait(&bars[BB_SDP + x], (g >> 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA) &&
           mbar_wait(&bars[BB_FULL + st], (g / kStages) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
      ok = __all_sync(0xffffffffu, ok);  // tcgen05 loads / stores below are warp-collective
      tc_fence_after();
      // x_ji (log2 units, minus the row offset) = scale2 * S^T_ji - kappa_j + (base_I - base_J) - rho_i
      const float cj = ((baseI_hi - baseJ_hi) + (baseI_lo - baseJ_lo)) - kap;
      const int c0 = ch * 32;
      const int qoff = half * kHalf;  // query offset of this half inside tile I (for the diagonal mask)
      // Each warp packs P^T and dS^T of its 32 queries over the S^T columns it has just
      // loaded ([c0, c0 + 32)), so the two warps of a lane quarter never touch each other's
      // columns and need no barrier between them.
      if (!ok) break;
      uint32_t rs[32], rp[32];
      tmem_ld32(tX + c0, rs);
      tmem_ld32(tX + 64 + c0, rp);
      tmem_ld_wait();
      uint32_t dd[16];
      if (causal && I == J)
        pds32<true, kExactSums>(tX, c0, qoff, jr, p.scale2, cj, dlt, rh, rs, rp, rsum, csum, dd);
      else
        pds32<false, kExactSums>(tX, c0, qoff, jr, p.scale2, cj, dlt, rh, rs, rp, rsum, csum, dd);
      // The readout warp of this lane quarter staged dQ of g - 2 over these rows of the dS^T
      // buffer; the bulk engine must have read it.
      if (g >= 2 && !__all_sync(0xffffffffu, mbar_wait(&bars[BB_DSFREE + x * 4 + wq], ((g - 2) >> 1) & 1, abort_flag,
                                                       p.err, DEV_ERR_TIMEOUT_SYNC)))
        break;
#pragma unroll
      for (int pc = 0; pc < 4; ++pc) {
        const int piece = (c0 >> 3) + pc;  // 16-byte piece = 8 queries
        sts_v4(sds_row + (uint32_t)((piece ^ (jr & 7)) << 4), dd[4 * pc], dd[4 * pc + 1], dd[4 * pc + 2],
               dd[4 * pc + 3]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();  // the warp's stores are ordered before the one arrival that speaks for it
      if (lane == 0) mbar_arrive(&bars[BB_PDS + x]);
    }
    const int j = J * kTile + jr;
    {
      // Column sums: half ch = 1 hands its partial to ch = 0 through shared memory.
      float* cs = reinterpret_cast<float*>(sm + L::kCs);
      if (ch == 1) cs[jr] = csum;
      named_bar_any(5, 256, false);
      if (ok && ch == 0) p.colsum[(size_t)bh * p.Npad + j] = csum + cs[jr];
    }
    // dK, dV epilogue: scaled, rounded to bf16 and staged in the shared memory of the K and V
    // tiles in the 128-byte-swizzled layout of the output tensor maps, then written by tensor
    // stores, whole 128-byte row pieces per 64-channel box (a thread's own 16-byte stores to
    // rows H d apart had cost about 2 us per CTA). The stores clip rows past N.
    // dK and dV are complete once the dV / dK MMAs of the last half-tile have retired. The V
    // tile is free then; the K tile only once that half-tile's dQ^T, which reads K^T, has too.
    {
      const int gl = *G_shared - 1;
      if (ok) ok = mbar_wait(&bars[BB_KVD + (gl & 1)], (gl >> 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      constexpr int kCols = D / 2;
      const int e0 = ch * kCols;
      const uint32_t tdK = tbase + 256 + lane_off, tdV = tbase + 256 + D + lane_off;
      // Two 32-column loads in flight per wait.
#pragma unroll
      for (int which = 0; which < 2; ++which) {  // dV, then dK
        if (which == 1) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars[BB_FINAL], 0, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA));
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t src = (which == 1 ? tdK : tdV) + e0;
        const float mul = which == 1 ? p.scale : 1.f;
        // row jr of the 64-channel box that holds channel e0 (16 KB per box, 128 B per row)
        const uint32_t row = smem_u32(sm + (which == 1 ? L::kK : L::kV) + (e0 / 64) * 16384) + (uint32_t)jr * 128u;
#pragma unroll
        for (int c = 0; c < kCols; c += 64) {
          uint32_t r[2][32];
          tmem_ld32(src + c, r[0]);
          if (c + 32 < kCols) tmem_ld32(src + c + 32, r[1]);
          tmem_ld_wait();
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            if (c + 32 * hh >= kCols) continue;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int piece = ((e0 % 64) + c + 32 * hh) / 8 + q4;  // 16-byte piece of the 128-byte row
              sts_v4(row + (uint32_t)((piece ^ (jr & 7)) << 4),
                     pack_bf16x2(__uint_as_float(r[hh][8 * q4 + 0]) * mul, __uint_as_float(r[hh][8 * q4 + 1]) * mul),
                     pack_bf16x2(__uint_as_float(r[hh][8 * q4 + 2]) * mul, __uint_as_float(r[hh][8 * q4 + 3]) * mul),
                     pack_bf16x2(__uint_as_float(r[hh][8 * q4 + 4]) * mul, __uint_as_float(r[hh][8 * q4 + 5]) * mul),
                     pack_bf16x2(__uint_as_float(r[hh][8 * q4 + 6]) * mul, __uint_as_float(r[hh][8 * q4 + 7]) * mul));
            }
          }
        }
      }
      fence_proxy_async_smem();
    }
    // The 256 elementwise threads meet (and agree whether every one of them staged its row);
    // one thread then issues the stores and waits until the bulk engine has read shared memory.
    if (!named_bar_any(4, 256, !ok) && threadIdx.x == 0) {
#pragma unroll
      for (int box = 0; box < D / 64; ++box) {
        tma_store_4d(&tmap_dk, sm + L::kK + box * 16384, box * 64, h, J * kTile, b);
        tma_store_4d(&tmap_dv, sm + L::kV + box * 16384, box * 64, h, J * kTile, b);
      }
      bulk_commit_group();
      bulk_wait_read<0>();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ---------------------------------------------------------------- dQ out
// One warp per 4 KB block of the accumulator (32 queries x 32 channels of one (b, h)): the
// block is read as eight contiguous 512-byte pieces, all issued first; each query's 32
// channels go out as one 64-byte piece of its dQ row.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(int B, int N, int H, int Npad, float scale,
                                                    const float* __restrict__ dqacc, __nv_bfloat16* __restrict__ dq) {
  grid_dep_trigger();  // the gate gradient may start launching
  grid_dep_wait();     // the dQ accumulator of the attention kernel
  const long long blk = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long nblk = (long long)B * H * (Npad / 32) * (D / 32);
  if (blk >= nblk) return;
  const int cb = (int)(blk % (D / 32));           // channel block
  const long long qbk = blk / (D / 32);
  const int qblk = (int)(qbk % (Npad / 32));      // query block
  const long long bh = qbk / (Npad / 32);
  const int b = (int)(bh / H), h = (int)(bh % H);
  const float4* src = reinterpret_cast<const float4*>(dqacc) + (size_t)blk * 256;  // 4 KB = 256 float4
  float4 v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) v[k] = src[k * 32 + lane];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int q = 4 * k + (lane >> 3), i = qblk * 32 + q;  // query of this piece
    if (i >= N) continue;
    __nv_bfloat16* dst = dq + (((size_t)b * N + i) * H + h) * D + cb * 32 + (lane & 7) * 4;
    uint2 w;
    w.x = pack_bf16x2(v[k].x * scale, v[k].y * scale);
    w.y = pack_bf16x2(v[k].z * scale, v[k].w * scale);
    *reinterpret_cast<uint2*>(dst) = w;
  }
}

// ---------------------------------------------------------- gate backward
// d a_t = sum_{s>=t} (R_s - C_s) (+ C_t when bias_from_j), dz_t = d a_t sigmoid(-z_t): a suffix
// scan along the sequence per (b, h), in one pass over R, C, z and dz (16 bytes per token and
// head) with a decoupled look-back across 128-token blocks:
//   - CTAs take tickets from a counter in the order blocks k = nT-1, nT-2, ..., 0 (the batches
//     and head groups of one k together), so every block a CTA waits on has already started;
//   - a CTA (block k, batch b, 32 heads) loads its R and C rows (coalesced along the tokens),
//     forms each head's block total of R - C and publishes it as the block's aggregate;
//   - it then sums the aggregates of the later blocks k+1, k+2, ... until it meets one whose
//     inclusive suffix sum is already published (32 blocks per round, one per lane), adds its
//     own total and publishes its inclusive suffix sum, in double-float (fp32 hi/lo pairs
//     with TwoSum: about 48 bits; fp64 runs at a small fraction of the fp32 rate here);
//   - the carry and the block-local suffix scan give d a, and dz is written along the heads
//     (coalesced [B, N, H] accesses).
// Each published value shares one 64-bit word with its ready flag (flag in the high half), so
// a reader that sees the flag sees the value. The status words and the ticket counter must be
// zero before the launch. A wait that runs out (one second) sets DEV_ERR_TIMEOUT_SYNC and the
// block goes on with what it has, so nothing waits forever.
// (hi, lo) += (bhi, blo) in double-float: Knuth's TwoSum on the high parts, the low parts
// added in fp32, renormalised with Dekker's FastTwoSum.
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float bhi, float blo) {
  const float s = hi + bhi;
  const float bb = s - hi;
  const float e = (hi - (s - bb)) + (bhi - bb) + (lo + blo);
  hi = s + e;
  lo = e - (hi - s);
}

// Status record of one (b h, block): the block total (aggregate) and the inclusive suffix sum
// (hi, lo), each 64-bit word = (1 << 32) | float bits once published.
struct GateStat {
  unsigned long long agg, inc_hi, inc_lo, pad;
};
__device__ __forceinline__ unsigned long long stat_word(float v) {
  return (1ull << 32) | static_cast<unsigned long long>(__float_as_uint(v));
}
__device__ __forceinline__ void stat_store(unsigned long long* w, float v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(w), "l"(stat_word(v)) : "memory");
}
__device__ __forceinline__ unsigned long long stat_load(const unsigned long long* w) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(w) : "memory");
  return v;
}

constexpr int kGateHeads = 32;     // heads per gate-gradient CTA
constexpr int kGateThreads = 512;  // 16 warps, two heads each
constexpr int kLookLanes = 16;     // lanes (blocks read per round) of one head's look-back

// Three CTAs per SM (40 registers, no spills): more blocks' loads in flight, since each CTA runs its
// loads, look-back and stores in sequence (two per SM: 190 us on B64 H32 N16384, three: 173 us).
__global__ void __launch_bounds__(kGateThreads, 3) gate_grad_kernel(int B, int N, int H, int nT, int stride,
                                                                 int bias_from_j, const float* __restrict__ colsum,
                                                                 const float* __restrict__ rowsum,
                                                                 const float* __restrict__ z, float* __restrict__ dz,
                                                                 GateStat* __restrict__ stat, unsigned* ticket,
                                                                 uint32_t* err) {
  constexpr int kPer = kTile * kGateHeads / kGateThreads;  // elements per thread of the (token, head) tile
  __shared__ float xs[kGateHeads][kTile + 1];               // [head][token]: R - C, then d a
  __shared__ float cs[kGateHeads][kTile + 1];               // C (bias_from_j)
  __shared__ unsigned s_ticket;
  grid_dep_wait();  // R and C of the attention kernel; the ticket and status records the row kernel cleared
  if (threadIdx.x == 0) s_ticket = atomicAdd(ticket, 1u);
  __syncthreads();
  const int HG = (H + kGateHeads - 1) / kGateHeads;
  const int per_k = B * HG;
  const int k = nT - 1 - static_cast<int>(s_ticket) / per_k;
  const int r = static_cast<int>(s_ticket) % per_k;
  const int b = r / HG, h0 = (r % HG) * kGateHeads;
  const int nh = min(kGateHeads, H - h0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = k * kTile;
  // All loads first: R and C rows (thread e covers token e % 128 of head e / 128, rows contiguous
  // per head) and z along the heads (token e / 32, head e % 32), for the dz pass at the end.
  float zv[kPer];
  {
    float rv[kPer], cv[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = threadIdx.x + u * kGateThreads, hh = e / kTile, t = e % kTile;
      const bool in = hh < nh && t0 + t < N;
      const size_t off = ((size_t)b * H + h0 + hh) * stride + t0 + t;
      rv[u] = in ? rowsum[off] : 0.f;
      cv[u] = in ? colsum[off] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = threadIdx.x + u * kGateThreads, t = e >> 5, hh = e & 31;
      zv[u] = (hh < nh && t0 + t < N) ? z[((size_t)b * N + t0 + t) * H + h0 + hh] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = threadIdx.x + u * kGateThreads, hh = e / kTile, t = e % kTile;
      xs[hh][t] = rv[u] - cv[u];
      cs[hh][t] = cv[u];
    }
  }
  __syncthreads();
  // Heads 2 warp and 2 warp + 1: lane holds tokens 4 lane .. 4 lane + 3 of each.
  float v[2][4], lane_later[2], lane_run[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int hh = 2 * warp + q;
    float run = 0.f;
#pragma unroll
    for (int e = 3; e >= 0; --e) {
      run += hh < nh ? xs[hh][4 * lane + e] : 0.f;
      v[q][e] = run;
    }
    float later = run;  // inclusive suffix over lanes lane .. 31 of the lane totals
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, later, o);
      if (lane + o < 32) later += y;
    }
    lane_later[q] = later;
    lane_run[q] = run;
    // lane 0's suffix is the block total: publish it (the last block's is also its inclusive sum)
    if (lane == 0 && hh < nh) {
      GateStat* st = stat + ((size_t)b * H + h0 + hh) * nT + k;
      stat_store(&st->agg, later);
      if (k == nT - 1) {
        stat_store(&st->inc_lo, 0.f);
        stat_store(&st->inc_hi, later);
      }
    }
  }
  // Look-back of both heads at once: lanes 16 g .. 16 g + 15 read blocks j0 + (lane % 16) of head
  // 2 warp + g, summing aggregates up to the first block whose inclusive sum is published.
  const int g = lane >> 4, gl = lane & 15;
  const int hh_g = 2 * warp + g;
  const GateStat* row = stat + ((size_t)b * H + h0 + min(hh_g, nh - 1)) * nT;
  float chi = 0.f, clo = 0.f;  // the carry of head hh_g (valid in every lane of the group)
  bool done = hh_g >= nh || k == nT - 1;
  int j0 = k + 1;
  bool timed_out = false;
  const uint64_t t_start = globaltimer_ns();
  for (uint32_t it = 0; __any_sync(0xffffffffu, !done); ++it) {
    const int j = j0 + gl;
    unsigned long long ih = 0, il = 0, ag = 0;
    if (!done && j < nT) {
      ih = stat_load(&row[j].inc_hi);
      il = stat_load(&row[j].inc_lo);
      ag = stat_load(&row[j].agg);
    }
    const bool have_inc = (ih >> 32) != 0 && (il >> 32) != 0;
    const bool have_agg = (ag >> 32) != 0;
    const unsigned inc_all = __ballot_sync(0xffffffffu, !done && j < nT && have_inc);
    const unsigned rdy_all = __ballot_sync(0xffffffffu, j >= nT || have_inc || have_agg);
    const unsigned inc = (inc_all >> (16 * g)) & 0xFFFFu, rdy = (rdy_all >> (16 * g)) & 0xFFFFu;
    // lanes up to the group's first inclusive one (or all 16) must be ready
    const unsigned need = inc ? ((inc & (0u - inc)) * 2u - 1u) : 0xFFFFu;
    const bool resolved = !done && (rdy & need) == need;
    float hi = 0.f, lo = 0.f;
    if (resolved && j < nT && ((need >> gl) & 1u)) {
      const bool first_inc = inc != 0 && gl == __ffs(inc) - 1;
      hi = __uint_as_float(static_cast<uint32_t>(first_inc ? ih : ag));
      lo = first_inc ? __uint_as_float(static_cast<uint32_t>(il)) : 0.f;
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1)  // within the 16-lane group
      two_sum_acc(hi, lo, __shfl_xor_sync(0xffffffffu, hi, o), __shfl_xor_sync(0xffffffffu, lo, o));
    if (resolved) {
      two_sum_acc(chi, clo, hi, lo);
      j0 += kLookLanes;
      done = inc != 0 || j0 >= nT;
    }
    if ((it & 31u) == 31u && __any_sync(0xffffffffu, globaltimer_ns() - t_start > FOX_WAIT_TIMEOUT_NS)) {
      timed_out = timed_out || !done;
      break;
    }
  }
  if (timed_out && gl == 0 && err) atomicOr(err, DEV_ERR_TIMEOUT_SYNC);
  const float carry_g = chi + clo;
  // the block totals of both heads (lane 0's suffixes), for the group of each
  const float tot0 = __shfl_sync(0xffffffffu, lane_later[0], 0), tot1 = __shfl_sync(0xffffffffu, lane_later[1], 0);
  if (gl == 0 && hh_g < nh && k < nT - 1) {
    // inclusive = carry + this block's total
    float ihi = chi, ilo = clo;
    two_sum_acc(ihi, ilo, g ? tot1 : tot0, 0.f);
    GateStat* st = stat + ((size_t)b * H + h0 + hh_g) * nT + k;
    stat_store(&st->inc_lo, ilo);
    stat_store(&st->inc_hi, ihi);
  }
  // d a inside the block: this lane's suffix, the later lanes, then the later blocks
  const float carry_h[2] = {__shfl_sync(0xffffffffu, carry_g, 0), __shfl_sync(0xffffffffu, carry_g, 16)};
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int hh = 2 * warp + q;
    if (hh >= nh) break;
    const float base = lane_later[q] - lane_run[q] + carry_h[q];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = 4 * lane + e;
      xs[hh][t] = bias_from_j ? v[q][e] + base + cs[hh][t] : v[q][e] + base;
    }
  }
  __syncthreads();
  // dz over (token, head), heads fastest: the [B, N, H] stores run along the heads
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = threadIdx.x + u * kGateThreads, t = e >> 5, hh = e & 31;
    if (hh < nh && t0 + t < N)
      dz[((size_t)b * N + t0 + t) * H + h0 + hh] = xs[hh][t] / (1.f + expf(zv[u]));  // d a sigmoid(-z)
  }
}

// ------------------------------------------------ gate backward, one sequence per CTA
// The same d a and dz when there are enough (b, head group) sequences to occupy every SM
// (B ceil(H / 4) >= the SM count): a CTA takes one batch b and kSeqHeads = 4 heads and walks
// their whole sequence from the last 128-token block to the first, carrying the suffix sum
// in double-float from block to block, so no CTA waits on another. Warp 0 streams R, C (rows
// of the 4 heads, [head][token] in shared memory) and z ([token][head]) through kSeqStages
// stages by TMA; warps 1-4 take 32 tokens each, one token per lane with all 4 heads in
// registers, so every shared-memory access of theirs is conflict-free. A consumer warp frees
// the stage as soon as its values are in registers and forms sigmoid(-z) at once, off the
// scan's path. Per block: x = R - C, the suffix sum within the warp by shuffles and across the
// four warps through shared memory (fp32, at most 128 terms, as in the look-back kernel),
// d a = that + the carry (+ C under the j convention), dz = d a sigmoid(-z), stored by each lane
// as one 16-byte piece of its token's dz row; then the carry takes the block total. Tokens past
// N arrive as zeros and their dz is not stored. Four heads per CTA (the least whose z row piece,
// 16 bytes, a tensor copy can move) give the most CTAs, and the number of independent sequences
// is what sets the rate: each CTA spends about 1 us per block. Large synthetic (B64 H32 N16384,
// 512 CTAs): 131 us. Measured slower: 8 heads per CTA (171 us; with two 4-head groups of four
// warps and dz through shared memory, whole 32-byte sectors, 140 us); dz written back by
// tensor stores (165 us at 8 heads); 6, 8 or 12 stages instead of 4 (135, 140, 236 us);
// sigmoid(-z) by the fast intrinsics gained 2 %; splitting each sequence between two CTAs (the
// earlier part first summing the later part's blocks, R and C only) 196 us: a block costs
// about the same whether it is summed or fully processed; the consumer warps taking two, three
// or four blocks per round (one meeting of the four warps per round, 4 to 9 stages) 136-144 us:
// the rounds of the consumer warps do not set the rate either; stages of two or four blocks (R and
// C rows read 1 or 2 KB at a time) 139-144 us. Timing copies: without the z loads 131 us; without
// the dz stores (and so most of the arithmetic) 118 us, the R and C loads alone at 2.3 TB/s.
constexpr int kSeqHeads = 4;
constexpr int kSeqStages = 4;
constexpr int kSeqConsumers = 4;  // warps of 32 tokens
constexpr int kSeqThreads = 32 * (1 + kSeqConsumers);
constexpr int kSeqBoxBytes = kTile * kSeqHeads * 4;                 // one of R, C, z per stage: 2 KB
constexpr int kSeqStageBytes = 3 * kSeqBoxBytes;  // R, C, z
constexpr int kSeqSmem = kSeqStages * kSeqStageBytes + 1024 + 512;  // stages, alignment slack, barriers etc.

__global__ void __launch_bounds__(kSeqThreads) gate_grad_seq_kernel(
    const __grid_constant__ CUtensorMap map_r, const __grid_constant__ CUtensorMap map_c,
    const __grid_constant__ CUtensorMap map_z, float* __restrict__ dz, int N, int H, int nT, int bias_from_j,
    uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSeqStages * kSeqStageBytes);  // FULL[S], FREE[S]
  float* wt = reinterpret_cast<float*>(bars + 2 * kSeqStages);                      // [2][consumers][heads]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(wt + 2 * kSeqConsumers * kSeqHeads);
  const int HG = (H + kSeqHeads - 1) / kSeqHeads;
  const int b = static_cast<int>(blockIdx.x) / HG, h0 = (static_cast<int>(blockIdx.x) % HG) * kSeqHeads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto buf = [&](int s, int which) { return reinterpret_cast<float*>(sm + s * kSeqStageBytes + which * kSeqBoxBytes); };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSeqStages; ++s) {
      mbar_init(&bars[s], 1);
      mbar_init(&bars[kSeqStages + s], kSeqConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dep_wait();  // R and C of the attention kernel

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&map_r);
      tma_prefetch_desc(&map_c);
      tma_prefetch_desc(&map_z);
      int loaded = 0;
      for (int i = 0; i < nT; ++i) {  // block k = nT - 1 - i into stage i % S
        const int s = i % kSeqStages, n = i / kSeqStages;
        if (n > 0 && !mbar_wait(&bars[kSeqStages + s], (n - 1) & 1, abort_flag, err, DEV_ERR_TIMEOUT_SYNC)) break;
        const int k = nT - 1 - i;
        mbar_arrive_expect_tx(&bars[s], 3 * kSeqBoxBytes);
        tma_load_3d(buf(s, 0), &map_r, &bars[s], k * kTile, h0, b);
        tma_load_3d(buf(s, 1), &map_c, &bars[s], k * kTile, h0, b);
        tma_load_3d(buf(s, 2), &map_z, &bars[s], h0, k * kTile, b);
        loaded = i + 1;
      }
      // every load issued must have landed before shared memory is released
      for (int i = loaded > kSeqStages ? loaded - kSeqStages : 0; i < loaded; ++i)
        mbar_wait_drain(&bars[i % kSeqStages], (i / kSeqStages) & 1);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int t = cw * 32 + lane;  // token within the block
    float chi[kSeqHeads], clo[kSeqHeads];
#pragma unroll
    for (int h = 0; h < kSeqHeads; ++h) chi[h] = clo[h] = 0.f;
    for (int i = 0; i < nT; ++i) {
      const int s = i % kSeqStages, n = i / kSeqStages;
      const bool ok = mbar_wait(&bars[s], n & 1, abort_flag, err, DEV_ERR_TIMEOUT_TMA);
      const float* r = buf(s, 0);
      const float* c = buf(s, 1);
      const float* zz = buf(s, 2);
      float x[kSeqHeads], cv[kSeqHeads], sg[kSeqHeads], zv[kSeqHeads];
#pragma unroll
      for (int q = 0; q < kSeqHeads; q += 4) {
        const float4 z4 = *reinterpret_cast<const float4*>(zz + t * kSeqHeads + q);
        zv[q] = z4.x, zv[q + 1] = z4.y, zv[q + 2] = z4.z, zv[q + 3] = z4.w;
      }
#pragma unroll
      for (int h = 0; h < kSeqHeads; ++h) {
        cv[h] = c[h * kTile + t];
        x[h] = r[h * kTile + t] - cv[h];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kSeqStages + s]);  // R, C and z of the stage are in registers
#pragma unroll
      for (int h = 0; h < kSeqHeads; ++h) sg[h] = 1.f / (1.f + expf(zv[h]));  // sigmoid(-z)
      // inclusive suffix over the warp's tokens t .. 32 cw + 31
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int h = 0; h < kSeqHeads; ++h) {
          const float y = __shfl_down_sync(0xffffffffu, x[h], o);
          if (lane + o < 32) x[h] += y;
        }
      }
      float* wb = wt + (i & 1) * kSeqConsumers * kSeqHeads;
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < kSeqHeads; ++h) wb[cw * kSeqHeads + h] = x[h];  // the warp's total
      }
      // the warp totals are visible; a failed wait anywhere stops all four warps together
      if (named_bar_any(1, 32 * kSeqConsumers, !ok)) break;
      float out[kSeqHeads];
#pragma unroll
      for (int h = 0; h < kSeqHeads; ++h) {
        float later = 0.f, total = 0.f;
#pragma unroll
        for (int w = 0; w < kSeqConsumers; ++w) {
          const float v = wb[w * kSeqHeads + h];
          total += v;
          if (w > cw) later += v;
        }
        const float da = x[h] + later + (chi[h] + clo[h]);
        out[h] = (bias_from_j ? da + cv[h] : da) * sg[h];
        two_sum_acc(chi[h], clo[h], total, 0.f);
      }
      const int tg = (nT - 1 - i) * kTile + t;
      if (tg < N) {
#pragma unroll
        for (int q = 0; q < kSeqHeads; q += 4)
          *reinterpret_cast<float4*>(dz + ((size_t)b * N + tg) * H + h0 + q) =
              make_float4(out[q], out[q + 1], out[q + 2], out[q + 3]);
      }
    }
  }
}

template <int D>
cudaError_t launch_bwd_d(const AttnBwdArgs& a, const GateLayout& g, const BwdLayout& w, const CUtensorMap* maps,
                         cudaStream_t s) {
  using L = BwdLayoutSmem<D>;
  static_assert(L::kAlloc <= 232448, "shared memory budget");
  const float* rowloc = reinterpret_cast<const float*>(a.ws + g.rowloc);
  const float* colrec = reinterpret_cast<const float*>(a.ws + g.colrec);
  float* delta = reinterpret_cast<float*>(a.ws + w.delta);
  float* rho = reinterpret_cast<float*>(a.ws + w.rho);
  float* colsum = reinterpret_cast<float*>(a.ws + w.colsum);
  float* rowsum = reinterpret_cast<float*>(a.ws + w.rowsum);
  float* dqacc = reinterpret_cast<float*>(a.ws + w.dqacc);
  uint32_t* err = reinterpret_cast<uint32_t*>(a.ws);
  const long long rows = (long long)a.B * g.Npad * a.H;
  {
    TraceScope trace("dq_zero", s);
    if (cudaMemsetAsync(dqacc, 0, (size_t)rows * D * sizeof(float), s) != cudaSuccess) return cudaGetLastError();
  }
  {
    TraceScope trace("bwd_rows", s);
    const long long octets = ((long long)a.B * a.N * a.H + 7) / 8;  // 8 rows per warp, 8 warps per block
    bwd_rows_kernel<D><<<(unsigned)((octets + 7) / 8), 256, 0, s>>>(
        a.B, a.N, a.H, g.Npad, static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dO), a.lse,
        rowloc, delta, rho, rowsum, a.delta_ready, reinterpret_cast<uint4*>(a.ws + w.gstat),
        kGateStatBytes * (size_t)g.BH * g.nT / 16, reinterpret_cast<unsigned*>(a.ws + kTicketOffset));
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kernel = a.non_causal ? fox_attn_bwd_kernel<D, true> : fox_attn_bwd_kernel<D, false>;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  BwdKParams p;
  p.B = a.B;
  p.N = a.N;
  p.H = a.H;
  p.nT = g.nT;
  p.Npad = g.Npad;
  p.non_causal = a.non_causal;
  p.scale = a.scale;
  p.scale2 = a.scale * kLog2e;
  p.colrec = colrec;
  p.delta = delta;
  p.rho = rho;
  p.colsum = colsum;
  p.rowsum = rowsum;
  p.dqacc = dqacc;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.err = err;
  p.imax = a.imax;
  const long long blocks = (long long)g.nT * g.BH;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  {
    TraceScope trace("attn_bwd", s);
    e = launch_dependent(kernel, dim3((unsigned)blocks), dim3(kBwdThreads), L::kAlloc, s, maps[0], maps[1], maps[2],
                         maps[3], maps[4], maps[5], p);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long dblocks = (long long)a.B * a.H * (g.Npad / 32) * (D / 32);  // 4 KB accumulator blocks
  {
    TraceScope trace("bwd_dq", s);
    e = launch_dependent(bwd_dq_kernel<D>, dim3((unsigned)((dblocks + 7) / 8)), dim3(256), 0, s, a.B, a.N, a.H,
                         g.Npad, a.scale, (const float*)dqacc, static_cast<__nv_bfloat16*>(a.dq));
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_gate_bwd(a.B, a.N, a.H, g.Npad, a.bias_from_j, colsum, rowsum, a.z, a.dz, a.ws + w.gstat,
                         reinterpret_cast<unsigned*>(a.ws + kTicketOffset), err, s);
}

}  // namespace

bool gate_bwd_streams(int B, int N, int H, int stride, const float* colsum, const float* rowsum, const float* z,
                      const float* dz) {
  if (B <= 0 || N <= 0 || H <= 0) return false;
  // tensor-map rules: 16-byte aligned bases and 16-byte multiples for every row pitch
  auto a16 = [](const void* ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; };
  if (!a16(colsum) || !a16(rowsum) || !a16(z) || !a16(dz) || stride % 4 != 0 || H % 4 != 0) return false;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  return (long long)B * ((H + kSeqHeads - 1) / kSeqHeads) >= sms;
}

cudaError_t launch_gate_bwd(int B, int N, int H, int stride, int bias_from_j, const float* colsum,
                            const float* rowsum, const float* z, float* dz, void* stat, unsigned* ticket,
                            uint32_t* err, cudaStream_t s) {
  const long long BH = (long long)B * H;
  if (BH == 0 || N == 0) return cudaSuccess;
  if (gate_bwd_streams(B, N, H, stride, colsum, rowsum, z, dz)) {
    // R, C as [B][H][stride] rows (box 128 tokens x 4 heads); z as [B][N][H] (box 4 heads x 128 tokens)
    CUtensorMap maps[3];
    if (!make_f32_3d_map(&maps[0], rowsum, N, H, B, (uint64_t)stride * 4, (uint64_t)stride * H * 4, kTile, kSeqHeads) ||
        !make_f32_3d_map(&maps[1], colsum, N, H, B, (uint64_t)stride * 4, (uint64_t)stride * H * 4, kTile, kSeqHeads) ||
        !make_f32_3d_map(&maps[2], z, H, N, B, (uint64_t)H * 4, (uint64_t)N * H * 4, kSeqHeads, kTile))
      return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gate_grad_seq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSeqSmem);
    if (e != cudaSuccess) return e;
    const long long ctas = (long long)B * ((H + kSeqHeads - 1) / kSeqHeads);
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int nT = (N + kTile - 1) / kTile;
    TraceScope trace("bwd_gate", s);
    e = launch_dependent(gate_grad_seq_kernel, dim3((unsigned)ctas), dim3(kSeqThreads), kSeqSmem, s, maps[0], maps[1],
                         maps[2], dz, N, H, nT, bias_from_j, err);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  const int nT = (N + kTile - 1) / kTile;
  const long long ctas = (long long)nT * B * ((H + kGateHeads - 1) / kGateHeads);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  {
    TraceScope trace("bwd_gate", s);
    const cudaError_t e = launch_dependent(gate_grad_kernel, dim3((unsigned)ctas), dim3(kGateThreads), 0, s, B, N, H,
                                           nT, stride, bias_from_j, colsum, rowsum, z, dz,
                                           static_cast<GateStat*>(stat), ticket, err);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const AttnBwdArgs& a, const GateLayout& g, const BwdLayout& w, const CUtensorMap* maps,
                            cudaStream_t s) {
  if (a.d == 64) return launch_bwd_d<64>(a, g, w, maps, s);
  if (a.d == 128) return launch_bwd_d<128>(a, g, w, maps, s);
  return cudaErrorInvalidValue;
}

}  // namespace fox
