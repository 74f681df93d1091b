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
//   bwd_rows      Delta_i, the row offset rho_i = LSE_i log2 e - l_i, zeroes the dQ accumulator
//   bwd_main      one CTA per (b, h, 128-key tile J), looping over query tiles I >= J:
//                 S^T = K Q^T and dP^T = V dO^T (tcgen05, TMEM), P^T and dS^T in registers,
//                 dV += P^T dO, dK += dS^T Q (A from TMEM), dQ_I = dS K (A from smem)
//                 reduced into the fp32 accumulator, and the column sums C_j kept in
//                 registers (the CTA owns every column j of its tile, no atomics). The
//                 dQ MMA of the last 64 output columns is widened by 16 columns whose
//                 B operand is a column of ones, so it also yields this tile's part of
//                 the row sums R_i (one atomic add per row and key tile).
//   bwd_dq        dQ = scale * accumulator -> bf16
//   bwd_gate      reverse prefix scan of C and the sigmoid chain rule -> dz
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fox_internal.h"
#include "fox_ptx.cuh"

namespace fox {
namespace {

constexpr int kBwdThreads = 320;
constexpr int kRecBytes = kColRec * 4;  // 528

// ------------------------------------------------------------------ rows
// One warp per (b, i, h) with i in [0, Npad).
template <int D>
__global__ void __launch_bounds__(256) bwd_rows_kernel(int B, int N, int H, int Npad, const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dO, const float* __restrict__ lse,
                                                      const float* __restrict__ rowloc, float* __restrict__ delta,
                                                      float* __restrict__ rho, float* __restrict__ rowsum,
                                                      float* __restrict__ dqacc) {
  constexpr int E = D / 32;  // elements per lane
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)B * Npad * H;
  if (row >= rows) return;
  const int h = (int)(row % H);
  const long long bi = row / H;
  const int i = (int)(bi % Npad);
  const int b = (int)(bi / Npad);
  const size_t bh = (size_t)b * H + h;
  float acc = 0.f;
  if (i < N) {
    const size_t base = (((size_t)b * N + i) * H + h) * D + lane * E;
    if (E == 4) {
      const uint2 ov = *reinterpret_cast<const uint2*>(o + base);
      const uint2 gv = *reinterpret_cast<const uint2*>(dO + base);
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float2 a = __bfloat1622float2(o2[e]), c = __bfloat1622float2(g2[e]);
        acc = fmaf(a.x, c.x, fmaf(a.y, c.y, acc));
      }
    } else {
      const __nv_bfloat162 ov = *reinterpret_cast<const __nv_bfloat162*>(o + base);
      const __nv_bfloat162 gv = *reinterpret_cast<const __nv_bfloat162*>(dO + base);
      const float2 a = __bfloat1622float2(ov), c = __bfloat1622float2(gv);
      acc = fmaf(a.x, c.x, a.y * c.y);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  float* dq = dqacc + (bh * Npad + i) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) dq[e] = 0.f;
  if (lane == 0) {
    rowsum[bh * Npad + i] = 0.f;
    delta[bh * Npad + i] = i < N ? acc : 0.f;
    rho[bh * Npad + i] =
        i < N ? lse[((size_t)b * N + i) * H + h] * kLog2e - rowloc[bh * Npad + i] : __int_as_float(0x7f800000);
  }
}

// ------------------------------------------------------------------ main
struct BwdKParams {
  int B, N, H, nT, Npad;
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
};

template <int D>
struct BwdLayoutSmem {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kTileBytes;
  static constexpr int kQ = 2 * kTileBytes;   // 2 stages
  static constexpr int kDO = 4 * kTileBytes;  // 1 stage
  static constexpr int kDS = 5 * kTileBytes;  // dS^T, 128 keys x 128 queries bf16 (32 KB)
  static constexpr int kRec = kDS + 32768;    // column record of tile J (528 B)
  static constexpr int kDR = kRec + 1024;     // Delta_I (512 B) then rho_I (512 B)
  static constexpr int kCs = kDR + 1024;      // column-sum exchange, 128 floats
  static constexpr int kOnes = kCs + 1024;    // 1024-aligned: 128 rows x 64 bf16, column 0 = 1, rest 0 (MN-major B)
  static constexpr int kBars = kOnes + 16384;
  static constexpr int kNumBars = 12;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = (kBytes + 1024) > 118784 ? (kBytes + 1024) : 118784;
};

enum BwdBar {
  BB_KV = 0,
  BB_QFULL = 1,   // +stage
  BB_QEMPTY = 3,  // +stage
  BB_DOFULL = 5,
  BB_DOEMPTY = 6,
  BB_SDP = 7,     // S^T and dP^T in TMEM
  BB_PDS = 8,     // P^T, dS^T written (count 256)
  BB_DQ = 9,      // dQ pair result in TMEM
  BB_DQFREE = 10, // dQ read out (count 256)
  BB_FINAL = 11,  // last dK/dV MMAs retired
};

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}
__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// P^T and dS^T for 32 queries (columns q0 .. q0+31 of this thread's key row).
// Writes packed bf16 pairs into 16 TMEM columns of each region and the dS^T
// row piece into the swizzled shared-memory tile; accumulates the column sum.
template <bool kDiag>
__device__ __forceinline__ void pds_chunk(uint32_t tA, uint32_t tB, int q0, int jr, float scale2, float cj,
                                          const float* dlt, const float* rh, uint32_t sds_row, float& csum) {
  uint32_t rs[32], rp[32];
  tmem_ld32(tA + q0, rs);
  tmem_ld32(tB + q0, rp);
  tmem_ld_wait();
  uint32_t pp[16], dd[16];
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    const float4 r4 = lds_f4(rh + q0 + 4 * e4);
    const float4 d4 = lds_f4(dlt + q0 + 4 * e4);
    const float rr[4] = {r4.x, r4.y, r4.z, r4.w};
    const float dl[4] = {d4.x, d4.y, d4.z, d4.w};
    float pv[4], dv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = 4 * e4 + e;
      float x = fmaf(__uint_as_float(rs[c]), scale2, cj) - rr[e];
      if (kDiag && q0 + c < jr) x = -INFINITY;
      pv[e] = ex2_approx(x);
      dv[e] = pv[e] * (__uint_as_float(rp[c]) - dl[e]);
    }
    pp[2 * e4] = pack_bf16x2(pv[0], pv[1]);
    pp[2 * e4 + 1] = pack_bf16x2(pv[2], pv[3]);
    dd[2 * e4] = pack_bf16x2(dv[0], dv[1]);
    dd[2 * e4 + 1] = pack_bf16x2(dv[2], dv[3]);
    // Column sums of the bf16-rounded dS, the same values the row sums R_i are
    // formed from on the tensor core, so sum_s (R_s - C_s) over a suffix is the
    // sum of one matrix's entries and carries no rounding drift along the sequence.
    csum += (__uint_as_float(dd[2 * e4] << 16) + __uint_as_float(dd[2 * e4] & 0xffff0000u)) +
            (__uint_as_float(dd[2 * e4 + 1] << 16) + __uint_as_float(dd[2 * e4 + 1] & 0xffff0000u));
  }
  // packed column of query pair (2c, 2c+1) is c = q / 2
  tmem_st16(tA + (q0 >> 1), pp);
  tmem_st16(tB + (q0 >> 1), dd);
  // dS^T row jr: queries q0 .. q0+31 are 16-byte pieces (q0 % 64) / 8 .. +3 of chunk q0 / 64
  const uint32_t row = sds_row + (uint32_t)(q0 >> 6) * 16384u;
#pragma unroll
  for (int pc = 0; pc < 4; ++pc) {
    const int piece = ((q0 & 63) >> 3) + pc;
    sts_v4(row + (uint32_t)((piece ^ (jr & 7)) << 4), dd[4 * pc], dd[4 * pc + 1], dd[4 * pc + 2], dd[4 * pc + 3]);
  }
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fox_attn_bwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                        const BwdKParams p) {
  using L = BwdLayoutSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  const int J = static_cast<int>(blockIdx.x) / BH;  // key tile; J = 0 has the most query tiles
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int b = bh / p.H, h = bh % p.H;
  const int nI = p.nT - J;

  if (threadIdx.x == 0) {
    mbar_init(&bars[BB_KV], 1);
    mbar_init(&bars[BB_QFULL + 0], 1);
    mbar_init(&bars[BB_QFULL + 1], 1);
    mbar_init(&bars[BB_QEMPTY + 0], 1);
    mbar_init(&bars[BB_QEMPTY + 1], 1);
    mbar_init(&bars[BB_DOFULL], 1);
    mbar_init(&bars[BB_DOEMPTY], 1);
    mbar_init(&bars[BB_SDP], 1);
    mbar_init(&bars[BB_PDS], 256);
    mbar_init(&bars[BB_DQ], 1);
    mbar_init(&bars[BB_DQFREE], 256);
    mbar_init(&bars[BB_FINAL], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  {
    // Ones column for the row sums: element (row r, column c) of this 64-wide MN-major
    // chunk sits in 16-byte piece (c / 8) ^ (r % 8) of row r; column 0 is 1.0, the rest 0.
    uint32_t* ones = reinterpret_cast<uint32_t*>(sm + L::kOnes);
    for (int e = threadIdx.x; e < 16384 / 4; e += blockDim.x) {
      const int r = e >> 5, word = e & 31;  // 32 words of 4 bytes per 128-byte row
      ones[e] = (word == ((r & 7) << 2)) ? 0x3F80u : 0u;  // bf16 1.0 in the low half = column 0
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // TMEM columns: A = S^T / P^T [0,128), B = dP^T / dS^T [128,256), dK [256, 256+D), dV [256+D, 256+2D).
  // dQ of a pair: D = 128 -> e in [0,64) at B+64, e in [64,128) at A+64;  D = 64 -> A+64.

  if (warp == 8) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
      tma_prefetch_desc(&tmap_do);
      constexpr uint32_t tb = L::kTileBytes;
      mbar_arrive_expect_tx(&bars[BB_KV], 2 * tb + kRecBytes);
      for (int x = 0; x < D / 64; ++x) {
        tma_load_4d(sm + L::kK + x * 16384, &tmap_k, &bars[BB_KV], x * 64, h, J * kTile, b);
        tma_load_4d(sm + L::kV + x * 16384, &tmap_v, &bars[BB_KV], x * 64, h, J * kTile, b);
      }
      bulk_load(sm + L::kRec, p.colrec + ((size_t)bh * p.nT + J) * kColRec, kRecBytes, &bars[BB_KV]);
      int qfills[2] = {0, 0}, dofills = 0;
      for (int u = 0; u < nI; ++u) {
        const int I = J + u, st = u & 1;
        if (u >= 2 && !mbar_wait(&bars[BB_QEMPTY + st], ((u >> 1) - 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC))
          break;
        mbar_arrive_expect_tx(&bars[BB_QFULL + st], tb);
        for (int x = 0; x < D / 64; ++x)
          tma_load_4d(sm + L::kQ + st * tb + x * 16384, &tmap_q, &bars[BB_QFULL + st], x * 64, h, I * kTile, b);
        ++qfills[st];
        if (u >= 1 && !mbar_wait(&bars[BB_DOEMPTY], (u - 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC)) break;
        mbar_arrive_expect_tx(&bars[BB_DOFULL], tb + 1024);
        for (int x = 0; x < D / 64; ++x)
          tma_load_4d(sm + L::kDO + x * 16384, &tmap_do, &bars[BB_DOFULL], x * 64, h, I * kTile, b);
        const size_t roff = (size_t)bh * p.Npad + (size_t)I * kTile;
        bulk_load(sm + L::kDR, p.delta + roff, 512, &bars[BB_DOFULL]);
        bulk_load(sm + L::kDR + 512, p.rho + roff, 512, &bars[BB_DOFULL]);
        ++dofills;
      }
      mbar_wait_drain(&bars[BB_KV], 0);
      for (int st = 0; st < 2; ++st)
        if (qfills[st] > 0) mbar_wait_drain(&bars[BB_QFULL + st], (qfills[st] - 1) & 1);
      if (dofills > 0) mbar_wait_drain(&bars[BB_DOFULL], (dofills - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t tb = L::kTileBytes;
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idKV = idesc_bf16(128, D, false, true);
      constexpr uint32_t idQ = idesc_bf16(128, 64, true, true);
      constexpr uint32_t idQR = idesc_bf16(128, 80, true, true);
      const uint32_t tA = tbase, tB = tbase + 128, tdK = tbase + 256, tdV = tbase + 256 + D;
      const uint32_t sK = smem_u32(sm + L::kK), sV = smem_u32(sm + L::kV), sQ = smem_u32(sm + L::kQ);
      const uint32_t sdO = smem_u32(sm + L::kDO), sdS = smem_u32(sm + L::kDS), sOnes = smem_u32(sm + L::kOnes);
      bool ok = mbar_wait(&bars[BB_KV], 0, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
      for (int u = 0; u < nI && ok; ++u) {
        const int st = u & 1;
        const uint32_t sQs = sQ + st * tb;
        ok = mbar_wait(&bars[BB_QFULL + st], (u >> 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA) &&
             mbar_wait(&bars[BB_DOFULL], u & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
        if (ok && u > 0) ok = mbar_wait(&bars[BB_DQFREE], (u - 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          umma_ss(tA, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQs + off, 16, 1024), idS, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          umma_ss(tB, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sdO + off, 16, 1024), idS, ks > 0);
        }
        umma_commit(&bars[BB_SDP]);
        ok = mbar_wait(&bars[BB_PDS], u & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC);
        if (!ok) break;
        tc_fence_after();
        // dV += P^T dO ; dK += dS^T Q   (A from TMEM, B MN-major from smem)
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks)
          umma_ts(tdV, tA + ks * 8, sdesc_sw128(sdO + ks * 2048, 16384, 1024), idKV, (u > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks)
          umma_ts(tdK, tB + ks * 8, sdesc_sw128(sQs + ks * 2048, 16384, 1024), idKV, (u > 0 || ks > 0) ? 1u : 0u);
        // dQ_I = dS K_J, 64 output columns per MMA (A = dS^T smem read as MN-major dS). The last
        // one is 80 wide: its B operand continues past the K chunk into the ones chunk, so
        // output column 64 is R_i's part from this key tile (columns 65..79 are zeros).
#pragma unroll
        for (int x = 0; x < D / 64; ++x) {
          const bool last = x == D / 64 - 1;
          const uint32_t tdq = (D == 128 && x == 0) ? tB + 64 : tA + 64;
          const uint32_t kchunk = sK + x * 16384;
          const uint32_t lbo = last ? sOnes - kchunk : 16384;
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            umma_ss(tdq, sdesc_sw128(sdS + ks * 2048, 16384, 1024), sdesc_sw128(kchunk + ks * 2048, lbo, 1024),
                    last ? idQR : idQ, ks > 0);
        }
        umma_commit(&bars[BB_DQ]);
        umma_commit(&bars[BB_QEMPTY + st]);
        umma_commit(&bars[BB_DOEMPTY]);
      }
      umma_commit(&bars[BB_FINAL]);
      mbar_wait_drain(&bars[BB_FINAL], 0);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------- P^T, dS^T, dQ, epilogue
    const int wq = warp & 3, ch = warp >> 2;
    const int jr = wq * 32 + lane;  // TMEM lane: key row for S^T/dP^T/dK/dV, query row for dQ
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tA = tbase + lane_off, tB = tbase + 128 + lane_off;
    const uint32_t tdK = tbase + 256 + lane_off, tdV = tbase + 256 + D + lane_off;
    const uint32_t sds_row = smem_u32(sm + L::kDS) + (uint32_t)jr * 128u;
    const float* dlt = reinterpret_cast<const float*>(sm + L::kDR);
    const float* rh = dlt + kTile;
    const float* rec = reinterpret_cast<const float*>(sm + L::kRec);
    float csum = 0.f;
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[BB_KV], 0, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA));
    float kap = 0.f, baseJ_hi = 0.f, baseJ_lo = 0.f;
    if (ok) {
      kap = rec[jr];
      baseJ_hi = rec[kTile];
      baseJ_lo = rec[kTile + 1];
    }
    const float* recs = p.colrec + (size_t)bh * p.nT * kColRec;
    for (int u = 0; u < nI && ok; ++u) {
      const int I = J + u;
      const float baseI_hi = recs[(size_t)I * kColRec + kTile], baseI_lo = recs[(size_t)I * kColRec + kTile + 1];
      ok = mbar_wait(&bars[BB_SDP], u & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA) &&
           mbar_wait(&bars[BB_DOFULL], u & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
      ok = __all_sync(0xffffffffu, ok);  // tcgen05 loads/stores below are warp-collective
      tc_fence_after();
      // x_ji (log2 units, minus the row offset) = scale2 * S^T_ji - kappa_j + (base_I - base_J) - rho_i
      const float cj = ((baseI_hi - baseJ_hi) + (baseI_lo - baseJ_lo)) - kap;
      // Half ch = 1 overwrites packed columns that still hold half 0's S / dP values
      // for queries 32..63: half 0 arrives on the quarter's barrier once it has read
      // them. Half 0 arrives once per iteration it enters, even after a failed wait,
      // so half 1 never waits on a barrier that cannot complete.
      if (ch == 0) {
        if (!ok) {
          named_bar_arrive(1 + wq, 64);
          break;
        }
        if (u == 0) {
          pds_chunk<true>(tA, tB, 0, jr, p.scale2, cj, dlt, rh, sds_row, csum);
          pds_chunk<true>(tA, tB, 32, jr, p.scale2, cj, dlt, rh, sds_row, csum);
        } else {
          pds_chunk<false>(tA, tB, 0, jr, p.scale2, cj, dlt, rh, sds_row, csum);
          pds_chunk<false>(tA, tB, 32, jr, p.scale2, cj, dlt, rh, sds_row, csum);
        }
        named_bar_arrive(1 + wq, 64);
      } else {
        if (!ok) break;
        named_bar_sync(1 + wq, 64);
        if (u == 0) {
          pds_chunk<true>(tA, tB, 64, jr, p.scale2, cj, dlt, rh, sds_row, csum);
          pds_chunk<true>(tA, tB, 96, jr, p.scale2, cj, dlt, rh, sds_row, csum);
        } else {
          pds_chunk<false>(tA, tB, 64, jr, p.scale2, cj, dlt, rh, sds_row, csum);
          pds_chunk<false>(tA, tB, 96, jr, p.scale2, cj, dlt, rh, sds_row, csum);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[BB_PDS]);
      // dQ of this pair: TMEM lane = query row of tile I
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[BB_DQ], u & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA));
      if (!ok) break;
      tc_fence_after();
      {
        constexpr int kCols = D / 2;  // this half's output columns
        const int e0 = ch * kCols;
        const uint32_t src = (D == 128) ? (ch == 0 ? tB + 64 : tA + 64) : (tA + 64 + e0);
        float* dst = p.dqacc + ((size_t)bh * p.Npad + (size_t)I * kTile + jr) * D + e0;
#pragma unroll
        for (int c = 0; c < kCols; c += 32) {
          uint32_t r[32];
          tmem_ld32(src + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            red_add_v4(dst + c + e, __uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                       __uint_as_float(r[e + 3]));
        }
        if (ch == 1) {  // this key tile's part of R_i, in the column after the last dQ column
          uint32_t rv;
          tmem_ld1(tA + 128, rv);
          tmem_ld_wait();
          atomicAdd(p.rowsum + (size_t)bh * p.Npad + (size_t)I * kTile + jr, __uint_as_float(rv));
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[BB_DQFREE]);
    }
    // Column sums: half 1 hands its partial to half 0 through shared memory.
    float* cs = reinterpret_cast<float*>(sm + L::kCs);
    if (ch == 1) cs[jr] = csum;
    named_bar_sync(5, 256);
    const int j = J * kTile + jr;
    if (ok && ch == 0) p.colsum[(size_t)bh * p.Npad + j] = csum + cs[jr];
    // dK, dV epilogue
    if (ok) ok = mbar_wait(&bars[BB_FINAL], 0, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      constexpr int kCols = D / 2;
      const int e0 = ch * kCols;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t src = (which == 0 ? tdK : tdV) + e0;
        const float mul = which == 0 ? p.scale : 1.f;
        __nv_bfloat16* outp = which == 0 ? p.dk : p.dv;
#pragma unroll
        for (int c = 0; c < kCols; c += 32) {
          uint32_t r[32];
          tmem_ld32(src + c, r);
          tmem_ld_wait();
          if (j < p.N) {
            uint4* dst = reinterpret_cast<uint4*>(outp + (((size_t)b * p.N + j) * p.H + h) * D + e0 + c);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(r[8 * q4 + 0]) * mul, __uint_as_float(r[8 * q4 + 1]) * mul);
              w.y = pack_bf16x2(__uint_as_float(r[8 * q4 + 2]) * mul, __uint_as_float(r[8 * q4 + 3]) * mul);
              w.z = pack_bf16x2(__uint_as_float(r[8 * q4 + 4]) * mul, __uint_as_float(r[8 * q4 + 5]) * mul);
              w.w = pack_bf16x2(__uint_as_float(r[8 * q4 + 6]) * mul, __uint_as_float(r[8 * q4 + 7]) * mul);
              dst[q4] = w;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ---------------------------------------------------------------- dQ out
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(int B, int N, int H, int Npad, float scale,
                                                    const float* __restrict__ dqacc, __nv_bfloat16* __restrict__ dq) {
  constexpr int E = D / 32;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (long long)B * N * H) return;
  const int h = (int)(row % H);
  const long long bi = row / H;
  const int i = (int)(bi % N);
  const int b = (int)(bi / N);
  const float* src = dqacc + (((size_t)b * H + h) * Npad + i) * D + lane * E;
  __nv_bfloat16* dst = dq + (size_t)row * D + lane * E;
  if (E == 4) {
    const float4 v = *reinterpret_cast<const float4*>(src);
    uint2 w;
    w.x = pack_bf16x2(v.x * scale, v.y * scale);
    w.y = pack_bf16x2(v.z * scale, v.w * scale);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
    const float2 v = *reinterpret_cast<const float2*>(src);
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(v.x * scale, v.y * scale);
  }
}

// ---------------------------------------------------------- gate backward
// One CTA (1024 threads) per (b, h): reverse inclusive scan of the column
// sums minus the column sums in chunks of 1024, from the end of the sequence.
__global__ void __launch_bounds__(1024) bwd_gate_kernel(int N, int H, int Npad, int bias_from_j,
                                                       const float* __restrict__ colsum,
                                                       const float* __restrict__ rowsum, const float* __restrict__ z,
                                                       float* __restrict__ dz) {
  __shared__ float wsum[32];
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh % H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* C = colsum + (size_t)bh * Npad;
  const float* R = rowsum + (size_t)bh * Npad;
  float carry = 0.f;
  const int nchunks = (N + 1023) / 1024;
  for (int ck = nchunks - 1; ck >= 0; --ck) {
    // element t = ck*1024 + 1023 - tid, so the scan in tid order is a suffix scan in t
    const int t = ck * 1024 + 1023 - tid;
    const float c = t < N ? C[t] : 0.f;
    float x = t < N ? R[t] - c : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      float w = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      wsum[lane] = w;
    }
    __syncthreads();
    const float incl = x + (warp > 0 ? wsum[warp - 1] : 0.f) + carry;  // sum_{s >= t} (R_s - C_s)
    if (t < N) {
      const float da = bias_from_j ? incl + c : incl;
      const float zt = z[((size_t)b * N + t) * H + h];
      const float sig_neg = 1.f / (1.f + expf(zt));  // sigmoid(-z); 0 at z = +inf
      dz[((size_t)b * N + t) * H + h] = da * sig_neg;
    }
    carry += wsum[31];
    __syncthreads();
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
    TraceScope trace("bwd_rows", s);
    bwd_rows_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(
        a.B, a.N, a.H, g.Npad, static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dO), a.lse,
        rowloc, delta, rho, rowsum, dqacc);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fox_attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  BwdKParams p;
  p.B = a.B;
  p.N = a.N;
  p.H = a.H;
  p.nT = g.nT;
  p.Npad = g.Npad;
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
  const long long blocks = (long long)g.nT * g.BH;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  {
    TraceScope trace("attn_bwd", s);
    fox_attn_bwd_kernel<D><<<(unsigned)blocks, kBwdThreads, L::kAlloc, s>>>(maps[0], maps[1], maps[2], maps[3], p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long drows = (long long)a.B * a.N * a.H;
  {
    TraceScope trace("bwd_dq", s);
    bwd_dq_kernel<D><<<(unsigned)((drows + 7) / 8), 256, 0, s>>>(a.B, a.N, a.H, g.Npad, a.scale, dqacc,
                                                                   static_cast<__nv_bfloat16*>(a.dq));
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    TraceScope trace("bwd_gate", s);
    bwd_gate_kernel<<<g.BH, 1024, 0, s>>>(a.N, a.H, g.Npad, a.bias_from_j, colsum, rowsum, a.z, a.dz);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(const AttnBwdArgs& a, const GateLayout& g, const BwdLayout& w, const CUtensorMap* maps,
                            cudaStream_t s) {
  if (a.d == 64) return launch_bwd_d<64>(a, g, w, maps, s);
  if (a.d == 128) return launch_bwd_d<128>(a, g, w, maps, s);
  return cudaErrorInvalidValue;
}

}  // namespace fox
