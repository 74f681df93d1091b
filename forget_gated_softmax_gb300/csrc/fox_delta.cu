// Delta_i = dO_i . O_i for the non-causal backward, formed without O: since
// O_i = sum_j P_ij v_j, Delta_i = sum_j P_ij (dO_i . v_j) = sum_j P_ij dP_ij, with
// P_ij = exp(x_ij - LSE_i) recomputed from the forward's LSE exactly as the backward
// kernel does ("Forgetting Transformer (FoX) Attention" module source,
// ForgettingAttention.forward, differentiated by the chain rule). Without the causal
// mask the gate gradient is a small difference of large row and column sums of
// dS = P (dP - Delta), and a Delta taken from the bf16-rounded O moves it by percents;
// here P and dP stay in fp32 throughout.
//
// One CTA per (b, h, 128-row Q tile), over every key tile. Per key tile the tensor core
// forms S = Q K^T and dP = dO V^T (tcgen05, fp32 in tensor memory, double-buffered over
// the key tiles); the softmax warps recompute P in registers and accumulate sum_j P dP.
// No running maximum is needed (LSE is known), so no row state crosses key tiles but the
// sum. Warp roles (320 threads):
//   warps 0-7  rows x column halves: warp w reads TMEM lanes 32 (w % 4) .. + 31 and
//              columns [64 (w / 4), + 64) of S and dP
//   warp  8    TMA producer (Q and dO once; K, V and the column-term record per key tile)
//   warp  9    TMEM allocator and single-thread MMA issuer
// Tensor memory: S0 [0, 128) S1 [128, 256) dP0 [256, 384) dP1 [384, 512).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fox_internal.h"
#include "fox_ptx.cuh"

namespace fox {
namespace {

constexpr int kDeltaThreads = 320;
constexpr int kRecBytes = kColRec * 4;  // 528

struct DeltaParams {
  int B, N, H, nT, Npad;
  float scale2;  // scale * log2 e
  const float* rowloc;
  const float* colrec;
  const float* lse;
  float* delta;
  uint32_t* err;
};

template <int D>
struct DeltaLayout {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kDO = kTileBytes;
  static constexpr int kK = 2 * kTileBytes;    // + stage * kTileBytes
  static constexpr int kV = 4 * kTileBytes;    // + stage * kTileBytes
  static constexpr int kRec = 6 * kTileBytes;  // + stage * kRecBytes
  static constexpr int kRed = kRec + 2 * kRecBytes;  // 128 floats: the column halves' partial sums
  static constexpr int kBars = kRed + kTile * 4;
  static constexpr int kNumBars = 16;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  // Slack for 1024-byte alignment; at least 116 KB so that one CTA (all 512 TMEM columns)
  // is resident per SM.
  static constexpr int kAlloc = (kBytes + 1024) > 118784 ? (kBytes + 1024) : 118784;
};

enum DeltaBar {
  DB_QO = 0,
  DB_KFULL = 1,   // +stage
  DB_KEMPTY = 3,  // +stage
  DB_VFULL = 5,   // +stage (V and the column-term record)
  DB_VEMPTY = 7,  // +stage
  DB_SFULL = 9,   // +buffer: S and dP of the key tile are in tensor memory
  DB_SFREE = 11,  // +buffer: the softmax warps are done with them (one arrival per warp)
  DB_DONE = 13,
};

template <int D>
__global__ void __launch_bounds__(kDeltaThreads, 1)
    fox_delta_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                     const DeltaParams p) {
  using L = DeltaLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Head-major order: the CTAs resident at once share one or two heads, whose K and V
  // then stay in L2 across their query tiles.
  const int I = static_cast<int>(blockIdx.x) % p.nT;
  const int bh = static_cast<int>(blockIdx.x) / p.nT;
  const int b = bh / p.H, h = bh % p.H;
  const int nJ = p.nT;

  if (threadIdx.x == 0) {
    mbar_init(&bars[DB_QO], 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars[DB_KFULL + t], 1);
      mbar_init(&bars[DB_KEMPTY + t], 1);
      mbar_init(&bars[DB_VFULL + t], 1);
      mbar_init(&bars[DB_VEMPTY + t], 1);
      mbar_init(&bars[DB_SFULL + t], 1);
      mbar_init(&bars[DB_SFREE + t], 8);
    }
    mbar_init(&bars[DB_DONE], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
      tma_prefetch_desc(&tmap_do);
      constexpr uint32_t tb = L::kTileBytes;
      mbar_arrive_expect_tx(&bars[DB_QO], 2 * tb);
      for (int x = 0; x < D / 64; ++x) {
        tma_load_4d(sm + L::kQ + x * 16384, &tmap_q, &bars[DB_QO], x * 64, h, I * kTile, b);
        tma_load_4d(sm + L::kDO + x * 16384, &tmap_do, &bars[DB_QO], x * 64, h, I * kTile, b);
      }
      const float* rec_base = p.colrec + (size_t)bh * p.nT * kColRec;
      int kf[2] = {0, 0}, vf[2] = {0, 0};  // fills issued per stage
      for (int s = 0; s < nJ; ++s) {
        const int st = s & 1, n = s >> 1, J = s;
        if (n > 0 && !mbar_wait(&bars[DB_KEMPTY + st], (n - 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC)) break;
        mbar_arrive_expect_tx(&bars[DB_KFULL + st], tb);
        for (int x = 0; x < D / 64; ++x)
          tma_load_4d(sm + L::kK + st * tb + x * 16384, &tmap_k, &bars[DB_KFULL + st], x * 64, h, J * kTile, b);
        ++kf[st];
        // V and the record of this stage are free once dP of key tile s - 2 retired and the
        // softmax warps have read that tile's record.
        if (n > 0 && !(mbar_wait(&bars[DB_VEMPTY + st], (n - 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC) &&
                       mbar_wait(&bars[DB_SFREE + st], (n - 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC)))
          break;
        mbar_arrive_expect_tx(&bars[DB_VFULL + st], tb + kRecBytes);
        for (int x = 0; x < D / 64; ++x)
          tma_load_4d(sm + L::kV + st * tb + x * 16384, &tmap_v, &bars[DB_VFULL + st], x * 64, h, J * kTile, b);
        bulk_load(sm + L::kRec + st * kRecBytes, rec_base + (size_t)J * kColRec, kRecBytes, &bars[DB_VFULL + st]);
        ++vf[st];
      }
      // Drain: every copy this CTA issued must land before shared memory is released.
      mbar_wait_drain(&bars[DB_QO], 0);
      for (int st = 0; st < 2; ++st) {
        if (kf[st] > 0) mbar_wait_drain(&bars[DB_KFULL + st], (kf[st] - 1) & 1);
        if (vf[st] > 0) mbar_wait_drain(&bars[DB_VFULL + st], (vf[st] - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // D = 128: the whole warp runs the issue loop and one elected lane issues (0.901 -> 0.706 ms
    // at B1 H32 N8192); D = 64 measured 4 % faster with lane 0 alone.
    if (D == 128 || lane == 0) {
      const uint32_t leader = D == 128 ? elect_lane() : 1u;  // the one lane that issues (see umma_ss_e)
      constexpr uint32_t tb = L::kTileBytes;
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
      // Operand descriptors, computed once: Q and dO (A), K and V per stage (B).
      uint64_t dQ[D / 16], dO_[D / 16], dK[2][D / 16], dV[2][D / 16];
      {
        const uint32_t sQ = smem_u32(sm + L::kQ), sDO = smem_u32(sm + L::kDO);
        const uint32_t sK = smem_u32(sm + L::kK), sV = smem_u32(sm + L::kV);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          dQ[ks] = sdesc_sw128(sQ + off, 16, 1024);
          dO_[ks] = sdesc_sw128(sDO + off, 16, 1024);
          dK[0][ks] = sdesc_sw128(sK + off, 16, 1024);
          dK[1][ks] = sdesc_sw128(sK + tb + off, 16, 1024);
          dV[0][ks] = sdesc_sw128(sV + off, 16, 1024);
          dV[1][ks] = sdesc_sw128(sV + tb + off, 16, 1024);
        }
      }
      bool ok = mbar_wait(&bars[DB_QO], 0, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
      for (int s = 0; s < nJ && ok; ++s) {
        const int st = s & 1, n = s >> 1;
        const uint32_t tS = tbase + 128 * st, tP = tbase + 256 + 128 * st;  // buffer = stage = s % 2
        if (n > 0 && !mbar_wait(&bars[DB_SFREE + st], (n - 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC)) break;
        if (!mbar_wait(&bars[DB_KFULL + st], n & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) umma_ss_e(leader, tS, dQ[ks], st ? dK[1][ks] : dK[0][ks], idS, ks > 0);
        umma_commit_e(leader, &bars[DB_KEMPTY + st]);
        if (!mbar_wait(&bars[DB_VFULL + st], n & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) umma_ss_e(leader, tP, dO_[ks], st ? dV[1][ks] : dV[0][ks], idS, ks > 0);
        umma_commit_e(leader, &bars[DB_VEMPTY + st]);
        umma_commit_e(leader, &bars[DB_SFULL + st]);
      }
      // Every MMA issued above must retire before tensor memory is freed.
      umma_commit_e(leader, &bars[DB_DONE]);
      mbar_wait_drain(&bars[DB_DONE], 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------- sum_j P dP over one column half
    const int wq = warp & 3, hf = warp >> 2;
    const int r = wq * 32 + lane;  // row within the Q tile = TMEM lane
    const int i = I * kTile + r;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float* recI = p.colrec + ((size_t)bh * p.nT + I) * kColRec;
    const float baseI_hi = recI[kTile], baseI_lo = recI[kTile + 1];
    // rho_i = LSE_i log2 e - l_i: P_ij = 2^(scale2 S_ij - kappa_j + (base_I - base_J) - rho_i)
    const float rho = i < p.N ? p.lse[((size_t)b * p.N + i) * p.H + h] * kLog2e - p.rowloc[(size_t)bh * p.Npad + i]
                              : INFINITY;
    const float2 sc2 = make_float2(p.scale2, p.scale2);
    float2 acc = make_float2(0.f, 0.f);
    bool ok = true;
    for (int s = 0; s < nJ && ok; ++s) {
      const int st = s & 1, n = s >> 1;
      ok = mbar_wait(&bars[DB_SFULL + st], n & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA) &&
           mbar_wait(&bars[DB_VFULL + st], n & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
      ok = __all_sync(0xffffffffu, ok);  // the tcgen05 loads below are warp-collective
      if (!ok) break;
      tc_fence_after();
      const float* kap = reinterpret_cast<const float*>(sm + L::kRec + st * kRecBytes);
      const float beta = (baseI_hi - kap[kTile]) + (baseI_lo - kap[kTile + 1]);
      const float2 noff = make_float2(beta - rho, beta - rho);  // = -(rho - beta)
      const uint32_t tS = tbase + 128 * st + lane_off + 64 * hf, tP = tbase + 256 + 128 * st + lane_off + 64 * hf;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t sv[32], pv[32];
        tmem_ld32(tS + 32 * half, sv);
        tmem_ld32(tP + 32 * half, pv);
        tmem_ld_wait();
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const int j = 64 * hf + 32 * half + 4 * j4;
          const float4 kk = lds_f4(kap + j);
          // t - off = scale2 S - kappa + (beta - rho) for columns j .. j + 3
          const float2 ta = fadd2(ffma2(make_float2(__uint_as_float(sv[4 * j4]), __uint_as_float(sv[4 * j4 + 1])), sc2,
                                        make_float2(-kk.x, -kk.y)),
                                  noff);
          const float2 tc = fadd2(ffma2(make_float2(__uint_as_float(sv[4 * j4 + 2]), __uint_as_float(sv[4 * j4 + 3])),
                                        sc2, make_float2(-kk.z, -kk.w)),
                                  noff);
          const float2 pa = make_float2(ex2_approx(ta.x), ex2_approx(ta.y));
          const float2 pc = make_float2(ex2_approx(tc.x), ex2_approx(tc.y));
          acc = ffma2(pa, make_float2(__uint_as_float(pv[4 * j4]), __uint_as_float(pv[4 * j4 + 1])), acc);
          acc = ffma2(pc, make_float2(__uint_as_float(pv[4 * j4 + 2]), __uint_as_float(pv[4 * j4 + 3])), acc);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[DB_SFREE + st]);
    }
    // The two column halves of each row: warp w + 4 hands its sum to warp w.
    float* red = reinterpret_cast<float*>(sm + L::kRed);
    if (hf == 1) red[r] = acc.x + acc.y;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (ok && hf == 0 && i < p.N) p.delta[(size_t)bh * p.Npad + i] = (acc.x + acc.y) + red[r];
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D>
cudaError_t launch_delta_d(const DeltaArgs& a, const CUtensorMap* maps, int nT, int Npad, cudaStream_t s) {
  using L = DeltaLayout<D>;
  static_assert(L::kAlloc <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(fox_delta_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  DeltaParams p;
  p.B = a.B;
  p.N = a.N;
  p.H = a.H;
  p.nT = nT;
  p.Npad = Npad;
  p.scale2 = a.scale * kLog2e;
  p.rowloc = a.rowloc;
  p.colrec = a.colrec;
  p.lse = a.lse;
  p.delta = a.delta;
  p.err = a.err;
  const long long blocks = (long long)nT * a.B * a.H;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  {
    TraceScope trace("delta_pass", s);
    fox_delta_kernel<D><<<static_cast<unsigned>(blocks), kDeltaThreads, L::kAlloc, s>>>(maps[0], maps[1], maps[2],
                                                                                         maps[3], p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_delta_pass(const DeltaArgs& a, const CUtensorMap* maps, int nT, int Npad, cudaStream_t s) {
  if (a.d == 64) return launch_delta_d<64>(a, maps, nT, Npad, s);
  if (a.d == 128) return launch_delta_d<128>(a, maps, nT, Npad, s);
  return cudaErrorInvalidValue;
}

}  // namespace fox
