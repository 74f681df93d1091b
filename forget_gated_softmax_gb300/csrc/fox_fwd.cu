// Fused causal forget-gated attention forward, bf16 in / fp32 accumulate, for
// sm_103a: TMA-staged Q/K/V tiles, S = Q K^T and O += P V as tcgen05 MMAs
// into tensor memory, the forget bias and causal mask folded into an online
// softmax in registers, fully masked tiles never visited.
//
// Math ("Forgetting Transformer (FoX) Attention" module source,
// ForgettingAttention.forward; foxwindow README, score form): for query row i
// and key j <= i,  x_ij = scale * q_i.k_j + c_i - c_j  (j+1 convention; the j
// convention swaps the column term for c_{j-1}), O_i = softmax_j(x_ij) V.
// In log2 units with the two-level gate terms (see fox_internal.h):
//   x_ij * log2e = l_i + [ scale*log2e * S_ij - kappa_j ] + (base_I - base_J).
// The row term l_i is constant along the row and cancels in the softmax; it
// is added back into LSE only.
//
// KV tiles are visited from the diagonal backwards. The forget bias falls
// monotonically with distance (foxwindow README, "The window is a
// first-passage time"), so the row maximum is almost always found in the
// first tile; later tiles then take a single pass with that maximum, and the
// rare tile whose maximum exceeds it by more than 2^8 is recomputed after
// rescaling O.
//
// CTA = one (b, h) and a block of 256 query rows = two 128-row Q tiles that
// share every K/V tile (ping-pong: while the softmax of one tile runs, the
// tensor core works on the other). Warp roles (384 threads):
//   warps 0-3  softmax + epilogue of Q tile 0 (thread = row = TMEM lane)
//   warps 4-7  softmax + epilogue of Q tile 1
//   warp  8    TMA producer (Q once; K, V and the column-term record per KV tile, 2 stages)
//   warp  9    TMEM allocator and MMA issuer (the whole warp runs the issue loop, one
//              elected lane issues)
//   warps 10-11 V converters: each V tile from bf16 to fp16, in place in shared memory
//               (only when V is not already in fp16: the caller's workspace normally holds
//               an fp16 copy, written once by the gate step's base-scan kernel, and these
//               warps do not exist)
// Tensor memory (512 columns): S0 [0,128) S1 [128,256) O0, O1 (d columns each).
// P (fp16) overwrites the first 64 columns of its S buffer and feeds the P V
// MMA straight from tensor memory.
//
// P V runs in fp16 (P and V both fp16, fp32 accumulation). With bf16 P its
// 8-bit significand adds up to about 2.5e-3 to O on these workloads, on top of
// the up to 2^-7 of O's own bf16 rounding, which passes the 1e-2 bound on O; the
// 11 bits of fp16 P leave only the output rounding. Every bf16 V value of
// magnitude in [2^-14, 65280] is exactly an fp16 value, smaller ones round to
// the nearest multiple of 2^-24, and a magnitude of 65536 or more (outside
// fp16) sets DEV_ERR_RANGE in the error word.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fox_internal.h"
#include "fox_ptx.cuh"

namespace fox {
namespace {

constexpr int kConvWarps = 2;  // V converter warps (one measured 21 % slower on the long workload, three or
                               // four 9-11 %: their threads lower the register cap of every warp to 128)
// Threads: with V in fp16 already (kPreV) there are no converter warps.
__host__ __device__ constexpr int fwd_threads(bool pre_v) { return 320 + (pre_v ? 0 : 32 * kConvWarps); }
constexpr int kKappaBytes = kColRec * 4;   // 528
constexpr float kRescaleThreshold = 8.0f;  // log2 units: keep a row maximum while the tile max stays within 2^8
// Heads whose query blocks are scheduled together: 8 at d = 128, 16 at d = 64.
template <int D>
__host__ __device__ constexpr int fwd_head_group() { return D == 128 ? 8 : 16; }

struct FwdKParams {
  int B, N, H, nT, nQB, Npad;
  int non_causal;
  float scale2;  // scale * log2 e
  const float* rowloc;
  const float* colrec;
  __nv_bfloat16* o;
  float* lse;
  uint32_t* err;
  const int* jmin;  // tile skipping: first key tile of each query tile ([bh][nT]), or null
};

template <int D>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kQ0 = 0;
  static constexpr int kQ1 = kTileBytes;
  static constexpr int kK = 2 * kTileBytes;
  static constexpr int kV = 4 * kTileBytes;
  static constexpr int kKappa = 6 * kTileBytes;
  static constexpr int kBars = kKappa + 2 * kKappaBytes;  // 8-byte aligned (528 * 2 = 1056)
  static constexpr int kNumBars = 18;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  // Slack for 1024-byte alignment of the base; at least 116 KB so that only one CTA (which
  // takes all 512 TMEM columns) is ever resident per SM.
  static constexpr int kAlloc = (kBytes + 1024) > 118784 ? (kBytes + 1024) : 118784;
};

enum Bar {
  B_Q = 0,
  B_KFULL = 1,    // +stage
  B_KEMPTY = 3,   // +stage
  B_VFULL = 5,    // +stage
  B_VEMPTY = 7,   // +stage
  B_SFULL = 9,    // +tile
  B_PFULL = 11,   // +tile (one arrival per softmax warp)
  B_OFINAL = 13,  // +tile
  B_DONE = 15,
  B_VCONV = 16,   // +stage: the V tile of the stage converted to fp16 (one arrival per converter warp)
};

// Row maximum of t_j = scale2 * S_j - kappa_j over the 128 columns of this
// thread's S row in tensor memory (columns j > r masked on the diagonal tile).
// The loops below work on column pairs in packed fp32 with the negated argument
// tn_j = kappa_j - scale2 * S_j = -t_j (exactly, as rounding is symmetric), so that the
// column term enters without a negation; t_j - off is then (-off) - tn_j, again exact.
template <bool kDiag>
__device__ __forceinline__ float row_max(uint32_t tS, const float* kap, float scale2, int r) {
  const float2 nsc = make_float2(-scale2, -scale2);
  float mn = INFINITY;  // min_j tn_j
#pragma unroll
  for (int qt = 0; qt < 4; ++qt) {
    uint32_t raw[32];
    tmem_ld32(tS + 32 * qt, raw);
    tmem_ld_wait();
#pragma unroll
    for (int j4 = 0; j4 < 8; ++j4) {
      const int j = 32 * qt + 4 * j4;
      const float4 kk = lds_f4(kap + j);
      float2 a = ffma2(make_float2(__uint_as_float(raw[4 * j4]), __uint_as_float(raw[4 * j4 + 1])), nsc,
                       make_float2(kk.x, kk.y));
      float2 c = ffma2(make_float2(__uint_as_float(raw[4 * j4 + 2]), __uint_as_float(raw[4 * j4 + 3])), nsc,
                       make_float2(kk.z, kk.w));
      if (kDiag) {
        if (j > r) a.x = INFINITY;
        if (j + 1 > r) a.y = INFINITY;
        if (j + 2 > r) c.x = INFINITY;
        if (j + 3 > r) c.y = INFINITY;
      }
      mn = fmin3(fmin3(mn, a.x, a.y), c.x, c.y);
    }
  }
  return -mn;
}

// p_j = 2^(t_j - off) for the 128 columns, written back as fp16 pairs into
// the first 64 columns of the same S row (chunk q's P lands on columns
// [16q, 16q+16), which only hold S values already read). Returns sum_j p_j (fp32).
template <bool kDiag>
__device__ __forceinline__ float exp_pass(uint32_t tS, const float* kap, float scale2, float off, int r) {
  const float2 nsc = make_float2(-scale2, -scale2), noff = make_float2(-off, -off);
  float2 s = make_float2(0.f, 0.f);  // sums of the even and odd columns
#pragma unroll
  for (int qt = 0; qt < 4; ++qt) {
    uint32_t raw[32];
    tmem_ld32(tS + 32 * qt, raw);
    tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int j4 = 0; j4 < 8; ++j4) {
      const int j = 32 * qt + 4 * j4;
      const float4 kk = lds_f4(kap + j);
      // w = t - off for columns j .. j+3
      float2 wa = fsub2(noff, ffma2(make_float2(__uint_as_float(raw[4 * j4]), __uint_as_float(raw[4 * j4 + 1])),
                                    nsc, make_float2(kk.x, kk.y)));
      float2 wc = fsub2(noff, ffma2(make_float2(__uint_as_float(raw[4 * j4 + 2]), __uint_as_float(raw[4 * j4 + 3])),
                                    nsc, make_float2(kk.z, kk.w)));
      if (kDiag) {
        if (j > r) wa.x = -INFINITY;
        if (j + 1 > r) wa.y = -INFINITY;
        if (j + 2 > r) wc.x = -INFINITY;
        if (j + 3 > r) wc.y = -INFINITY;
      }
      float pr[4];
      pr[0] = ex2_approx(wa.x);
      pr[1] = ex2_approx(wa.y);
      pr[2] = ex2_approx(wc.x);
      pr[3] = ex2_approx(wc.y);
      s = fadd2(s, fadd2(make_float2(pr[0], pr[1]), make_float2(pr[2], pr[3])));
      pk[2 * j4] = pack_f16x2(pr[0], pr[1]);
      pk[2 * j4 + 1] = pack_f16x2(pr[2], pr[3]);
    }
    tmem_st16(tS + 16 * qt, pk);
  }
  return s.x + s.y;
}

// One pass over the row for the tiles after the first: p_j = 2^(t_j - off) into
// registers (pk, packed fp16, not yet stored) together with max_j t_j (tmax), so
// that S is read from tensor memory once. The caller stores pk over the first 64
// columns, or, in the rare case that the row maximum grew past the threshold,
// discards it and recomputes P with the new maximum (S is still intact then).
__device__ __forceinline__ float exp_pass_deferred(uint32_t tS, const float* kap, float scale2, float off,
                                                   uint32_t* pk, float& tmax) {
  const float2 nsc = make_float2(-scale2, -scale2), noff = make_float2(-off, -off);
  float2 s = make_float2(0.f, 0.f);  // sums of the even and odd columns
  float mn = INFINITY;                // min_j tn_j = -max_j t_j
  uint32_t rawb[2][32];               // chunk qt in rawb[qt & 1]; the next chunk loads during this one's arithmetic
  tmem_ld32(tS, rawb[0]);
#pragma unroll
  for (int qt = 0; qt < 4; ++qt) {
    tmem_ld_wait();
    if (qt + 1 < 4) tmem_ld32(tS + 32 * (qt + 1), rawb[(qt + 1) & 1]);
    const uint32_t* raw = rawb[qt & 1];
#pragma unroll
    for (int j4 = 0; j4 < 8; ++j4) {
      const int j = 32 * qt + 4 * j4;
      const float4 kk = lds_f4(kap + j);
      const float2 a = ffma2(make_float2(__uint_as_float(raw[4 * j4]), __uint_as_float(raw[4 * j4 + 1])), nsc,
                             make_float2(kk.x, kk.y));
      const float2 c = ffma2(make_float2(__uint_as_float(raw[4 * j4 + 2]), __uint_as_float(raw[4 * j4 + 3])), nsc,
                             make_float2(kk.z, kk.w));
      mn = fmin3(fmin3(mn, a.x, a.y), c.x, c.y);
      const float2 wa = fsub2(noff, a), wc = fsub2(noff, c);  // t - off
      float pr[4];
      pr[0] = ex2_approx(wa.x);
      pr[1] = ex2_approx(wa.y);
      pr[2] = ex2_approx(wc.x);
      pr[3] = ex2_approx(wc.y);
      s = fadd2(s, fadd2(make_float2(pr[0], pr[1]), make_float2(pr[2], pr[3])));
      pk[16 * qt + 2 * j4] = pack_f16x2(pr[0], pr[1]);
      pk[16 * qt + 2 * j4 + 1] = pack_f16x2(pr[2], pr[3]);
    }
  }
  tmax = -mn;
  return s.x + s.y;
}

// A stage index as a type, for code specialised on it.
template <int V>
struct StageC {
  static constexpr int value = V;
};

template <int D, bool kPreV>
__global__ void __launch_bounds__(fwd_threads(kPreV), 1)
    fox_attn_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const FwdKParams p) {
  using L = FwdLayout<D>;
  // Launched as a programmatic dependent of the gate kernels (launch_dependent): the CTAs can be
  // resident when those finish, and wait here for their results. (Issuing the Q loads before the
  // wait, with the tile-span reads moved after it, measured 4 % slower on the long workload: the
  // compiled softmax and issue code changed.)
  grid_dep_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  // Work order: groups of heads, one after the other, and within a group the longest causal
  // rows first with the group's heads interleaved. The CTAs resident at once then share few
  // heads, whose K / V streams stay in L2. Against all heads interleaved: long workload
  // 1.477 -> 1.383 ms with groups of 16; groups of 8 then took its DRAM traffic per launch from
  // 1.11 to 0.55 GB at the same time, and the d = 128, N = 4096 shapes 1-2 % faster. At d = 64
  // (mid workload) groups of 16 measured 67.6 -> 63.4 us, groups of 8 slower than all heads.
  int qb, bh;
  {
    constexpr int kG = fwd_head_group<D>();
    const int idx = static_cast<int>(blockIdx.x);
    const int full = (BH / kG) * kG * p.nQB;
    const int gsize = idx < full ? kG : BH % kG;
    const int gbase = idx < full ? (idx / (kG * p.nQB)) * kG : BH - BH % kG;
    const int r = idx < full ? idx % (kG * p.nQB) : idx - full;
    qb = p.nQB - 1 - r / gsize;
    bh = gbase + r % gsize;
  }
  const int b = bh / p.H, h = bh % p.H;
  // Q tile k covers rows [128*I_k, 128*I_k + 128). KV tiles are streamed in
  // sequence order s = 0, 1, ..., nJ-1 with J = Jtop - s; tile k takes part
  // for s >= first_k. Causal: the stream starts at the last diagonal tile and
  // tile k's first tile is its own diagonal. Non-causal: every tile, from the
  // last one back (the bias c_i - c_j grows with j, so the largest bias comes first).
  // With tile skipping (causal only), tile k stops at key tile jmin(I_k): it takes
  // part for first_k <= s < end_k.
  const int I0 = 2 * qb, I1 = 2 * qb + 1;
  const bool has1 = I1 < p.nT;
  const bool causal = !p.non_causal;
  const int Jtop = causal ? (has1 ? I1 : I0) : p.nT - 1;
  const int first0 = (causal && has1) ? 1 : 0;
  const int jm0 = p.jmin ? p.jmin[(size_t)bh * p.nT + I0] : 0;
  const int jm1 = (p.jmin && has1) ? p.jmin[(size_t)bh * p.nT + I1] : 0;
  const int end0 = Jtop - jm0 + 1;
  const int end1 = has1 ? Jtop - jm1 + 1 : 0;
  const int nJ = end0 > end1 ? end0 : end1;

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_Q], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[B_KFULL + s], 1);
      mbar_init(&bars[B_KEMPTY + s], 1);
      mbar_init(&bars[B_VFULL + s], 1);
      mbar_init(&bars[B_VEMPTY + s], 1);
      mbar_init(&bars[B_SFULL + s], 1);
      mbar_init(&bars[B_PFULL + s], 4);
      mbar_init(&bars[B_OFINAL + s], 1);
      if (!kPreV) mbar_init(&bars[B_VCONV + s], kConvWarps);
    }
    mbar_init(&bars[B_DONE], 1);
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
      constexpr uint32_t tb = L::kTileBytes;
      mbar_arrive_expect_tx(&bars[B_Q], has1 ? 2 * tb : tb);
      for (int x = 0; x < D / 64; ++x) {
        tma_load_4d(sm + L::kQ0 + x * 16384, &tmap_q, &bars[B_Q], x * 64, h, I0 * kTile, b);
        if (has1) tma_load_4d(sm + L::kQ1 + x * 16384, &tmap_q, &bars[B_Q], x * 64, h, I1 * kTile, b);
      }
      const float* rec_base = p.colrec + (size_t)bh * p.nT * kColRec;
      int fills[2] = {0, 0};  // fills issued per stage (K and V of a stage go in lock step)
      for (int s = 0; s < nJ; ++s) {
        const int st = s & 1, n = s >> 1, J = Jtop - s;
        if (n > 0 && !mbar_wait(&bars[B_KEMPTY + st], (n - 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC)) break;
        mbar_arrive_expect_tx(&bars[B_KFULL + st], tb);
        for (int x = 0; x < D / 64; ++x)
          tma_load_4d(sm + L::kK + st * tb + x * 16384, &tmap_k, &bars[B_KFULL + st], x * 64, h, J * kTile, b);
        if (n > 0 && !mbar_wait(&bars[B_VEMPTY + st], (n - 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC)) {
          mbar_wait_drain(&bars[B_KFULL + st], n & 1);  // the K copy of this fill is in flight
          break;
        }
        mbar_arrive_expect_tx(&bars[B_VFULL + st], tb + kKappaBytes);
        for (int x = 0; x < D / 64; ++x)
          tma_load_4d(sm + L::kV + st * tb + x * 16384, &tmap_v, &bars[B_VFULL + st], x * 64, h, J * kTile, b);
        bulk_load(sm + L::kKappa + st * kKappaBytes, rec_base + (size_t)J * kColRec, kKappaBytes,
                  &bars[B_VFULL + st]);
        ++fills[st];
      }
      // Drain: every copy this CTA issued must land before shared memory is released.
      mbar_wait_drain(&bars[B_Q], 0);
      for (int st = 0; st < 2; ++st) {
        if (fills[st] == 0) continue;
        mbar_wait_drain(&bars[B_KFULL + st], (fills[st] - 1) & 1);
        mbar_wait_drain(&bars[B_VFULL + st], (fills[st] - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    {
      const uint32_t leader = elect_lane();  // the one lane that issues (see umma_ss_e)
      constexpr uint32_t tb = L::kTileBytes;
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idO = idesc_f16(128, D, false, true);  // P (TMEM) and V fp16
      // V of a stage is ready for P V once it landed (kPreV: loaded as fp16) or was converted.
      constexpr uint32_t kVErr = kPreV ? DEV_ERR_TIMEOUT_TMA : DEV_ERR_TIMEOUT_SYNC;
      const uint32_t tS[2] = {tbase, tbase + 128};
      const uint32_t tO[2] = {tbase + 256, tbase + 256 + D};
      // Descriptors of each operand tile's base. Shared-memory addresses stay below 2^18, so
      // the 14-bit start-address field of base + offset never carries: an operand at a byte
      // offset is the base descriptor plus offset / 16.
      const uint64_t dQ0 = sdesc_sw128(smem_u32(sm + L::kQ0), 16, 1024);
      const uint64_t dQ1 = sdesc_sw128(smem_u32(sm + L::kQ1), 16, 1024);
      const uint64_t dK0 = sdesc_sw128(smem_u32(sm + L::kK), 16, 1024);
      const uint64_t dK1 = sdesc_sw128(smem_u32(sm + L::kK + tb), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sm + L::kV), 16384, 1024);
      const uint64_t dV1 = sdesc_sw128(smem_u32(sm + L::kV + tb), 16384, 1024);
      const int first[2] = {first0, 0};
      const int end[2] = {end0, end1};
      const bool active[2] = {true, has1};
      // Every operand descriptor of the S and P V groups, computed once.
      uint64_t dA[2][D / 16], dB[2][D / 16], dVs[2][kTile / 16];
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t off = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
        dA[0][ks] = dQ0 + off;
        dA[1][ks] = dQ1 + off;
        dB[0][ks] = dK0 + off;
        dB[1][ks] = dK1 + off;
      }
#pragma unroll
      for (int ks = 0; ks < kTile / 16; ++ks) {
        dVs[0][ks] = dV0 + static_cast<uint64_t>((ks * 2048) >> 4);
        dVs[1][ks] = dV1 + static_cast<uint64_t>((ks * 2048) >> 4);
      }
      auto issue_s = [&](int k, int st) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) umma_ss_e(leader, tS[k], dA[k][ks], st ? dB[1][ks] : dB[0][ks], idS, ks > 0);
      };
      auto issue_pv = [&](int k, int st, bool acc) {
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) {
          const uint64_t dv = st ? dVs[1][ks] : dVs[0][ks];
          umma_ts_e(leader, tO[k], tS[k] + ks * 8, dv, idO, (acc || ks > 0) ? 1u : 0u);
        }
      };
      // One K-step of P V for Q tile k with the V descriptor dv.
      auto pv_ks = [&](int k, int ks, bool acc, uint64_t dv) {
        umma_ts_e(leader, tO[k], tS[k] + ks * 8, dv, idO, (acc || ks > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(&bars[B_Q], 0, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA) &&
                mbar_wait(&bars[B_KFULL + 0], 0, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
      if (ok) {
        tc_fence_after();
        for (int k = 0; k < 2; ++k)
          if (active[k] && first[k] == 0) {
            issue_s(k, 0);
            umma_commit_e(leader, &bars[B_SFULL + k]);
          }
        umma_commit_e(leader, &bars[B_KEMPTY + 0]);
      }
      for (int s = 0; s < nJ && ok; ++s) {
        const int st = s & 1, nst = (s + 1) & 1;
        bool kready = false;
        auto wait_next_k = [&]() -> bool {
          if (!kready) {
            if (!mbar_wait(&bars[B_KFULL + nst], ((s + 1) >> 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA))
              return false;
            tc_fence_after();
            kready = true;
          }
          return true;
        };
        // Both tiles take part in this step and the next: straight-line issue, specialised
        // on the stage parity so that every descriptor and barrier address is fixed.
        auto straight = [&](auto stage) -> bool {
          constexpr int ST = decltype(stage)::value, NST = ST ^ 1;
          bool ok = mbar_wait(&bars[(kPreV ? B_VFULL : B_VCONV) + ST], (s >> 1) & 1, abort_flag, p.err, kVErr) &&
                    mbar_wait(&bars[B_PFULL + 0], (s - first0) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC);
          if (!ok) return false;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks) pv_ks(0, ks, s > first0, dVs[ST][ks]);
          ok = mbar_wait(&bars[B_KFULL + NST], ((s + 1) >> 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
          if (!ok) return false;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) umma_ss_e(leader, tS[0], dA[0][ks], dB[NST][ks], idS, ks > 0);
          umma_commit_e(leader, &bars[B_SFULL + 0]);
          ok = mbar_wait(&bars[B_PFULL + 1], s & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC);
          if (!ok) return false;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks) pv_ks(1, ks, s > 0, dVs[ST][ks]);
          // The V stage is free once the last P V reading it retires: released before the next
          // S group so that the following V load (and its conversion) starts earlier.
          umma_commit_e(leader, &bars[B_VEMPTY + ST]);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) umma_ss_e(leader, tS[1], dA[1][ks], dB[NST][ks], idS, ks > 0);
          umma_commit_e(leader, &bars[B_SFULL + 1]);
          umma_commit_e(leader, &bars[B_KEMPTY + NST]);
          return true;
        };
        if (has1 && s >= first0 && s + 1 < end0 && s + 1 < end1) {
          ok = (s & 1) ? straight(StageC<1>{}) : straight(StageC<0>{});
          if (!ok) break;
          continue;
        }
        ok = mbar_wait(&bars[(kPreV ? B_VFULL : B_VCONV) + st], (s >> 1) & 1, abort_flag, p.err, kVErr);
        for (int k = 0; k < 2 && ok; ++k) {
          if (!active[k]) continue;
          if (s >= first[k] && s < end[k]) {
            ok = mbar_wait(&bars[B_PFULL + k], (s - first[k]) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_SYNC);
            if (!ok) break;
            tc_fence_after();
            issue_pv(k, st, s > first[k]);
            if (s + 1 < end[k]) {
              if (!(ok = wait_next_k())) break;
              issue_s(k, nst);
              umma_commit_e(leader, &bars[B_SFULL + k]);
            } else {
              umma_commit_e(leader, &bars[B_OFINAL + k]);
            }
          } else if (s + 1 == first[k]) {
            if (!(ok = wait_next_k())) break;
            issue_s(k, nst);
            umma_commit_e(leader, &bars[B_SFULL + k]);
          }
        }
        if (!ok) break;
        umma_commit_e(leader, &bars[B_VEMPTY + st]);
        if (kready) umma_commit_e(leader, &bars[B_KEMPTY + nst]);
      }
      // Every MMA issued above must retire before tensor memory is freed.
      umma_commit_e(leader, &bars[B_DONE]);
      mbar_wait_drain(&bars[B_DONE], 0);
    }
    __syncwarp();
  } else if (!kPreV && warp >= 10) {
    // ----------------------------------------------------------- V converters
    // Each V tile in place from bf16 to fp16, the two warps taking alternate 16-byte pieces
    // of the swizzled layout TMA wrote (the conversion is per element, so the layout is
    // unchanged), then a proxy fence so that the MMA's reads see the generic-proxy stores.
    uint32_t vmax = 0u;  // largest |v| bit pattern seen, per bf16 half
    for (int s = 0; s < nJ; ++s) {
      const int st = s & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_VFULL + st], (s >> 1) & 1, abort_flag, p.err,
                                                         DEV_ERR_TIMEOUT_TMA));
      if (!ok) break;
      uint4* tile = reinterpret_cast<uint4*>(sm + L::kV + st * L::kTileBytes);
#pragma unroll 4
      for (int e = (warp - 10) * 32 + lane; e < L::kTileBytes / 16; e += 32 * kConvWarps) {
        const uint4 w = tile[e];
        const uint32_t in[4] = {w.x, w.y, w.z, w.w};
        uint32_t out[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          out[c] = pack_f16x2(__uint_as_float(in[c] << 16), __uint_as_float(in[c] & 0xFFFF0000u));
          asm("max.u16x2 %0, %0, %1;" : "+r"(vmax) : "r"(in[c] & 0x7FFF7FFFu));
        }
        tile[e] = make_uint4(out[0], out[1], out[2], out[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_VCONV + st]);
    }
    // |v| >= 65536 (bf16 pattern 0x4780 and above, infinities included) is outside fp16.
    const bool over = (vmax & 0xFFFFu) >= 0x4780u || (vmax >> 16) >= 0x4780u;
    if (__any_sync(0xffffffffu, over) && lane == 0) atomicOr(p.err, DEV_ERR_RANGE);
  } else {
    // ------------------------------------------------------ softmax / epilogue
    const int k = warp >> 2;        // Q tile of this warpgroup
    const int wq = warp & 3;        // TMEM lane quarter
    const int r = wq * 32 + lane;   // row within the Q tile
    const int I = k ? I1 : I0;
    const int first = k ? 0 : first0;
    const int nJk = (k == 1 && !has1) ? 0 : (k ? end1 : end0 - first0);
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tbase + k * 128 + lane_off;
    const uint32_t tO = tbase + 256 + k * D + lane_off;
    const int i = I * kTile + r;
    if (nJk > 0) {
      const float* recI = p.colrec + ((size_t)bh * p.nT + I) * kColRec;
      const float baseI_hi = recI[kTile], baseI_lo = recI[kTile + 1];
      const float row_term = p.rowloc[(size_t)bh * p.Npad + i];
      float m_used = -INFINITY, l_sum = 0.f;
      bool ok = true;
      // First tile (u = 0): exact row maximum, then one pass. Causal: the diagonal tile
      // (base_I - base_J = 0), masked; non-causal: the last tile, unmasked.
      ok = mbar_wait(&bars[B_SFULL + k], 0, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA) &&
           mbar_wait(&bars[B_VFULL + (first & 1)], (first >> 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
      ok = __all_sync(0xffffffffu, ok);  // the tcgen05 loads below are warp-collective
      if (ok) {
        tc_fence_after();
        const float* kap = reinterpret_cast<const float*>(sm + L::kKappa + (first & 1) * kKappaBytes);
        // The first tile holds the largest bias (base_I - base_J is its offset; 0 on the diagonal).
        const float beta0 = (baseI_hi - kap[kTile]) + (baseI_lo - kap[kTile + 1]);
        if (causal) {
          m_used = row_max<true>(tS, kap, p.scale2, r);
          l_sum = exp_pass<true>(tS, kap, p.scale2, m_used, r);
        } else {
          m_used = row_max<false>(tS, kap, p.scale2, r) + beta0;
          l_sum = exp_pass<false>(tS, kap, p.scale2, m_used - beta0, r);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_PFULL + k]);
      }
      for (int u = 1; u < nJk && ok; ++u) {
        const int s = first + u, st = s & 1;
        ok = mbar_wait(&bars[B_SFULL + k], u & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA) &&
             mbar_wait(&bars[B_VFULL + st], (s >> 1) & 1, abort_flag, p.err, DEV_ERR_TIMEOUT_TMA);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float* kap = reinterpret_cast<const float*>(sm + L::kKappa + st * kKappaBytes);
        const float beta = (baseI_hi - kap[kTile]) + (baseI_lo - kap[kTile + 1]);
        // Rescale O and l of the rows whose maximum grew by more than 2^8 (alpha = 1 for
        // the others; the TMEM loads/stores are warp-collective, so the whole warp takes
        // this branch). s_full of this tile was committed after the previous P V, so O is
        // settled.
        auto rescale = [&](float m_cand, bool grow) {
          const float alpha = grow ? ex2_approx(m_used - m_cand) : 1.f;
          l_sum *= alpha;
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_ld32(tO + c, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + c, o);
          }
          if (grow) m_used = m_cand;
        };
        // One pass with the running maximum; the exact row maximum comes with it.
        uint32_t pk[64];
        float tmax;
        const float lsum_tile = exp_pass_deferred(tS, kap, p.scale2, m_used - beta, pk, tmax);
        const float m_cand = tmax + beta;
        const bool grow = m_cand > m_used + kRescaleThreshold;
        if (__any_sync(0xffffffffu, grow)) {  // rare: redo the tile with the new maximum
          rescale(m_cand, grow);
          l_sum += exp_pass<false>(tS, kap, p.scale2, m_used - beta, r);
        } else {
          l_sum += lsum_tile;
          tmem_st32(tS, pk);
          tmem_st32(tS + 32, pk + 32);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_PFULL + k]);
      }
      if (ok) ok = mbar_wait(&bars[B_OFINAL + k], 0, abort_flag, p.err, DEV_ERR_TIMEOUT_MMA);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        const float inv = 1.f / l_sum;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          tmem_ld_wait();
          if (i < p.N) {
            uint4* dst = reinterpret_cast<uint4*>(p.o + (((size_t)b * p.N + i) * p.H + h) * D + c);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[8 * q4 + 0]) * inv, __uint_as_float(o[8 * q4 + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv, __uint_as_float(o[8 * q4 + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv, __uint_as_float(o[8 * q4 + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv, __uint_as_float(o[8 * q4 + 7]) * inv);
              dst[q4] = w;
            }
          }
        }
        if (i < p.N) p.lse[((size_t)b * p.N + i) * p.H + h] = (m_used + __log2f(l_sum) + row_term) * kLn2;
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

template <int D, bool kPreV>
cudaError_t launch_d(const AttnFwdArgs& a, const CUtensorMap* maps, int nT, int Npad, cudaStream_t s) {
  using L = FwdLayout<D>;
  static_assert(L::kAlloc <= 232448, "shared memory budget");
  auto kernel = fox_attn_fwd_kernel<D, kPreV>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  FwdKParams p;
  p.B = a.B;
  p.N = a.N;
  p.H = a.H;
  p.nT = nT;
  p.nQB = (nT + 1) / 2;
  p.non_causal = a.non_causal;
  p.Npad = Npad;
  p.scale2 = a.scale * kLog2e;
  p.rowloc = a.rowloc;
  p.colrec = a.colrec;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.err = a.err;
  p.jmin = a.jmin;
  const long long blocks = (long long)p.nQB * a.B * a.H;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  {
    TraceScope trace("attn_fwd", s);
    e = launch_dependent(kernel, dim3(static_cast<unsigned>(blocks)), dim3(fwd_threads(kPreV)), L::kAlloc, s, maps[0], maps[1],
                         maps[2], p);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd_bf16(const AttnFwdArgs& a, const CUtensorMap* maps, int nT, int Npad, cudaStream_t s) {
  if (a.d == 64) return a.v16 ? launch_d<64, true>(a, maps, nT, Npad, s) : launch_d<64, false>(a, maps, nT, Npad, s);
  if (a.d == 128) return a.v16 ? launch_d<128, true>(a, maps, nT, Npad, s) : launch_d<128, false>(a, maps, nT, Npad, s);
  return cudaErrorInvalidValue;
}

}  // namespace fox
