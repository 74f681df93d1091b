// Internal layout and launcher declarations shared by the library's
// translation units (host side and kernels). Not part of the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda.h>

namespace fox {

constexpr int kTile = 128;          // tokens per sequence tile (MMA M and KV tile)
constexpr int kColRec = kTile + 4;  // floats per column record: 128 column terms + base hi, base lo, 2 pad
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Gate terms the attention kernels read, all in log2 units (natural value * log2 e).
//   rowloc[bh][t]   l_t  = sum_{l = 128*T .. t} a_l          (T = t / 128; inclusive, tile-local)
//   colrec[bh][T]   { kappa_j for j in tile T (tile-local column term:
//                     inclusive for the j+1 convention, exclusive for the j convention;
//                     +inf past the sequence end, which removes those keys from every row),
//                     base_T hi, base_T lo, 0, 0 },  base_T = sum_{l < 128*T} a_l (double-float scan, hi+lo)
//   tiletot[bh][T]  sum of a over tile T (fp32, scratch between the two gate kernels)
// so that, for i in tile I and j in tile J, D_ij * log2 e = l_i - kappa_j + (base_I - base_J).
// Tile-skip arrays (written only when skipping is requested):
//   qmax, kmax [bh][T]  largest row norm of q, k in tile T (fp32)
//   kpre       [bh][T]  running maximum of kmax over tiles 0..T
//   jmin       [bh][I]  first key tile query tile I visits (int)
//   imax       [bh][J]  last query tile key tile J serves (int)
struct GateLayout {
  int BH = 0, N = 0, nT = 0, Npad = 0;
  size_t rowloc = 0, colrec = 0, tiletot = 0;  // byte offsets from the workspace base
  size_t qmax = 0, kmax = 0, kpre = 0, jmin = 0, imax = 0;
  size_t end = 0;
};

// Backward-only buffers that follow the gate buffers.
struct BwdLayout {
  size_t delta = 0;   // float [BH][Npad]   Delta_i = dO_i . O_i (0 past the sequence end)
  size_t rho = 0;     // float [BH][Npad]   LSE_i * log2 e - l_i: row offset to recompute P (+inf past the end)
  size_t colsum = 0;  // float [BH][Npad]   C_j = sum_i dS_ij
  size_t rowsum = 0;  // float [BH][Npad]   R_i = sum_j dS_ij (0 in exact arithmetic; accumulated across key tiles)
  size_t dqacc = 0;   // float [BH][Npad][d] dQ accumulator (fp32, unscaled)
  size_t gstat = 0;   // [BH][nT] 32-byte status records of the gate gradient's look-back
  size_t end = 0;
};

constexpr size_t kErrWordBytes = 256;  // workspace header: uint32 error word + padding
constexpr size_t kTicketOffset = 128;  // header byte offset of the gate gradient's ticket counter
constexpr size_t kGateStatBytes = 32;  // bytes per (b h, 128-token block) look-back status record

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline GateLayout gate_layout(int B, int N, int H) {
  GateLayout g;
  g.BH = B * H;
  g.N = N;
  g.nT = (N + kTile - 1) / kTile;
  g.Npad = g.nT * kTile;
  size_t off = kErrWordBytes;
  g.rowloc = off;
  off = align_up(off + sizeof(float) * (size_t)g.BH * g.Npad, 256);
  g.colrec = off;
  off = align_up(off + sizeof(float) * (size_t)g.BH * g.nT * kColRec, 256);
  g.tiletot = off;
  const size_t per_tile = sizeof(float) * (size_t)g.BH * g.nT;  // sizeof(int) == sizeof(float)
  off = align_up(off + per_tile, 256);
  g.qmax = off;
  off = align_up(off + per_tile, 256);
  g.kmax = off;
  off = align_up(off + per_tile, 256);
  g.kpre = off;
  off = align_up(off + per_tile, 256);
  g.jmin = off;
  off = align_up(off + per_tile, 256);
  g.imax = off;
  off = align_up(off + per_tile, 256);
  g.end = off;
  return g;
}

inline BwdLayout bwd_layout(const GateLayout& g, int d) {
  BwdLayout w;
  size_t off = g.end;
  const size_t row = sizeof(float) * (size_t)g.BH * g.Npad;
  w.delta = off;
  off = align_up(off + row, 256);
  w.rho = off;
  off = align_up(off + row, 256);
  w.colsum = off;
  off = align_up(off + row, 256);
  w.rowsum = off;
  off = align_up(off + row, 256);
  w.dqacc = off;
  off = align_up(off + row * (size_t)d, 256);
  w.gstat = off;
  off = align_up(off + kGateStatBytes * (size_t)g.BH * g.nT, 256);
  w.end = off;
  return w;
}

// ---- kernel tracing (benchmark support) ----
// While tracing is on, TraceScope brackets a launch with two CUDA events on
// its stream; fox_trace_end() reports each launch's name and duration.
bool trace_enabled();
struct TraceScope {
  int slot = -1;
  cudaStream_t stream = nullptr;
  TraceScope(const char* name, cudaStream_t s);
  ~TraceScope();
};

// Launch `kernel` on `s` as a programmatic dependent of the kernel launched just before it on
// the same stream: it may start while that kernel still runs, so it must call grid_dep_wait()
// (fox_ptx.cuh) before reading anything that kernel (or any earlier one) wrote. Its prologue
// (barrier set-up, tensor-memory allocation, loads of the caller's inputs) then overlaps the
// end of the kernel before it.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ---- launchers (return cudaGetLastError() of the launch) ----
// c[b,t,h] = (base_T + local_t) / log2 e from the gate terms in the workspace (fp64 sum, fp32 out).
cudaError_t launch_gate_cumulative(const void* ws, const GateLayout& g, int B, int N, int H, float* c, cudaStream_t s);
// d a_t = sum_{s>=t} (R_s - C_s) (+ C_t when bias_from_j), dz = d a_t sigmoid(-z), in one pass with a
// decoupled look-back; R and C rows of `stride` floats per (b, h). `stat` (B * H * ceil(N / 128)
// records of kGateStatBytes) and `ticket` must be zero at the launch; err is the error word.
// True when the gate gradient takes one sequence per CTA (no look-back, no status records or
// ticket needed): enough (b, 4-head) sequences to occupy every SM, and tensor-map alignment.
bool gate_bwd_streams(int B, int N, int H, int stride, const float* colsum, const float* rowsum, const float* z,
                      const float* dz);
cudaError_t launch_gate_bwd(int B, int N, int H, int stride, int bias_from_j, const float* colsum,
                            const float* rowsum, const float* z, float* dz, void* stat, unsigned* ticket,
                            uint32_t* err, cudaStream_t s);
// The forward's fp16 copy of V: v (bf16, n elements, a multiple of 8, 16-byte aligned) to v16.
// Given to the gate launchers, it is done by the base-scan kernel, which runs alongside the
// tile scan; a magnitude of 65536 or more (outside fp16) sets DEV_ERR_RANGE.
struct V16Job {
  const void* v;
  void* v16;
  size_t n;
};
cudaError_t launch_gate_scan(const float* z, int B, int N, int H, int bias_from_j, void* ws, const GateLayout& g,
                             cudaStream_t s, const V16Job* v16 = nullptr);

struct AttnFwdArgs {
  int B, N, H, d;
  int non_causal;
  float scale;
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const float* rowloc;
  const float* colrec;
  uint32_t* err;
  const int* jmin = nullptr;  // tile skipping: first key tile of each query tile ([bh][nT]), or null
  const void* v16 = nullptr;  // fp16 copy of v ([B, N, H, d]), or null: the kernel then converts V on chip
};

// The forward's fp16 copy of V sits after the gate terms: B N H d halves.
inline size_t fwd_v16_offset(const GateLayout& g) { return g.end; }
inline size_t fwd_v16_bytes(int B, int N, int H, int d) { return (size_t)B * N * H * d * 2; }


cudaError_t launch_attn_fwd_bf16(const AttnFwdArgs& a, const CUtensorMap* maps /* q, k, v (v16 when set) */, int nT, int Npad,
                                 cudaStream_t s);
cudaError_t launch_attn_fwd_f32(const AttnFwdArgs& a, int nT, int Npad, cudaStream_t s);

struct AttnBwdArgs {
  int B, N, H, d, bias_from_j;
  int non_causal;
  float scale;
  const void* q;
  const void* k;
  const void* v;
  const float* z;
  const void* o;
  const float* lse;
  const void* dO;
  void* dq;
  void* dk;
  void* dv;
  float* dz;
  char* ws;  // workspace base (gate layout, then the backward layout)
  // Set when Delta of rows i < N is already in the backward layout (the non-causal
  // backward's Delta pass wrote it); the row kernel then only writes the padding.
  int delta_ready = 0;
  const int* imax = nullptr;  // tile skipping: last query tile of each key tile ([bh][nT]), or null
};

// Delta_i = dO_i . O_i = sum_j P_ij dP_ij for every query row of the non-causal backward,
// from S = Q K^T and dP = dO V^T on the tensor core and P recomputed from the forward's LSE
// (no O needed): writes delta[bh][i] for i < N (layout [BH][Npad]).
struct DeltaArgs {
  int B, N, H, d;
  float scale;
  const float* rowloc;
  const float* colrec;
  const float* lse;
  float* delta;
  uint32_t* err;
};
cudaError_t launch_delta_pass(const DeltaArgs& a, const CUtensorMap* maps /* q, k, v, dO (128-row boxes) */, int nT,
                              int Npad, cudaStream_t s);

// Delta/rho rows, dQ accumulator zeroing, the fused backward kernel, the dQ
// conversion and the reverse gate scan; the gate scan must already be in ws.
cudaError_t launch_attn_bwd(const AttnBwdArgs& a, const GateLayout& g, const BwdLayout& w,
                            const CUtensorMap* maps /* q (64-row box), k, v (128-row box), dO (64-row box),
                                                       dk, dv (128-row box, stored) */,
                            cudaStream_t s);

// Gate projection z = x W_f^T + b_f (tensor cores) fused with the tile scan, then the base
// scan: fills the same gate terms as launch_gate_scan and writes z when z_out is set.
// maps: x as [B, N, hidden] (box 64 x 128 x 1), W_f as [H, hidden] (box 64 x Hpad), both bf16,
// 128-byte swizzle; H <= 256.
cudaError_t launch_gate_proj_scan(const CUtensorMap* maps, const float* bias, int hidden, float* z_out, int B, int N,
                                  int H, int bias_from_j, void* ws, const GateLayout& g, cudaStream_t s,
                                  const V16Job* v16 = nullptr);

// Decay-aware tile skipping: per-tile norms of q and k, then the key-tile span of every
// query tile (jmin) and the query-tile span of every key tile (imax); needs the gate scan.
cudaError_t launch_tile_span(const void* q, const void* k, int B, int N, int H, int d, float scale,
                             const GateLayout& g, void* ws, cudaStream_t s);

// Epsilon-effective window per query row (fp64 prefix scan + binary search).
cudaError_t launch_window(const float* z, int B, int N, int H, double eps, int* out, void* ws, cudaStream_t s);
size_t window_workspace_bytes(int B, int N, int H);

// Host helper: 4-D bf16 tensor map over [B, N, H, d] with a box of 64 channels x 1 head x
// box_rows tokens x 1 batch and 128-byte swizzle. Returns false when the driver entry point is
// unavailable or encoding fails.
// fp32 3-D tensor map (d0 innermost; pitches of dims 1 and 2 in bytes), box (box0, box1, 1), no swizzle.
bool make_f32_3d_map(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t pitch1,
                     uint64_t pitch2, uint32_t box0, uint32_t box1);
bool make_bnhd_map(CUtensorMap* map, const void* base, int B, int N, int H, int d, int box_rows = kTile,
                   bool f16 = false);
// Host helpers for the gate projection: x [B, N, hidden] with a box of 64 x 128 x 1, and
// W_f [H, hidden] with a box of 64 x (H rounded up to 16); bf16, 128-byte swizzle.
bool make_x_map(CUtensorMap* map, const void* base, int B, int N, int hidden);
bool make_wf_map(CUtensorMap* map, const void* base, int H, int hidden);

}  // namespace fox
