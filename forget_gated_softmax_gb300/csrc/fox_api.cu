// C ABI of libfox.so: argument validation, workspace layout, TMA descriptor
// construction and kernel launches. See include/fox.h for the contract.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fox.h"
#include "fox_internal.h"

namespace fox {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

bool make_bnhd_map(CUtensorMap* map, const void* base, int B, int N, int H, int d, int box_rows, bool f16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2, (cuuint64_t)N * H * d * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  return enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base),
             dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_f32_3d_map(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t pitch1,
                     uint64_t pitch2, uint32_t box0, uint32_t box1) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {pitch1, pitch2};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_x_map(CUtensorMap* map, const void* base, int B, int N, int hidden) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)hidden, (cuuint64_t)N, (cuuint64_t)B};
  const cuuint64_t strides[2] = {(cuuint64_t)hidden * 2, (cuuint64_t)N * hidden * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_wf_map(CUtensorMap* map, const void* base, int H, int hidden) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)hidden, (cuuint64_t)H};
  const cuuint64_t strides[1] = {(cuuint64_t)hidden * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)((H + 15) / 16 * 16)};
  const cuuint32_t estr[2] = {1, 1};
  std::memset(map, 0, sizeof(*map));
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ tracing
namespace {
struct TraceRec {
  const char* name;
  cudaEvent_t start, stop;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace_pool;  // events are created once and reused
size_t g_trace_used = 0;
}  // namespace

bool trace_enabled() {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  return g_trace_on;
}

TraceScope::TraceScope(const char* name, cudaStream_t s) : stream(s) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (!g_trace_on) return;
  if (g_trace_used == g_trace_pool.size()) {
    TraceRec r{name, nullptr, nullptr};
    if (cudaEventCreate(&r.start) != cudaSuccess) return;
    if (cudaEventCreate(&r.stop) != cudaSuccess) {
      cudaEventDestroy(r.start);
      return;
    }
    g_trace_pool.push_back(r);
  }
  slot = static_cast<int>(g_trace_used++);
  g_trace_pool[slot].name = name;
  cudaEventRecord(g_trace_pool[slot].start, s);
}

TraceScope::~TraceScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  cudaEventRecord(g_trace_pool[slot].stop, stream);
}

}  // namespace fox

using namespace fox;

namespace {

constexpr long long kMaxTokens = (1LL << 31) - 1;

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Shape/flag checks shared by both directions. Pointers are checked separately.
fox_status check_params(const fox_params* p) {
  if (!p) return FOX_ERR_INVALID_ARG;
  if (p->B < 0 || p->N < 0 || p->H < 0 || p->d <= 0) return FOX_ERR_INVALID_ARG;
  if (p->dtype != FOX_DTYPE_BF16 && p->dtype != FOX_DTYPE_F32) return FOX_ERR_INVALID_ARG;
  if (p->bias_from_j != 0 && p->bias_from_j != 1) return FOX_ERR_INVALID_ARG;
  if (p->non_causal != 0 && p->non_causal != 1) return FOX_ERR_INVALID_ARG;
  if (p->tile_skip != 0 && p->tile_skip != 1) return FOX_ERR_INVALID_ARG;
  if (p->gate_ready != 0 && p->gate_ready != 1) return FOX_ERR_INVALID_ARG;
  if (!(p->scale >= 0.f) || std::isinf(p->scale)) return FOX_ERR_INVALID_ARG;
  if (p->d != 64 && p->d != 128) return FOX_ERR_UNSUPPORTED;
  if (p->tile_skip && (p->non_causal || p->dtype != FOX_DTYPE_BF16)) return FOX_ERR_UNSUPPORTED;
  const long long BH = (long long)p->B * p->H;
  if (BH > kMaxTokens || (long long)p->N > kMaxTokens - 2 * kTile) return FOX_ERR_INVALID_ARG;
  if (BH * (long long)p->N > kMaxTokens) return FOX_ERR_INVALID_ARG;
  return FOX_OK;
}

float effective_scale(const fox_params* p) { return p->scale == 0.f ? 1.f / std::sqrt((float)p->d) : p->scale; }

bool empty_problem(const fox_params* p) { return p->B == 0 || p->H == 0 || p->N == 0; }

fox_status check_workspace(void* ws, size_t bytes, size_t need) {
  if (!ws || !aligned(ws, 256) || bytes < need) return FOX_ERR_WORKSPACE;
  return FOX_OK;
}

}  // namespace

extern "C" {

int fox_version(void) { return 100; }

const char* fox_status_string(fox_status s) {
  switch (s) {
    case FOX_OK: return "FOX_OK";
    case FOX_ERR_INVALID_ARG: return "FOX_ERR_INVALID_ARG: invalid argument (null pointer, size, alignment or flag)";
    case FOX_ERR_UNSUPPORTED: return "FOX_ERR_UNSUPPORTED: head dimension, dtype or flag combination not implemented";
    case FOX_ERR_WORKSPACE: return "FOX_ERR_WORKSPACE: workspace null, misaligned or too small";
    case FOX_ERR_CUDA: return "FOX_ERR_CUDA: a CUDA call or kernel launch failed";
    case FOX_ERR_TIMEOUT: return "FOX_ERR_TIMEOUT: a device-side wait gave up";
    case FOX_ERR_DEVICE: return "FOX_ERR_DEVICE: device-side error bit set";
  }
  return "FOX_ERR_UNKNOWN";
}

size_t fox_fwd_min_workspace_bytes(const fox_params* p) {
  if (check_params(p) != FOX_OK) return 0;
  return gate_layout(p->B, p->N, p->H).end;
}

size_t fox_fwd_workspace_bytes(const fox_params* p) {
  if (check_params(p) != FOX_OK) return 0;
  const GateLayout g = gate_layout(p->B, p->N, p->H);
  if (p->dtype != FOX_DTYPE_BF16) return g.end;
  return fwd_v16_offset(g) + fwd_v16_bytes(p->B, p->N, p->H, p->d);
}

size_t fox_bwd_workspace_bytes(const fox_params* p) {
  if (check_params(p) != FOX_OK) return 0;
  const GateLayout g = gate_layout(p->B, p->N, p->H);
  return bwd_layout(g, p->d).end;
}

}  // extern "C"

namespace {

// Where the forward's fp16 copy of V goes (bf16 with a workspace that has room for it), or null:
// the attention kernel then converts each V tile on chip.
void* fwd_v16_slot(const fox_params* p, void* workspace, size_t workspace_bytes, const GateLayout& g) {
  if (p->dtype != FOX_DTYPE_BF16) return nullptr;
  if (workspace_bytes < fwd_v16_offset(g) + fwd_v16_bytes(p->B, p->N, p->H, p->d)) return nullptr;
  return static_cast<char*>(workspace) + fwd_v16_offset(g);
}

// The forward after the gate terms (and the fp16 copy of V, when v16 is set) are in the
// workspace: tile spans (tile_skip), then the attention kernel.
fox_status fwd_after_gate(const fox_params* p, const void* q, const void* k, const void* v, void* o, float* lse,
                          void* workspace, const void* v16, const GateLayout& g, cudaStream_t s) {
  if (p->tile_skip &&
      launch_tile_span(q, k, p->B, p->N, p->H, p->d, effective_scale(p), g, workspace, s) != cudaSuccess)
    return FOX_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  AttnFwdArgs a;
  a.B = p->B;
  a.N = p->N;
  a.H = p->H;
  a.d = p->d;
  a.scale = effective_scale(p);
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.rowloc = reinterpret_cast<const float*>(ws + g.rowloc);
  a.colrec = reinterpret_cast<const float*>(ws + g.colrec);
  a.err = reinterpret_cast<uint32_t*>(ws);
  a.non_causal = p->non_causal;
  if (p->tile_skip) a.jmin = reinterpret_cast<const int*>(ws + g.jmin);
  if (p->dtype == FOX_DTYPE_F32) {
    if (p->non_causal) return FOX_ERR_UNSUPPORTED;
    if (p->B * p->H > 65535) return FOX_ERR_UNSUPPORTED;
    return launch_attn_fwd_f32(a, g.nT, g.Npad, s) == cudaSuccess ? FOX_OK : FOX_ERR_CUDA;
  }
  a.v16 = v16;
  CUtensorMap maps[3];
  if (!make_bnhd_map(&maps[0], q, p->B, p->N, p->H, p->d) || !make_bnhd_map(&maps[1], k, p->B, p->N, p->H, p->d) ||
      !make_bnhd_map(&maps[2], a.v16 ? a.v16 : v, p->B, p->N, p->H, p->d, kTile, a.v16 != nullptr))
    return FOX_ERR_CUDA;
  return launch_attn_fwd_bf16(a, maps, g.nT, g.Npad, s) == cudaSuccess ? FOX_OK : FOX_ERR_CUDA;
}

// Checks and the fused projection + scan shared by fox_gate_proj and fox_fwd_xgate.
fox_status gate_proj(const fox_params* p, int hidden, const void* x, const void* w_f, const float* b_f, float* z,
                     void* workspace, size_t workspace_bytes, const GateLayout& g, cudaStream_t s,
                     const V16Job* v16 = nullptr) {
  if (p->dtype != FOX_DTYPE_BF16) return FOX_ERR_UNSUPPORTED;
  if (hidden <= 0 || hidden % 8 != 0) return FOX_ERR_INVALID_ARG;
  if (p->H > 256) return FOX_ERR_UNSUPPORTED;
  if ((long long)p->B * p->N * (long long)hidden > (1LL << 40)) return FOX_ERR_INVALID_ARG;
  if (!x || !w_f || !b_f) return FOX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_f, 16) || !aligned(b_f, 4) || (z && !aligned(z, 4))) return FOX_ERR_INVALID_ARG;
  fox_status st = check_workspace(workspace, workspace_bytes, g.end);
  if (st != FOX_OK) return st;
  CUtensorMap maps[2];
  if (!make_x_map(&maps[0], x, p->B, p->N, hidden) || !make_wf_map(&maps[1], w_f, p->H, hidden)) return FOX_ERR_CUDA;
  return launch_gate_proj_scan(maps, b_f, hidden, z, p->B, p->N, p->H, p->bias_from_j, workspace, g, s, v16) ==
                 cudaSuccess
             ? FOX_OK
             : FOX_ERR_CUDA;
}

}  // namespace

extern "C" {

fox_status fox_fwd(const fox_params* p, const void* q, const void* k, const void* v, const float* z, void* o,
                   float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  fox_status st = check_params(p);
  if (st != FOX_OK) return st;
  if (empty_problem(p)) return FOX_OK;
  if (!q || !k || !v || !z || !o || !lse) return FOX_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(z, 4) ||
      !aligned(lse, 4))
    return FOX_ERR_INVALID_ARG;
  const GateLayout g = gate_layout(p->B, p->N, p->H);
  st = check_workspace(workspace, workspace_bytes, g.end);
  if (st != FOX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* v16 = fwd_v16_slot(p, workspace, workspace_bytes, g);
  const V16Job job{v, v16, fwd_v16_bytes(p->B, p->N, p->H, p->d) / 2};
  if (launch_gate_scan(z, p->B, p->N, p->H, p->bias_from_j, workspace, g, s, v16 ? &job : nullptr) != cudaSuccess)
    return FOX_ERR_CUDA;
  return fwd_after_gate(p, q, k, v, o, lse, workspace, v16, g, s);
}

fox_status fox_gate_proj(const fox_params* p, int hidden, const void* x, const void* w_f, const float* b_f, float* z,
                         void* workspace, size_t workspace_bytes, void* stream) {
  fox_status st = check_params(p);
  if (st != FOX_OK) return st;
  if (empty_problem(p)) return FOX_OK;
  if (!z) return FOX_ERR_INVALID_ARG;
  const GateLayout g = gate_layout(p->B, p->N, p->H);
  return gate_proj(p, hidden, x, w_f, b_f, z, workspace, workspace_bytes, g, static_cast<cudaStream_t>(stream));
}

fox_status fox_fwd_xgate(const fox_params* p, int hidden, const void* q, const void* k, const void* v, const void* x,
                         const void* w_f, const float* b_f, float* z, void* o, float* lse, void* workspace,
                         size_t workspace_bytes, void* stream) {
  fox_status st = check_params(p);
  if (st != FOX_OK) return st;
  if (empty_problem(p)) return FOX_OK;
  if (!q || !k || !v || !o || !lse) return FOX_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FOX_ERR_INVALID_ARG;
  const GateLayout g = gate_layout(p->B, p->N, p->H);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* v16 = fwd_v16_slot(p, workspace, workspace_bytes, g);
  const V16Job job{v, v16, fwd_v16_bytes(p->B, p->N, p->H, p->d) / 2};
  st = gate_proj(p, hidden, x, w_f, b_f, z, workspace, workspace_bytes, g, s, v16 ? &job : nullptr);
  if (st != FOX_OK) return st;
  return fwd_after_gate(p, q, k, v, o, lse, workspace, v16, g, s);
}

fox_status fox_bwd(const fox_params* p, const void* q, const void* k, const void* v, const float* z, const void* o,
                   const float* lse, const void* dO, void* dq, void* dk, void* dv, float* dz, void* workspace,
                   size_t workspace_bytes, void* stream) {
  fox_status st = check_params(p);
  if (st != FOX_OK) return st;
  if (p->dtype != FOX_DTYPE_BF16) return FOX_ERR_UNSUPPORTED;
  if (empty_problem(p)) return FOX_OK;
  if (!q || !k || !v || !z || !o || !lse || !dO || !dq || !dk || !dv || !dz) return FOX_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dO, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(z, 4) || !aligned(lse, 4) ||
      !aligned(dz, 4))
    return FOX_ERR_INVALID_ARG;
  const GateLayout g = gate_layout(p->B, p->N, p->H);
  const BwdLayout w = bwd_layout(g, p->d);
  st = check_workspace(workspace, workspace_bytes, w.end);
  if (st != FOX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // With gate_ready the workspace holds the forward's gate terms of this z (the caller's contract).
  if (!p->gate_ready &&
      launch_gate_scan(z, p->B, p->N, p->H, p->bias_from_j, workspace, g, s) != cudaSuccess)
    return FOX_ERR_CUDA;
  if (p->tile_skip &&
      launch_tile_span(q, k, p->B, p->N, p->H, p->d, effective_scale(p), g, workspace, s) != cudaSuccess)
    return FOX_ERR_CUDA;
  CUtensorMap maps[6];
  if (!make_bnhd_map(&maps[0], q, p->B, p->N, p->H, p->d, 64) ||
      !make_bnhd_map(&maps[1], k, p->B, p->N, p->H, p->d, kTile) ||
      !make_bnhd_map(&maps[2], v, p->B, p->N, p->H, p->d, kTile) ||
      !make_bnhd_map(&maps[3], dO, p->B, p->N, p->H, p->d, 64) ||
      !make_bnhd_map(&maps[4], dk, p->B, p->N, p->H, p->d, kTile) ||
      !make_bnhd_map(&maps[5], dv, p->B, p->N, p->H, p->d, kTile))
    return FOX_ERR_CUDA;
  AttnBwdArgs a;
  a.B = p->B;
  a.N = p->N;
  a.H = p->H;
  a.d = p->d;
  a.bias_from_j = p->bias_from_j;
  a.non_causal = p->non_causal;
  a.scale = effective_scale(p);
  a.q = q;
  a.k = k;
  a.v = v;
  a.z = z;
  a.o = o;
  a.lse = lse;
  a.dO = dO;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dz = dz;
  a.ws = static_cast<char*>(workspace);
  if (p->tile_skip) a.imax = reinterpret_cast<const int*>(a.ws + g.imax);
  if (p->non_causal) {
    // Without the causal mask the gate gradient is a small difference of large
    // row and column sums of dS = P (dP - Delta), and a Delta_i = dO_i . O_i
    // taken from the bf16 O moves it by several percent. Form Delta_i as
    // sum_j P_ij dP_ij instead, from S = Q K^T and dP = dO V^T with P recomputed
    // from LSE, all in fp32 (O is not read).
    CUtensorMap dmaps[4];
    if (!make_bnhd_map(&dmaps[0], q, p->B, p->N, p->H, p->d) ||
        !make_bnhd_map(&dmaps[3], dO, p->B, p->N, p->H, p->d))
      return FOX_ERR_CUDA;
    dmaps[1] = maps[1];
    dmaps[2] = maps[2];
    DeltaArgs da;
    da.B = p->B;
    da.N = p->N;
    da.H = p->H;
    da.d = p->d;
    da.scale = a.scale;
    da.rowloc = reinterpret_cast<const float*>(a.ws + g.rowloc);
    da.colrec = reinterpret_cast<const float*>(a.ws + g.colrec);
    da.lse = lse;
    da.delta = reinterpret_cast<float*>(a.ws + w.delta);
    da.err = reinterpret_cast<uint32_t*>(a.ws);
    if (launch_delta_pass(da, dmaps, g.nT, g.Npad, s) != cudaSuccess) return FOX_ERR_CUDA;
    a.delta_ready = 1;
  }
  return launch_attn_bwd(a, g, w, maps, s) == cudaSuccess ? FOX_OK : FOX_ERR_CUDA;
}

fox_status fox_tile_span(const fox_params* p, const void* q, const void* k, const float* z, int32_t* jmin,
                         int32_t* imax, void* workspace, size_t workspace_bytes, void* stream) {
  fox_status st = check_params(p);
  if (st != FOX_OK) return st;
  if (p->dtype != FOX_DTYPE_BF16 || p->non_causal) return FOX_ERR_UNSUPPORTED;
  if (empty_problem(p)) return FOX_OK;
  if (!q || !k || !z || !jmin || !imax) return FOX_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(z, 4) || !aligned(jmin, 4) || !aligned(imax, 4))
    return FOX_ERR_INVALID_ARG;
  const GateLayout g = gate_layout(p->B, p->N, p->H);
  st = check_workspace(workspace, workspace_bytes, g.end);
  if (st != FOX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_gate_scan(z, p->B, p->N, p->H, p->bias_from_j, workspace, g, s) != cudaSuccess) return FOX_ERR_CUDA;
  if (launch_tile_span(q, k, p->B, p->N, p->H, p->d, effective_scale(p), g, workspace, s) != cudaSuccess)
    return FOX_ERR_CUDA;
  const char* ws = static_cast<const char*>(workspace);
  const size_t bytes = sizeof(int32_t) * (size_t)g.BH * g.nT;
  if (cudaMemcpyAsync(jmin, ws + g.jmin, bytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(imax, ws + g.imax, bytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return FOX_ERR_CUDA;
  return FOX_OK;
}

// Shape and flag checks of the gate-only calls (d, dtype, scale and the attention flags unused).
static fox_status check_gate_params(const fox_params* p) {
  if (!p || p->B < 0 || p->N < 0 || p->H < 0) return FOX_ERR_INVALID_ARG;
  if (p->bias_from_j != 0 && p->bias_from_j != 1) return FOX_ERR_INVALID_ARG;
  const long long BH = (long long)p->B * p->H;
  if (BH > kMaxTokens || (long long)p->N > kMaxTokens - 2 * kTile || BH * (long long)p->N > kMaxTokens)
    return FOX_ERR_INVALID_ARG;
  return FOX_OK;
}

size_t fox_gate_scan_workspace_bytes(const fox_params* p) {
  if (check_gate_params(p) != FOX_OK) return 0;
  return gate_layout(p->B, p->N, p->H).end;
}

fox_status fox_gate_scan(const fox_params* p, const float* z, float* c, void* workspace, size_t workspace_bytes,
                         void* stream) {
  fox_status st = check_gate_params(p);
  if (st != FOX_OK) return st;
  if (p->B == 0 || p->H == 0 || p->N == 0) return FOX_OK;
  if (!z || !aligned(z, 4) || (c && !aligned(c, 4))) return FOX_ERR_INVALID_ARG;
  const GateLayout g = gate_layout(p->B, p->N, p->H);
  st = check_workspace(workspace, workspace_bytes, g.end);
  if (st != FOX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_gate_scan(z, p->B, p->N, p->H, p->bias_from_j, workspace, g, s) != cudaSuccess) return FOX_ERR_CUDA;
  if (c && launch_gate_cumulative(workspace, g, p->B, p->N, p->H, c, s) != cudaSuccess) return FOX_ERR_CUDA;
  return FOX_OK;
}

size_t fox_gate_bwd_workspace_bytes(const fox_params* p) {
  if (check_gate_params(p) != FOX_OK) return 0;
  const size_t nT = ((size_t)p->N + kTile - 1) / kTile;
  return kErrWordBytes + align_up(kGateStatBytes * (size_t)p->B * p->H * nT, 256);
}

fox_status fox_gate_bwd(const fox_params* p, const float* z, const float* R, const float* C, float* dz,
                        void* workspace, size_t workspace_bytes, void* stream) {
  fox_status st = check_gate_params(p);
  if (st != FOX_OK) return st;
  if (p->B == 0 || p->H == 0 || p->N == 0) return FOX_OK;
  if (!z || !R || !C || !dz || !aligned(z, 4) || !aligned(R, 4) || !aligned(C, 4) || !aligned(dz, 4))
    return FOX_ERR_INVALID_ARG;
  const size_t need = fox_gate_bwd_workspace_bytes(p);
  st = check_workspace(workspace, workspace_bytes, need);
  if (st != FOX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  // the error word, and for the look-back kernel its ticket counter and status records, start at zero
  const bool seq = gate_bwd_streams(p->B, p->N, p->H, p->N, C, R, z, dz);
  if (cudaMemsetAsync(ws, 0, seq ? kErrWordBytes : need, s) != cudaSuccess) return FOX_ERR_CUDA;
  return launch_gate_bwd(p->B, p->N, p->H, p->N, p->bias_from_j, C, R, z, dz, ws + kErrWordBytes,
                         reinterpret_cast<unsigned*>(ws + kTicketOffset), reinterpret_cast<uint32_t*>(ws), s) ==
                 cudaSuccess
             ? FOX_OK
             : FOX_ERR_CUDA;
}

size_t fox_window_workspace_bytes(const fox_params* p) {
  if (!p || p->B < 0 || p->N < 0 || p->H < 0) return 0;
  if ((long long)p->B * p->H > kMaxTokens || (long long)p->B * p->H * (long long)p->N > kMaxTokens) return 0;
  return window_workspace_bytes(p->B, p->N, p->H);
}

fox_status fox_window(const fox_params* p, const float* z, double eps, int32_t* window, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!p || p->B < 0 || p->N < 0 || p->H < 0) return FOX_ERR_INVALID_ARG;
  if (!(eps > 0.0 && eps < 1.0)) return FOX_ERR_INVALID_ARG;
  const size_t need = fox_window_workspace_bytes(p);
  if (need == 0) return FOX_ERR_INVALID_ARG;
  if (p->B == 0 || p->H == 0 || p->N == 0) return FOX_OK;
  if (!z || !window || !aligned(z, 4) || !aligned(window, 4)) return FOX_ERR_INVALID_ARG;
  fox_status st = check_workspace(workspace, workspace_bytes, need);
  if (st != FOX_OK) return st;
  return launch_window(z, p->B, p->N, p->H, eps, window, workspace, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FOX_OK
             : FOX_ERR_CUDA;
}

fox_status fox_trace_begin(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = true;
  g_trace_used = 0;
  return FOX_OK;
}

int fox_trace_end(fox_trace_record* out, int max_records) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = false;
  const int n = static_cast<int>(g_trace_used);
  for (int i = 0; i < n; ++i) {
    if (cudaEventSynchronize(g_trace_pool[i].stop) != cudaSuccess) return -1;
    if (out && i < max_records) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, g_trace_pool[i].start, g_trace_pool[i].stop) != cudaSuccess) return -1;
      out[i].kernel = g_trace_pool[i].name;
      out[i].ms = ms;
    }
  }
  g_trace_used = 0;
  return n;
}

fox_status fox_check_error(void* workspace, void* stream) {
  if (!workspace || !aligned(workspace, 256)) return FOX_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FOX_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FOX_ERR_CUDA;
  if (word == 0) return FOX_OK;
  if (cudaMemsetAsync(workspace, 0, sizeof(word), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return FOX_ERR_CUDA;
  const uint32_t timeout_bits = 0x7u;
  return (word & timeout_bits) ? FOX_ERR_TIMEOUT : FOX_ERR_DEVICE;
}

}  // extern "C"
