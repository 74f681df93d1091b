/*
 * fox.h — C ABI of the forget-gated causal softmax attention library (libfox.so).
 *
 * The operation (Forgetting Transformer, FoX). Per batch b and head h, with
 * tokens t = 0..N-1:
 *   f_t = sigmoid(z_t),  a_t = log f_t,  c_t = sum_{l<=t} a_l
 *   D_ij = c_i - c_j          (bias_from_j = 0, the default; D_ii = 0)
 *   D_ij = c_i - c_{j-1}      (bias_from_j = 1; c_{-1} = 0)
 *   S_ij = scale * q_i . k_j + D_ij  for j <= i  (causal; j > i excluded unless non_causal)
 *   LSE_i = ln sum_{j<=i} exp(S_ij),  O_i = sum_{j<=i} exp(S_ij - LSE_i) v_j
 * Sources: "Forgetting Transformer (FoX) Attention" module source
 * (frankenstein-transformer docs, fox_attn: module docstring formula and
 * ForgettingAttention.forward — sigmoid gate, log, cumsum, outer difference,
 * causal mask, scaled logits + bias, softmax, attn @ v); foxwindow README,
 * "The window is a first-passage time" (score form with the sum from j+1);
 * fast-transformers "Creating a custom attention layer", "New Attention"
 * (attention-only call on projected, head-split inputs, [batch, length,
 * heads, dim] layout). The backward is the chain rule through the same
 * formula; the gate gradient is d a_t = sum_{s>=t} (R_s - C_s) (+ C_t under
 * bias_from_j = 1), R/C the row/column sums of dS, and dz_t = d a_t * sigmoid(-z_t).
 *
 * Layout (all row-major, contiguous, device memory):
 *   q, k, v, o, dO, dq, dk, dv : [B, N, H, d], element type per params.dtype
 *   z, lse, dz                  : [B, N, H] fp32
 * Alignment: q, k, v, o, dO, dq, dk, dv 16-byte aligned; z, lse, dz 4-byte
 * aligned; workspace 256-byte aligned.
 *
 * Ownership and threading: the caller owns every buffer, the workspace
 * included. The library allocates no device memory, keeps no state between
 * calls except a lazily-resolved driver entry point, and never synchronises
 * (fox_check_error excepted). All work is enqueued on `stream` (a
 * cudaStream_t; NULL means the legacy default stream) of the current device.
 * Outputs are fully overwritten. Calls on different streams must use
 * different workspaces.
 *
 * Errors: every call validates its arguments on the host and returns a
 * fox_status without touching the GPU when they are wrong. Device-side waits
 * are bounded; a wait that gives up sets a bit in the workspace's error word
 * (reset by each fox_fwd / fox_bwd call) and the kernel exits cleanly;
 * fox_check_error reports it.
 */
#ifndef FOX_H_
#define FOX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fox_status {
  FOX_OK = 0,
  FOX_ERR_INVALID_ARG = 1, /* null pointer, negative size, misalignment, bad flag or dtype */
  FOX_ERR_UNSUPPORTED = 2, /* well-formed but not implemented (d not in {64, 128}; fp32 backward;
                              non_causal or tile_skip with fp32; tile_skip with non_causal) */
  FOX_ERR_WORKSPACE = 3,   /* workspace null, misaligned or smaller than the size query */
  FOX_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  FOX_ERR_TIMEOUT = 5,     /* a device-side bounded wait gave up (from fox_check_error) */
  FOX_ERR_DEVICE = 6       /* another device-side error bit was set (from fox_check_error), e.g. a
                              V value outside the fp16 range of the forward's P V product */
} fox_status;

enum { FOX_DTYPE_BF16 = 0, FOX_DTYPE_F32 = 1 };

typedef struct fox_params {
  int B;           /* batch size, >= 0 */
  int N;           /* sequence length, >= 0 (any value; no multiple-of-tile requirement) */
  int H;           /* heads, >= 0; q, k and v have the same head count */
  int d;           /* head dimension: 64 or 128 */
  int dtype;       /* FOX_DTYPE_BF16 (tensor cores) or FOX_DTYPE_F32 (forward only) */
  float scale;     /* multiplies q.k only; 0 selects d^-1/2 (module __init__: head_dim ** -0.5) */
  int bias_from_j; /* 0: D_ij = sum_{l=j+1}^{i} log f_l (module code, foxwindow); 1: sum_{l=j}^{i} (module docstring) */
  int non_causal;  /* 0: causal (the module's "decoder" mode, the default); 1: every key, the module's
                      "encoder" mode, where the same outer difference D_ij = c_i - c_j (positive for
                      j > i) biases keys after the query too. bf16 forward and backward only. */
  int tile_skip;   /* 0: visit every causal tile pair (default). 1: skip the (query tile, key tile)
                      pairs whose every weight the decay bound puts below 2^-150 of its row's
                      largest (see fox_tile_span); outputs are bit-identical to tile_skip = 0 for
                      the forward, dK and dV, and equal up to the order of fp32 atomic sums for dQ
                      and dz. Causal bf16 only (FOX_ERR_UNSUPPORTED otherwise). */
  int gate_ready;  /* fox_bwd only (ignored elsewhere). 0: the backward runs its own gate scan (default).
                      1: the workspace already holds the gate terms of this z, written by a fox_fwd
                      (or fox_fwd_xgate, fox_gate_proj, fox_gate_scan) call with the same B, N, H and
                      bias_from_j on the same workspace, and nothing has written the workspace since:
                      the backward skips the scan and reads them. The workspace must then be at least
                      the larger of the fox_fwd and fox_bwd sizes. The backward also leaves the
                      workspace's error word as the forward left it (errors of both calls accumulate
                      until fox_check_error clears them). With a workspace that does not hold them, the
                      results are wrong (nothing faults: every index comes from B, N, H). */
} fox_params;

/*
 * Workspace bytes for these params (0 if params are invalid).
 * fox_fwd_workspace_bytes: the gate terms plus, for bf16, an fp16 copy of V
 *   (B*N*H*d*2 bytes), which fox_fwd writes once and the attention kernel reads.
 * fox_fwd_min_workspace_bytes: the gate terms alone, the least fox_fwd accepts.
 *   With less than fox_fwd_workspace_bytes the attention kernel converts every
 *   V tile it loads on chip instead (same results, bit for bit; slower).
 * fox_bwd_workspace_bytes: everything fox_bwd needs (more than the forward's).
 */
size_t fox_fwd_workspace_bytes(const fox_params* p);
size_t fox_fwd_min_workspace_bytes(const fox_params* p);
size_t fox_bwd_workspace_bytes(const fox_params* p);

/*
 * Forward. Reads q, k, v [B,N,H,d] and gate logits z [B,N,H] (fp32; +inf
 * allowed and means f = 1; -inf and NaN are outside the domain). Writes
 * O [B,N,H,d] (params.dtype; bf16 rounded to nearest even) and
 * LSE [B,N,H] (fp32, natural log, bias included).
 * Steps: gate log-sigmoid + per-head prefix scan into the workspace, V to fp16
 * into the workspace (when it has room, see above), then the fused causal
 * attention kernel. B*H == 0 or N == 0 returns FOX_OK with no work.
 * Workspace: at least fox_fwd_min_workspace_bytes(p), else FOX_ERR_WORKSPACE.
 * Precision (bf16): S = Q K^T in bf16 with fp32 accumulation, the softmax in
 * fp32, and P V in fp16 (P on chip and V converted to fp16, fp32 accumulation),
 * so that the weights carry 11 significant bits instead of bf16's 8. Every bf16
 * V value of magnitude 2^-14 .. 65280 converts exactly; smaller ones round to a
 * multiple of 2^-24; a V value of magnitude 65536 or more sets a device error
 * bit (fox_check_error then returns FOX_ERR_DEVICE).
 */
fox_status fox_fwd(const fox_params* p, const void* q, const void* k, const void* v, const float* z, void* o,
                   float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Gate projection ("Forgetting Transformer (FoX) Attention" module source:
 * f_proj = Linear(hidden_size, num_heads, bias=True), f = sigmoid(f_proj(x))):
 *   z[b,t,h] = sum_e x[b,t,e] W_f[h,e] + b_f[h]
 * x: [B,N,hidden] bf16. W_f: [H,hidden] bf16 (the Linear's weight layout).
 * b_f: [H] fp32. z: [B,N,H] fp32. All arrays are device pointers.
 * One kernel computes the 128-token x H blocks of z on the tensor cores
 * (fp32 accumulation) and runs the gate scan of fox_fwd on them in the same
 * pass, so fox_fwd_xgate's gate terms never round-trip through z.
 * Requires dtype bf16, hidden a positive multiple of 8, and H <= 256.
 * Workspace: fox_fwd_workspace_bytes(p) (its gate terms are also written).
 */
fox_status fox_gate_proj(const fox_params* p, int hidden, const void* x, const void* w_f, const float* b_f, float* z,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward from the layer input's gate projection instead of z: the fused
 * projection + gate scan above, then the attention as in fox_fwd. Writes
 * O, LSE and, when z is not null, z for the backward (fox_bwd takes z).
 * The same requirements as fox_gate_proj apply; tile_skip is honoured.
 */
fox_status fox_fwd_xgate(const fox_params* p, int hidden, const void* q, const void* k, const void* v, const void* x,
                         const void* w_f, const float* b_f, float* z, void* o, float* lse, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * Backward (bf16 only). Reads q, k, v, z, the forward's O and LSE, and the
 * upstream gradient dO; writes dq, dk, dv [B,N,H,d] bf16 and dz [B,N,H] fp32.
 * Steps: gate scan (skipped with p->gate_ready), the fp32 dQ accumulator in the
 * workspace cleared (a stream-ordered cudaMemsetAsync), Delta_i = dO_i . O_i,
 * the fused recompute-and-backward attention kernel (dK, dV, dQ accumulator and
 * the row and column sums of dS), the dQ conversion and the reverse gate scan
 * (one pass: a decoupled look-back across 128-token blocks or, with at least
 * one (b, 4-head) sequence per SM, one CTA walking each whole sequence).
 * With non_causal = 1, Delta is not taken from the bf16 O: a pass of its own
 * forms Delta_i = sum_j P_ij dP_ij from S = Q K^T and dP = dO V^T with P
 * recomputed from LSE, in fp32 (the gate gradient is a small difference of
 * large sums of dS there, and the bf16 rounding of O moves it by percents).
 * The extra pass costs about one forward.
 */
fox_status fox_bwd(const fox_params* p, const void* q, const void* k, const void* v, const float* z, const void* o,
                   const float* lse, const void* dO, void* dq, void* dk, void* dv, float* dz, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * The gate step alone: log f_t = log sigmoid(z_t) and its prefix sum along the
 * sequence per (b, h) ("Forgetting Transformer (FoX) Attention" module source,
 * ForgettingAttention.forward: sigmoid of the gate logits, log, cumsum), as the
 * first launches of fox_fwd and fox_bwd compute them. The gate terms are left in
 * the workspace; when c is not NULL the cumulative log gate
 *   c[b,t,h] = sum_{l<=t} log sigmoid(z[b,l,h])   (natural log, fp32, [B,N,H])
 * is written as well. No later call reads the workspace's gate terms (fox_fwd and
 * fox_bwd always recompute them): the call exists to check and time this step on
 * its own, at sizes where the attention itself would not fit. Only B, N, H and
 * bias_from_j are read from p. z is [B,N,H] fp32. Workspace:
 * fox_gate_scan_workspace_bytes(p) (the same as fox_fwd's for the same B, N, H).
 */
size_t fox_gate_scan_workspace_bytes(const fox_params* p);
fox_status fox_gate_scan(const fox_params* p, const float* z, float* c, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * The gate gradient from the row and column sums of dS, the last step of
 * fox_bwd: with R[b,h,t] = sum_j dS_tj and C[b,h,t] = sum_i dS_it,
 *   d a_t = sum_{s>=t} (R_s - C_s)          (bias_from_j = 0)
 *   d a_t = sum_{s>=t} (R_s - C_s) + C_t    (bias_from_j = 1)
 *   dz[b,t,h] = d a_t * sigmoid(-z[b,t,h])  (d/dz log sigmoid(z) = sigmoid(-z))
 * (chain rule through D_ij = c_i - c_j of the module's forward; the suffix form
 * holds with or without the causal mask). R, C: [B,H,N] fp32, each (b, h) row
 * contiguous; z, dz: [B,N,H] fp32. The sums are fp32 within 128-token blocks and
 * double-float (two fp32 values, about 48 bits) across them. Only B, N, H and
 * bias_from_j are read from p. Workspace (block sums): fox_gate_bwd_workspace_bytes(p).
 */
size_t fox_gate_bwd_workspace_bytes(const fox_params* p);
fox_status fox_gate_bwd(const fox_params* p, const float* z, const float* R, const float* C, float* dz,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Epsilon-effective window of every query row (foxwindow README, "The window is
 * a first-passage time"): with X_t = -log sigmoid(z_t) and L = ln(1/eps),
 *   window[b,i,h] = inf{ n >= 1 : X_i + X_{i-1} + ... + X_{i-n+1} > L },
 * one more than the largest distance n whose decay prod_{t=i-n+1..i} f_t is
 * still >= eps; -1 if the whole prefix (n = i+1) does not pass L. Uses the
 * score form's sum from j+1 (bias_from_j, d, dtype and scale are ignored).
 * z is [B,N,H] fp32, window [B,N,H] int32; 0 < eps < 1. The prefix sums and
 * the comparisons are fp64. Workspace: fox_window_workspace_bytes(p).
 */
size_t fox_window_workspace_bytes(const fox_params* p);
fox_status fox_window(const fox_params* p, const float* z, double eps, int32_t* window, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * Tile spans of the decay-aware tile skip (tile_skip = 1). The bias falls
 * monotonically with distance because every log f_t < 0 (foxwindow README,
 * "The window is a first-passage time"). So for query tile I (rows
 * 128I..128I+127) and an earlier key tile J, in log2 units,
 *   U(I,J) = scale log2e qmax_I (kmax_{<=J} + kmax_I) + (colterm(128I) - colterm(128J+127)) log2e
 * bounds x_ij - max_j' x_ij' over the pair. Here:
 *   - qmax_T, kmax_T are the largest row norms of q, k in tile T;
 *   - kmax_{<=J} is the largest kmax over tiles 0..J;
 *   - colterm(t) = c_t, or c_{t-1} when bias_from_j = 1.
 * Pairs with U < -150 are skipped. Every weight in such a pair is then
 * below 2^-150 of its row's largest, and the kernels' flushing exp2 makes it
 * exactly 0. Outputs, int32 [B*H][nT] with nT = ceil(N/128):
 *   jmin[bh][I]  first key tile that query tile I visits. It is made
 *                non-decreasing in I by a suffix minimum, which only keeps
 *                more pairs.
 *   imax[bh][J]  last query tile that key tile J serves:
 *                the largest I with jmin[bh][I] <= J.
 * q, k: [B,N,H,d] bf16; z: [B,N,H] fp32; causal bf16 params only.
 * Workspace: fox_fwd_workspace_bytes(p). jmin and imax are device pointers,
 * written by stream-ordered copies.
 */
fox_status fox_tile_span(const fox_params* p, const void* q, const void* k, const float* z, int32_t* jmin,
                         int32_t* imax, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward without a caller-provided workspace, for callers that cannot
 * allocate device memory where they run this code (a plugin in a host
 * application that owns all device memory, a latency-bound loop that cannot
 * take an allocation's implicit synchronisation). The pages have no
 * counterpart: this is a library convenience, not part of the method.
 * Same arguments and results as fox_fwd, minus the workspace: the scratch
 * for the gate terms is a fixed array of fox_noalloc_scratch_bytes() (16 MiB)
 * compiled into the library, which every GPU that loads the library holds
 * until the process exits. Problems whose fox_fwd_min_workspace_bytes exceeds
 * it return FOX_ERR_WORKSPACE without touching the GPU; the fp16 copy of V is
 * used when fox_fwd_workspace_bytes fits too. Allocates nothing
 * (no cudaMalloc, cudaFree or allocating library call). The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture. All calls
 * share the one array and the last call's contents stay in it: each call
 * rewrites it completely (the error word included), and calls whose work
 * overlaps on the GPU race on it. The device address is cached per device for
 * the life of the process: a cudaDeviceReset() on a device destroys the array
 * with the context, and fox_fwd_noalloc must not be called on that device
 * again in the same process.
 */
fox_status fox_fwd_noalloc(const fox_params* p, const void* q, const void* k, const void* v, const float* z,
                           void* o, float* lse, void* stream);
size_t fox_noalloc_scratch_bytes(void);
/*
 * fox_check_error for fox_fwd_noalloc: synchronises `stream`, reads and clears
 * the error word of the fixed scratch array of the current device (the one the
 * last fox_fwd_noalloc on that device used), with fox_check_error's results.
 * Allocates nothing.
 */
fox_status fox_noalloc_check_error(void* stream);

/*
 * Synchronises `stream`, reads and clears the device error word of
 * `workspace` (the one passed to the last fox_fwd / fox_bwd on it).
 * Returns FOX_OK, FOX_ERR_TIMEOUT or FOX_ERR_DEVICE, or FOX_ERR_CUDA if the
 * stream itself reports an error.
 */
fox_status fox_check_error(void* workspace, void* stream);

/*
 * Self-test of the device-side error path (the pages have no counterpart: this
 * checks the library's own failure reporting). One kernel on `stream` waits on
 * an mbarrier that nothing arrives at, with the attention kernels' bounded-wait
 * code and a limit of limit_us microseconds (1 .. 100000), while a second wait
 * of 16x that limit must be released by the first one's abort flag. Afterwards
 * the workspace's error word holds the timeout bit of the first wait only, so
 * fox_check_error(workspace, stream) returns FOX_ERR_TIMEOUT and clears it; the
 * next two 32-bit words of the header hold what each wait returned (0 = gave
 * up). Nothing faults; the context stays usable. workspace: >= 256 bytes,
 * 256-byte aligned (any fox_* workspace qualifies). Returns FOX_ERR_INVALID_ARG
 * for a limit out of range.
 */
fox_status fox_selftest_wait_timeout(unsigned limit_us, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Kernel-level timing, for benchmarks. Between fox_trace_begin() and
 * fox_trace_end(), every kernel launch this library enqueues (from any host
 * thread) is bracketed by two CUDA events recorded on its stream; events are
 * created on first use and reused. fox_trace_end() stops recording, waits for
 * the recorded events, writes up to max_records {kernel name, milliseconds}
 * in launch order into `out` (may be NULL), and returns the number of
 * launches recorded, or -1 if a CUDA event call failed. Names are static strings.
 */
typedef struct fox_trace_record {
  const char* kernel;
  float ms;
} fox_trace_record;
fox_status fox_trace_begin(void);
int fox_trace_end(fox_trace_record* out, int max_records);

/* Static string naming a status. */
const char* fox_status_string(fox_status s);

/* Library ABI version (major * 100 + minor). */
int fox_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FOX_H_ */
