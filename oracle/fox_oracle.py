"""CPU fp64 oracle for forget-gated causal softmax attention (FoX).

TEST INFRASTRUCTURE ONLY. This module is the plain, slow, obviously-correct
statement of what the CUDA path computes. Only the test suite, the smoke check
of the package entry file and the benchmark's CPU-baseline / reference arm may
import it; the library and its Python binding never do.

Sources (web pages, cited by title and section):
  [FoX-module]  "Forgetting Transformer (FoX) Attention" module source
                (frankenstein-transformer docs, fox_attn), class
                ForgettingAttention: module docstring formula and forward().
  [foxwindow]   foxwindow README, sections "The window is a first-passage time"
                and "ALiBi is the zero-variance limit".
  [foxwindow-len] foxwindow README, "The window is a first-passage time"
                (the epsilon-effective window) and "An exact two-moment law".
  [foxwindow-mono] foxwindow README, "The window is a first-passage time":
                every log f_t < 0, so the bias falls monotonically with the
                distance i - j (the basis of the tile-skip bound below).
  [fast-tf]     fast-transformers "Creating a custom attention layer",
                section "New Attention" (inputs already projected and split
                into heads; einsum layout "nlhe,nshe->nhls", i.e. [B, N, H, d]).

Notation: tokens t = 0..N-1 per (batch b, head h); a_t = log f_t with
f_t = sigmoid(z_t); c_t = sum_{l<=t} a_l; scale defaults to d^-1/2.

Readings taken where the pages are silent or disagree (each also a flag or a
fixed choice here):
  * Lower summation limit. The module docstring writes D_ij = sum_{l=j}^{i}
    log f_l; the module's code (cumsum then outer difference) and the foxwindow
    score form give sum_{l=j+1}^{i}. Both are implemented: bias_from_j=False
    (default) is j+1, so D_ii = 0; bias_from_j=True is j.
  * The module adds 1e-6 inside the log. The formula in both pages has no such
    term; the oracle uses the exact log-sigmoid.
  * The scale multiplies q.k only, never D (module forward()).
  * Causal by default (the module's "decoder" mode); causal=False is its
    "encoder" mode, where the same outer difference biases every key. No dropout.
  * LSE (not on the pages) is the natural-log normaliser of the biased,
    scaled scores, per row, layout [B, N, H].
  * z = +inf means f = 1 exactly (log f = 0).
  * The backward pass is not on the pages; it is the chain rule through the
    same forward formula.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "log_forget_gate",
    "cumulative_log_gate",
    "forget_bias",
    "attention_head",
    "attention_rows",
    "attention_head_blocked",
    "forward",
    "backward_head",
    "backward_head_blocked",
    "backward",
    "gate_grad_bruteforce",
    "gate_grad_from_sums",
    "default_scale",
    "effective_window",
    "tile_pair_bound",
    "tile_pair_excess",
    "tile_span",
    "SKIP_THRESHOLD_LOG2",
    "gate_projection",
]

# A causal (query tile, key tile) pair is skipped when the bound below says
# every weight in it is under 2^-150 of its row's largest weight. 2^-150 is
# past the smallest subnormal fp32 (2^-149); an fp32 exponential that flushes
# subnormals returns exactly 0 below 2^-126, so the 24 binary orders between
# the two cover the rounding of the quantities the bound is formed from.
SKIP_THRESHOLD_LOG2 = 150.0


LOG2E = 1.0 / math.log(2.0)


def default_scale(d: int) -> float:
    """d^-1/2 [FoX-module, __init__: scale = head_dim ** -0.5]."""
    return float(d) ** -0.5


def gate_projection(x, w_f, b_f) -> np.ndarray:
    """Gate logits z = x W_f^T + b_f, x [..., hidden] -> z [..., H], in fp64.

    [FoX-module, __init__: f_proj = Linear(hidden_size, num_heads, bias=True);
    forward(): f = sigmoid(f_proj(x))]. The Linear's weight is laid out
    [out_features, in_features] = [H, hidden]; this returns its pre-sigmoid
    output, the z every other function here takes. A library matmul is the step.
    """
    x = np.asarray(x, np.float64)
    w_f = np.asarray(w_f, np.float64)
    return x @ w_f.T + np.asarray(b_f, np.float64)


def log_forget_gate(z) -> np.ndarray:
    """a = log sigmoid(z) in fp64 [FoX-module, forward(): sigmoid of the gate
    projection, then its log].

    Evaluated as min(z, 0) - log1p(exp(-|z|)), which equals log(1/(1+e^-z))
    for every real z without overflow; z = +inf gives exactly 0.
    """
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        return np.minimum(z, 0.0) - np.log1p(np.exp(-np.abs(z)))


def cumulative_log_gate(a: np.ndarray) -> np.ndarray:
    """c_t = sum_{l<=t} a_l along the last axis [FoX-module, forward(): cumsum of log f]."""
    return np.cumsum(np.asarray(a, dtype=np.float64), axis=-1)


def forget_bias(a: np.ndarray, bias_from_j: bool = False) -> np.ndarray:
    """D [N, N] for one head, from its log gates a [N].

    j+1 convention: D_ij = sum_{l=j+1}^{i} a_l = c_i - c_j
        [FoX-module, forward(): outer difference of the cumsum;
         foxwindow, "The window is a first-passage time": score form].
    j convention:   D_ij = sum_{l=j}^{i} a_l = c_i - c_{j-1}, c_{-1} = 0
        [FoX-module, module docstring formula].
    Entries above the diagonal are returned as computed; the causal mask is
    applied by the caller.
    """
    c = cumulative_log_gate(a)
    col = c - a if bias_from_j else c
    return c[:, None] - col[None, :]


def attention_head(q, k, v, z, scale=None, bias_from_j=False, return_p=False, causal=True):
    """Forward of one (b, h): q, k, v [N, d], z [N] -> O [N, d], LSE [N].

    S_ij = scale * q_i . k_j + D_ij for j <= i, -inf for j > i
        [FoX-module, forward(): logits (q @ k^T) * scale + bias, causal
         triu(diagonal=1) mask set to -inf in decoder mode];
    causal=False is the module's "encoder" mode: no mask, so the same outer
    difference D_ij = c_i - c_j (positive for j > i) biases every key;
    LSE_i = M_i + ln sum_j exp(S_ij - M_i), M_i = max_j S_ij;
    P_ij = exp(S_ij - LSE_i) [FoX-module, forward(): softmax over keys];
    O_i = sum_j P_ij v_j [FoX-module, forward(): attn @ v].
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    N, d = q.shape
    if scale is None:
        scale = default_scale(d)
    if N == 0:
        empty = (np.zeros((0, v.shape[1])), np.zeros(0))
        return empty + (np.zeros((0, 0)),) if return_p else empty
    D = forget_bias(log_forget_gate(z), bias_from_j)
    S = scale * (q @ k.T) + D
    if causal:
        S[np.triu(np.ones((N, N), dtype=bool), k=1)] = -np.inf
    M = S.max(axis=1)
    lse = M + np.log(np.exp(S - M[:, None]).sum(axis=1))
    P = np.exp(S - lse[:, None])
    O = P @ v
    return (O, lse, P) if return_p else (O, lse)


def attention_rows(q, k, v, z, rows, scale=None, bias_from_j=False, causal=True):
    """The forward of one (b, h) restricted to the query rows `rows`.

    Row i of O and LSE depends only on row i of S, so this is the same
    definition as attention_head evaluated for the listed rows only (used for
    sequences too long to hold S whole).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    N, d = q.shape
    if scale is None:
        scale = default_scale(d)
    a = log_forget_gate(z)
    c = cumulative_log_gate(a)
    col = c - a if bias_from_j else c
    rows = np.asarray(rows, dtype=np.int64)
    O = np.empty((rows.size, v.shape[1]))
    lse = np.empty(rows.size)
    for n, i in enumerate(rows):
        last = i + 1 if causal else N
        s = scale * (k[:last] @ q[i]) + (c[i] - col[:last])
        m = s.max()
        lse[n] = m + np.log(np.exp(s - m).sum())
        O[n] = np.exp(s - lse[n]) @ v[:last]
    return O, lse


def _row_block_scores(q, k, c, col, r0, r1, scale, causal):
    """S of query rows r0..r1-1 against the keys they see, as attention_head forms it:
    scale * q_i . k_j + (c_i - colterm_j), with keys j > i set to -inf under the causal
    mask [FoX-module, forward()]. Causal rows r0..r1-1 see keys 0..r1-1 only, so the
    keys past r1 (all -inf for these rows) are left out. Returns (S, number of keys)."""
    last = r1 if causal else k.shape[0]
    S = scale * (q[r0:r1] @ k[:last].T) + (c[r0:r1, None] - col[None, :last])
    if causal:
        S[np.arange(r0, r1)[:, None] < np.arange(last)[None, :]] = -np.inf
    return S, last


def attention_head_blocked(q, k, v, z, scale=None, bias_from_j=False, causal=True, block=1024):
    """attention_head's forward of one (b, h), evaluated one block of query rows at a time.

    Row i of S (and so of P, O and LSE) depends only on q_i and the keys, so the
    definition applied to rows r0..r1-1 alone gives exactly those rows. Memory is
    O(block * N) instead of O(N^2): for sequences too long to hold S whole. The steps
    per block are attention_head's: biased scaled logits, causal mask, LSE, P, P @ v.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    N, d = q.shape
    if scale is None:
        scale = default_scale(d)
    a = log_forget_gate(z)
    c = cumulative_log_gate(a)
    col = _column_term(c, a, bias_from_j)
    O = np.empty((N, v.shape[1]))
    lse = np.empty(N)
    for r0 in range(0, N, block):
        r1 = min(N, r0 + block)
        S, last = _row_block_scores(q, k, c, col, r0, r1, scale, causal)
        M = S.max(axis=1)
        lse[r0:r1] = M + np.log(np.exp(S - M[:, None]).sum(axis=1))
        O[r0:r1] = np.exp(S - lse[r0:r1, None]) @ v[:last]
    return O, lse


def backward_head_blocked(q, k, v, z, dO, scale=None, bias_from_j=False, causal=True, block=1024,
                          return_sums=False):
    """backward_head's gradients of one (b, h), one block of query rows at a time.

    For rows r0..r1-1: S, LSE, P and O of those rows (attention_head_blocked), then the
    same chain rule as backward_head restricted to them:
      dP = dO_blk v^T,  Delta = rowsum(dO_blk * O_blk),  dS = P (dP - Delta),
      dQ_blk = scale dS k;  dV += P^T dO_blk;  dK += scale dS^T q_blk;
      R_blk = rowsum(dS);  C += colsum(dS).
    Every dS_ij lands in exactly one block (its row's), so the sums over blocks are
    backward_head's sums over i. The gate gradient is then gate_grad_from_sums(R, C, z).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dO = np.asarray(dO, np.float64)
    z = np.asarray(z, np.float64)
    N, d = q.shape
    if scale is None:
        scale = default_scale(d)
    a = log_forget_gate(z)
    c = cumulative_log_gate(a)
    col = _column_term(c, a, bias_from_j)
    dQ = np.empty((N, d))
    dK = np.zeros((N, d))
    dV = np.zeros((N, v.shape[1]))
    R = np.empty(N)
    C = np.zeros(N)
    for r0 in range(0, N, block):
        r1 = min(N, r0 + block)
        S, last = _row_block_scores(q, k, c, col, r0, r1, scale, causal)
        M = S.max(axis=1)
        lse = M + np.log(np.exp(S - M[:, None]).sum(axis=1))
        P = np.exp(S - lse[:, None])
        O = P @ v[:last]
        dP = dO[r0:r1] @ v[:last].T
        delta = (dO[r0:r1] * O).sum(axis=1)
        dS = P * (dP - delta[:, None])
        dQ[r0:r1] = scale * (dS @ k[:last])
        dV[:last] += P.T @ dO[r0:r1]
        dK[:last] += scale * (dS.T @ q[r0:r1])
        R[r0:r1] = dS.sum(axis=1)
        C[:last] += dS.sum(axis=0)
    dz = gate_grad_from_sums(R, C, z, bias_from_j)
    if return_sums:
        return dQ, dK, dV, dz, {"R": R, "C": C}
    return dQ, dK, dV, dz


def forward(q, k, v, z, scale=None, bias_from_j=False, causal=True):
    """Batched forward. q, k, v [B, N, H, d]; z [B, N, H] -> O [B, N, H, d], LSE [B, N, H].

    Layout per [fast-tf, "New Attention"]: inputs already projected and split
    into heads, [batch, length, heads, dim]; every (b, h) is independent.
    """
    q = np.asarray(q, np.float64)
    B, N, H, d = q.shape
    O = np.empty((B, N, H, v.shape[-1]))
    lse = np.empty((B, N, H))
    for b in range(B):
        for h in range(H):
            O[b, :, h], lse[b, :, h] = attention_head(
                q[b, :, h], k[b, :, h], v[b, :, h], z[b, :, h], scale, bias_from_j, causal=causal
            )
    return O, lse


def backward_head(q, k, v, z, dO, scale=None, bias_from_j=False, return_sums=False, causal=True):
    """Gradients of one (b, h) by the chain rule through attention_head.

    dP_ij = dO_i . v_j;  Delta_i = dO_i . O_i;  dS_ij = P_ij (dP_ij - Delta_i)
    dV_j = sum_i P_ij dO_i;  dQ_i = scale sum_j dS_ij k_j;  dK_j = scale sum_i dS_ij q_i
    Gate: R_i = sum_j dS_ij (row sums), C_j = sum_i dS_ij (column sums).
      j+1: d a_t = sum_{s>=t} (R_s - C_s)
      j  : d a_t = sum_{s>=t} (R_s - C_s) + C_t
    (a reverse prefix sum; gate_grad_bruteforce states the same quantity as
    the double sum over the entries of D that contain a_t). Without the causal
    mask the same formula holds: D_ij = c_i - c_j contains +a_t when j < t <= i
    and -a_t when i < t <= j, and both parts telescope into the suffix sums. And
    dz_t = d a_t * sigmoid(-z_t), since d/dz log sigmoid(z) = sigmoid(-z).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dO = np.asarray(dO, np.float64)
    z = np.asarray(z, np.float64)
    N, d = q.shape
    if scale is None:
        scale = default_scale(d)
    O, lse, P = attention_head(q, k, v, z, scale, bias_from_j, return_p=True, causal=causal)
    dP = dO @ v.T
    delta = (dO * O).sum(axis=1)
    dS = P * (dP - delta[:, None])
    dV = P.T @ dO
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q)
    R = dS.sum(axis=1)
    C = dS.sum(axis=0)
    suffix = np.cumsum((R - C)[::-1])[::-1]
    da = suffix + C if bias_from_j else suffix
    with np.errstate(over="ignore"):
        sig_neg = 1.0 / (1.0 + np.exp(z))  # sigmoid(-z); exactly 0 at z = +inf
    dz = da * sig_neg
    if return_sums:
        return dQ, dK, dV, dz, {"R": R, "C": C, "dS": dS, "da": da, "O": O, "lse": lse, "P": P}
    return dQ, dK, dV, dz


def gate_grad_bruteforce(dS: np.ndarray, bias_from_j: bool = False) -> np.ndarray:
    """d a_t as the plain double sum over the bias entries that contain a_t.

    j+1: D_ij = c_i - c_j holds +a_t iff j < t <= i (and -a_t iff i < t <= j,
         which only entries above the diagonal have), so
         d a_t = sum_{i>=t} sum_{j<t} dS_ij - sum_{i<t} sum_{j>=t} dS_ij.
    j  : D_ij = c_i - c_{j-1} holds +a_t iff j <= t <= i (and -a_t iff
         i < t < j), so d a_t = sum_{i>=t} sum_{j<=t} dS_ij - sum_{i<t} sum_{j>t} dS_ij.
    Under the causal mask dS is zero above the diagonal and the second sums vanish.
    O(N^3); for small N only.
    """
    N = dS.shape[0]
    da = np.zeros(N)
    for t in range(N):
        split = t + 1 if bias_from_j else t  # keys j < split take +a_t (for rows i >= t)
        da[t] = dS[t:, :split].sum() - dS[:t, split:].sum()
    return da


def gate_grad_from_sums(R, C, z, bias_from_j: bool = False) -> np.ndarray:
    """dz of one (b, h) from the row sums R and column sums C of dS, z [N].

    The gate part of backward_head on its own ([FoX-module] forward: D_ij = c_i - c_j
    with c the cumsum of log sigmoid(z); chain rule):
      j+1: d a_t = sum_{s>=t} (R_s - C_s);   j: d a_t = sum_{s>=t} (R_s - C_s) + C_t;
      dz_t = d a_t * sigmoid(-z_t).
    """
    R = np.asarray(R, np.float64)
    C = np.asarray(C, np.float64)
    z = np.asarray(z, np.float64)
    da = np.zeros(R.shape[0])
    run = 0.0
    for t in range(R.shape[0] - 1, -1, -1):  # the suffix sum, one term at a time
        run += R[t] - C[t]
        da[t] = run + C[t] if bias_from_j else run
    with np.errstate(over="ignore"):
        sig_neg = 1.0 / (1.0 + np.exp(z))  # sigmoid(-z); exactly 0 at z = +inf
    return da * sig_neg


def backward(q, k, v, z, dO, scale=None, bias_from_j=False, causal=True):
    """Batched backward over [B, N, H, d]: returns dQ, dK, dV [B, N, H, d], dz [B, N, H]."""
    q = np.asarray(q, np.float64)
    B, N, H, d = q.shape
    dQ = np.empty((B, N, H, d))
    dK = np.empty((B, N, H, d))
    dV = np.empty((B, N, H, v.shape[-1]))
    dz = np.empty((B, N, H))
    for b in range(B):
        for h in range(H):
            dQ[b, :, h], dK[b, :, h], dV[b, :, h], dz[b, :, h] = backward_head(
                q[b, :, h], k[b, :, h], v[b, :, h], z[b, :, h], dO[b, :, h], scale, bias_from_j, causal=causal
            )
    return dQ, dK, dV, dz


def effective_window(z, eps: float, rows=None) -> np.ndarray:
    """Epsilon-effective window of every query row of one head, z [N] -> int64 [N].

    [foxwindow-len]: with the positive increments X_t = -log g_t (g = sigmoid(z)),
    row i's window is the first-passage index of the walk read back from i,
        N_i(eps) = inf{ n >= 1 : X_i + X_{i-1} + ... + X_{i-n+1} > L },  L = ln(1/eps),
    i.e. one more than the largest distance n whose decay prod_{t=i-n+1..i} g_t is
    still >= eps (the page names the latter "the largest distance with D >= eps" and
    the former the first-passage index; this returns the first-passage index). The walk
    has i+1 increments; if their sum never exceeds L the window is not reached inside
    the sequence and the entry is -1.
    Evaluated literally: accumulate the increments from i backwards until the sum
    passes L. O(N * window); for tests. With `rows`, only those rows are evaluated
    (each row's window is defined on its own); the result then has len(rows) entries.
    """
    X = -log_forget_gate(z)
    L = math.log(1.0 / eps)
    N = X.shape[0]
    rows = range(N) if rows is None else [int(r) for r in rows]
    out = np.full(len(rows), -1, dtype=np.int64)
    for o, i in enumerate(rows):
        acc = 0.0
        for n in range(1, i + 2):
            acc += X[i - n + 1]
            if acc > L:
                out[o] = n
                break
    return out


def _column_term(c: np.ndarray, a: np.ndarray, bias_from_j: bool) -> np.ndarray:
    """The key-side term of D: D_ij = c_i - colterm_j [FoX-module, forward()]:
    colterm_j = c_j (j+1 convention) or c_{j-1} = c_j - a_j (j convention)."""
    return c - a if bias_from_j else c


def tile_pair_bound(q, k, z, scale=None, bias_from_j=False, tile=128) -> np.ndarray:
    """Upper bound U[I, J] (log2 units) on x_ij - M_i over query tile I and key tile J < I
    of one head (q, k [N, d], z [N]); +inf where J >= I. x_ij = (scale q_i.k_j + D_ij) log2 e
    and M_i = max_{j<=i} x_ij is the row's largest causal logit.

    [foxwindow-mono]: a_t <= 0, so colterm_t is non-increasing in t. With i in
    tile I (i >= i0, its first row) and j in tile J (j <= j1, its last key),
        x_ij - M_i <= x_ij - x_ii = scale log2e (q_i.k_j - q_i.k_i) + (colterm_i - colterm_j) log2e
                   <= |scale| log2e qmax_I (kmax_J + kmax_I) + (colterm_{i0} - colterm_{j1}) log2e
    (Cauchy-Schwarz on both dot products; qmax_T, kmax_T = largest row norm of q, k
    in tile T). kmax_J is replaced by the largest kmax over tiles 0..J, which keeps the
    bound valid and makes it non-increasing as J moves back from the diagonal."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    N, d = q.shape
    if scale is None:
        scale = default_scale(d)
    a = log_forget_gate(z)
    colterm = _column_term(cumulative_log_gate(a), a, bias_from_j)
    nT = (N + tile - 1) // tile
    qn = np.sqrt((q * q).sum(axis=1))
    kn = np.sqrt((k * k).sum(axis=1))
    qmax = np.array([qn[T * tile:(T + 1) * tile].max() for T in range(nT)])
    kmax = np.array([kn[T * tile:(T + 1) * tile].max() for T in range(nT)])
    kpre = np.maximum.accumulate(kmax)
    s2 = abs(scale) * LOG2E
    U = np.full((nT, nT), np.inf)
    for I in range(nT):
        for J in range(I):
            U[I, J] = s2 * qmax[I] * (kpre[J] + kmax[I]) + (colterm[I * tile] - colterm[J * tile + tile - 1]) * LOG2E
    return U


def tile_pair_excess(q, k, z, scale=None, bias_from_j=False, tile=128) -> np.ndarray:
    """The exact quantity tile_pair_bound bounds: E[I, J] = max over rows i (< N) of
    tile I and keys j of tile J with j <= i of x_ij - M_i (log2 units), from the full
    fp64 logits of attention_head; -inf where the pair holds no causal entry. Brute
    force; for tests."""
    q = np.asarray(q, np.float64)
    N, d = q.shape
    if scale is None:
        scale = default_scale(d)
    D = forget_bias(log_forget_gate(z), bias_from_j)
    X = (scale * (q @ np.asarray(k, np.float64).T) + D) * LOG2E
    X[np.triu(np.ones((N, N), dtype=bool), k=1)] = -np.inf
    M = X.max(axis=1)
    nT = (N + tile - 1) // tile
    E = np.full((nT, nT), -np.inf)
    for I in range(nT):
        rows = slice(I * tile, min(N, (I + 1) * tile))
        for J in range(I + 1):
            cols = slice(J * tile, min(N, (J + 1) * tile))
            E[I, J] = (X[rows, cols] - M[rows, None]).max()
    return E


def tile_span(q, k, z, scale=None, bias_from_j=False, tile=128, threshold=SKIP_THRESHOLD_LOG2):
    """Key-tile span of every query tile under the tile-skip rule, one head.

    Pair (I, J), J < I, is negligible when tile_pair_bound U[I, J] < -threshold.
    U is non-increasing as J moves back from the diagonal, so the negligible key tiles
    of query tile I are J < jraw(I) (jraw(I) = 0 if there are none). To give every key
    tile a contiguous range of query tiles, the start is made non-decreasing in I:
        jmin(I) = min_{I' >= I} jraw(I')   (this only keeps more pairs than jraw does),
        imax(J) = max{ I : jmin(I) <= J }  (>= J, since jmin(J) <= J).
    Query tile I then visits key tiles jmin(I)..I and key tile J serves query tiles
    J..imax(J). Returns (jmin, imax), int64 [nT] each."""
    U = tile_pair_bound(q, k, z, scale, bias_from_j, tile)
    nT = U.shape[0]
    jraw = np.zeros(nT, dtype=np.int64)
    for I in range(nT):
        for J in range(I - 1, -1, -1):
            if U[I, J] < -threshold:
                jraw[I] = J + 1
                break
    jmin = np.minimum.accumulate(jraw[::-1])[::-1].copy()
    imax = np.array([max(I for I in range(nT) if jmin[I] <= J) for J in range(nT)], dtype=np.int64)
    return jmin, imax
