"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties the oracle to something other than itself: a library routine
for a special case (torch scaled_dot_product_attention, scipy log_expit,
torch.logsumexp), a closed form, an invariant the pages state, or brute force
(finite differences, explicit sums) on tiny inputs. Chosen so that a dropped
term, a wrong sign, an off-by-one in the summation limit or a transposed
operand in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

from oracle import fox_oracle as ora

RNG = np.random.default_rng(12345)


def _rand_head(N, d, gate_mu=1.5, gate_sigma=1.0, seed=0):
    r = np.random.default_rng(seed)
    q, k, v, dO = (r.standard_normal((N, d)) for _ in range(4))
    z = gate_mu + gate_sigma * r.standard_normal(N)
    return q, k, v, z, dO


def _sdpa(q, k, v, scale, bias=None):
    """torch SDPA in fp64 on CPU, causal, with an optional additive bias."""
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64)[None, None] for x in (q, k, v))
    N = q.shape[0]
    if bias is None:
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=scale)
    else:
        mask = torch.tensor(bias, dtype=torch.float64)
        mask = mask.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask[None, None], scale=scale)
    return out[0, 0].numpy()


def _lse_lib(q, k, scale, bias):
    s = torch.tensor(scale * (q @ k.T) + bias, dtype=torch.float64)
    N = q.shape[0]
    s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    return torch.logsumexp(s, dim=1).numpy()


# ----------------------------------------------------------------- gate


def test_log_forget_gate_matches_scipy_log_expit():
    z = np.concatenate([np.linspace(-60, 60, 2001), [-1e-300, 0.0, 1e-300, 700.0, -700.0]])
    np.testing.assert_allclose(ora.log_forget_gate(z), scipy.special.log_expit(z), rtol=1e-14, atol=1e-300)


def test_log_forget_gate_special_values():
    assert ora.log_forget_gate(0.0) == pytest.approx(-math.log(2.0), rel=1e-15)
    assert ora.log_forget_gate(np.inf) == 0.0
    # far negative logit: log sigmoid(z) = z - log1p(e^z) -> z
    assert ora.log_forget_gate(-40.0) == pytest.approx(-40.0 - math.exp(-40.0), rel=1e-15)
    assert np.all(ora.log_forget_gate(np.linspace(-30, 30, 101)) < 0)


def test_bias_is_explicit_sum_of_log_gates():
    """D_ij against the sum written term by term (j+1: l = j+1..i; j: l = j..i)."""
    N = 11
    z = RNG.normal(1.0, 2.0, N)
    for from_j in (False, True):
        D = ora.forget_bias(ora.log_forget_gate(z), from_j)
        for i in range(N):
            for j in range(i + 1):
                lo = j if from_j else j + 1
                ref = sum(math.log(1.0 / (1.0 + math.exp(-z[l]))) for l in range(lo, i + 1))
                assert D[i, j] == pytest.approx(ref, abs=1e-13)


def test_bias_diagonal_and_strict_monotone_decrease_in_distance():
    """The bias falls strictly with distance i-j when every gate is below 1
    (foxwindow, "The window is a first-passage time")."""
    N = 200
    z = RNG.normal(3.0, 2.0, N)
    a = ora.log_forget_gate(z)
    D = ora.forget_bias(a, False)
    np.testing.assert_array_equal(np.diag(D), 0.0)
    np.testing.assert_allclose(np.diag(ora.forget_bias(a, True)), a, rtol=0, atol=1e-12)
    for i in range(N):
        row = D[i, : i + 1]  # j = 0..i, distance i-j shrinks as j grows
        assert np.all(np.diff(row) > 0)


# --------------------------------------------------------------- forward


@pytest.mark.parametrize("N,d", [(1, 4), (7, 3), (64, 16), (130, 32)])
def test_open_gate_is_causal_softmax_attention(N, d):
    """f = 1 (z = +inf) removes the bias: plain causal attention (torch SDPA)."""
    q, k, v, _, _ = _rand_head(N, d, seed=N)
    z = np.full(N, np.inf)
    for from_j in (False, True):
        O, lse = ora.attention_head(q, k, v, z, bias_from_j=from_j)
        np.testing.assert_allclose(O, _sdpa(q, k, v, d**-0.5), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, _lse_lib(q, k, d**-0.5, np.zeros((N, N))), rtol=0, atol=1e-12)


def test_custom_scale_applies_to_scores_only():
    N, d = 33, 8
    q, k, v, z, _ = _rand_head(N, d, seed=3)
    D = ora.forget_bias(ora.log_forget_gate(z))
    for scale in (0.1, 1.0, 2.5):
        O, lse = ora.attention_head(q, k, v, z, scale=scale)
        np.testing.assert_allclose(O, _sdpa(q, k, v, scale, D), atol=1e-12)
        np.testing.assert_allclose(lse, _lse_lib(q, k, scale, D), atol=1e-12)


@pytest.mark.parametrize("t0", [0, 1, 5, 12])
def test_single_closing_gate_is_a_block_bias(t0):
    """One gate f_t0 < 1, all others 1: the bias is log f_t0 exactly on the
    entries whose sum range contains t0 (j < t0 <= i for j+1; j <= t0 <= i for j).
    Library SDPA with that explicit block bias must agree. Pins the limit."""
    N, d = 13, 5
    q, k, v, _, _ = _rand_head(N, d, seed=7 + t0)
    z = np.full(N, np.inf)
    z[t0] = -0.7
    a0 = math.log(1.0 / (1.0 + math.exp(0.7)))
    for from_j in (False, True):
        bias = np.zeros((N, N))
        for i in range(N):
            for j in range(i + 1):
                inside = (j <= t0 <= i) if from_j else (j < t0 <= i)
                bias[i, j] = a0 if inside else 0.0
        O, lse = ora.attention_head(q, k, v, z, bias_from_j=from_j)
        np.testing.assert_allclose(O, _sdpa(q, k, v, d**-0.5, bias), atol=1e-12)
        np.testing.assert_allclose(lse, _lse_lib(q, k, d**-0.5, bias), atol=1e-12)


@pytest.mark.parametrize("m", [0.05, 0.1, 0.7071, 3.0])
def test_constant_gate_is_alibi(m):
    """Constant gate f = e^-m gives the bias -m(i-j) (foxwindow, "ALiBi is the
    zero-variance limit"); under the j convention the bias gains one more -m,
    which leaves O unchanged and lowers LSE by exactly m."""
    N, d = 96, 16
    q, k, v, _, _ = _rand_head(N, d, seed=int(m * 1000))
    z = np.full(N, -math.log(math.expm1(m)))  # sigmoid(z) = e^-m
    i, j = np.meshgrid(np.arange(N), np.arange(N), indexing="ij")
    alibi = -m * (i - j).astype(np.float64)
    O1, lse1 = ora.attention_head(q, k, v, z)
    np.testing.assert_allclose(O1, _sdpa(q, k, v, d**-0.5, alibi), atol=1e-11)
    np.testing.assert_allclose(lse1, _lse_lib(q, k, d**-0.5, alibi), atol=1e-11)
    O0, lse0 = ora.attention_head(q, k, v, z, bias_from_j=True)
    np.testing.assert_allclose(O0, O1, atol=1e-12)
    np.testing.assert_allclose(lse0, lse1 - m, atol=1e-11)


@pytest.mark.parametrize("m", [0.0, 0.05, 0.69, 2.0])
def test_constant_gate_closed_form(m):
    """q = k = 0, constant gate r = e^-m, v_j = j: the weights are geometric.
    LSE_i = ln sum_{s=0}^{i} r^s and O_i = i - (sum_s s r^s)/(sum_s r^s)."""
    N = 50
    q = np.zeros((N, 2))
    k = np.zeros((N, 2))
    v = np.arange(N, dtype=np.float64)[:, None]
    z = np.full(N, np.inf if m == 0.0 else -math.log(math.expm1(m)))
    O, lse = ora.attention_head(q, k, v, z)
    r = math.exp(-m)
    for i in range(N):
        if m == 0.0:
            G, K = i + 1.0, i * (i + 1) / 2.0
        else:
            G = (1 - r ** (i + 1)) / (1 - r)
            K = r * (1 - (i + 1) * r**i + i * r ** (i + 1)) / (1 - r) ** 2
        assert lse[i] == pytest.approx(math.log(G), abs=1e-12)
        assert O[i, 0] == pytest.approx(i - K / G, abs=1e-10)


def test_rows_sum_to_one_and_ones_in_ones_out():
    N, d = 70, 8
    q, k, v, z, _ = _rand_head(N, d, gate_mu=0.0, gate_sigma=3.0, seed=11)
    for from_j in (False, True):
        O, lse, P = ora.attention_head(q, k, v, z, bias_from_j=from_j, return_p=True)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-13)
        assert np.all(np.triu(P, 1) == 0)
        O1, _ = ora.attention_head(q, k, np.ones((N, 3)), z, bias_from_j=from_j)
        np.testing.assert_allclose(O1, 1.0, atol=1e-13)


def test_rows_variant_matches_whole_head():
    N, d = 150, 16
    q, k, v, z, _ = _rand_head(N, d, seed=5)
    rows = [0, 1, 63, 64, 127, 128, 149]
    for from_j in (False, True):
        O, lse = ora.attention_head(q, k, v, z, bias_from_j=from_j)
        Or, lr = ora.attention_rows(q, k, v, z, rows, bias_from_j=from_j)
        np.testing.assert_allclose(Or, O[rows], atol=1e-12)
        np.testing.assert_allclose(lr, lse[rows], atol=1e-12)


def test_batched_layout_matches_einsum_convention():
    """[B, N, H, d] in and out, as the einsum 'nlhe,nshe->nhls' / 'nhls,nshd->nlhd'
    of fast-transformers' "New Attention"; checked with f = 1 against einsum."""
    B, N, H, d = 2, 9, 3, 4
    r = np.random.default_rng(2)
    q, k, v = (r.standard_normal((B, N, H, d)) for _ in range(3))
    z = np.full((B, N, H), np.inf)
    O, lse = ora.forward(q, k, v, z)
    tq, tk, tv = (torch.tensor(x) for x in (q, k, v))
    s = torch.einsum("nlhe,nshe->nhls", tq, tk) * d**-0.5
    s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    ref = torch.einsum("nhls,nshd->nlhd", torch.softmax(s, -1), tv).numpy()
    np.testing.assert_allclose(O, ref, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).permute(0, 2, 1).numpy(), atol=1e-12)


def test_module_forward_reexpressed_in_torch():
    """Cross-check: the module's forward() steps (sigmoid, log, cumsum, outer
    difference, triu mask, scaled logits + bias, softmax, @ v) in torch fp64
    without the 1e-6 term, on projected inputs. Agrees with the j+1 reading."""
    N, d = 40, 8
    q, k, v, z, _ = _rand_head(N, d, seed=9)
    tq, tk, tv, tz = (torch.tensor(x) for x in (q, k, v, z))
    logf = torch.log(torch.sigmoid(tz))
    cum = torch.cumsum(logf, dim=-1)
    bias = cum.unsqueeze(-1) - cum.unsqueeze(-2)
    bias = bias.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    out = torch.softmax((tq @ tk.T) * d**-0.5 + bias, dim=-1) @ tv
    O, _ = ora.attention_head(q, k, v, z)
    np.testing.assert_allclose(O, out.numpy(), atol=1e-12)


def test_empty_sequence():
    O, lse = ora.attention_head(np.zeros((0, 4)), np.zeros((0, 4)), np.zeros((0, 4)), np.zeros(0))
    assert O.shape == (0, 4) and lse.shape == (0,)


# -------------------------------------------------------------- backward


def _loss(q, k, v, z, dO, from_j, scale=None):
    O, _ = ora.attention_head(q, k, v, z, scale=scale, bias_from_j=from_j)
    return float((O * dO).sum())


@pytest.mark.parametrize("from_j", [False, True])
@pytest.mark.parametrize("N", [1, 5, 16])
def test_backward_matches_central_differences(N, from_j):
    """Analytic dQ, dK, dV, dz against central differences of L = sum(O * dO) in fp64."""
    d = 4
    q, k, v, z, dO = _rand_head(N, d, gate_mu=0.5, gate_sigma=1.5, seed=100 + N)
    dQ, dK, dV, dz = ora.backward_head(q, k, v, z, dO, bias_from_j=from_j)
    h = 1e-6
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV), ("z", z, dz)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v, "z": z}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], args["z"], dO, from_j)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], args["z"], dO, from_j)
            num[idx] = (lp - lm) / (2 * h)
        # gradients that vanish identically (N = 1: q, k, z do not move O) are
        # checked against an absolute floor set by the difference quotient's rounding
        err = np.linalg.norm(num - g)
        assert err <= 1e-6 * np.linalg.norm(num) + 1e-8, (name, err, np.linalg.norm(num))


def test_backward_custom_scale_by_differences():
    N, d, scale = 6, 3, 0.37
    q, k, v, z, dO = _rand_head(N, d, seed=42)
    dQ, dK, _, _ = ora.backward_head(q, k, v, z, dO, scale=scale)
    h = 1e-6
    for x, g in ((q, dQ), (k, dK)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            if x is q:
                num[idx] = (_loss(xp, k, v, z, dO, False, scale) - _loss(xm, k, v, z, dO, False, scale)) / (2 * h)
            else:
                num[idx] = (_loss(q, xp, v, z, dO, False, scale) - _loss(q, xm, v, z, dO, False, scale)) / (2 * h)
        assert np.linalg.norm(num - g) / np.linalg.norm(num) <= 1e-6


@pytest.mark.parametrize("from_j", [False, True])
def test_gate_grad_suffix_scan_equals_double_sum(from_j):
    N, d = 40, 8
    q, k, v, z, dO = _rand_head(N, d, seed=77)
    _, _, _, _, ex = ora.backward_head(q, k, v, z, dO, bias_from_j=from_j, return_sums=True)
    np.testing.assert_allclose(ex["da"], ora.gate_grad_bruteforce(ex["dS"], from_j), atol=1e-12)


@pytest.mark.parametrize("from_j", [False, True])
@pytest.mark.parametrize("causal", [True, False])
def test_gate_grad_from_sums_equals_double_sum(from_j, causal):
    """The gate gradient from R and C alone (the standalone gate-backward step) equals the
    brute-force double sum over the bias entries that hold a_t, for any dS (masked or not),
    times sigmoid(-z) from scipy; z = +inf gives exactly 0."""
    N = 37
    r = np.random.default_rng(91 + 2 * from_j + causal)
    dS = r.standard_normal((N, N))
    if causal:
        dS = np.tril(dS)
    z = 1.0 + r.standard_normal(N)
    z[5] = np.inf
    dz = ora.gate_grad_from_sums(dS.sum(axis=1), dS.sum(axis=0), z, from_j)
    want = ora.gate_grad_bruteforce(dS, from_j) * scipy.special.expit(-z)
    np.testing.assert_allclose(dz, want, rtol=1e-12, atol=1e-12)
    assert dz[5] == 0.0


def test_row_shift_invariance_sums():
    """Adding a constant to a row of S leaves O unchanged, so every row sum of dS
    is 0 and the column sums add to 0; under j+1, a_0 enters no bias entry."""
    N, d = 64, 8
    q, k, v, z, dO = _rand_head(N, d, seed=8)
    _, _, _, dz, ex = ora.backward_head(q, k, v, z, dO, return_sums=True)
    np.testing.assert_allclose(ex["R"], 0.0, atol=1e-12)
    assert abs(ex["C"].sum()) < 1e-11
    assert dz[0] == pytest.approx(0.0, abs=1e-12)


def test_open_gate_backward_matches_torch_autograd_sdpa():
    """With f = 1 the attention part reduces to causal SDPA: dQ, dK, dV against
    torch autograd through the library routine; dz is 0 there (sigmoid(-inf) = 0)."""
    N, d = 48, 8
    q, k, v, _, dO = _rand_head(N, d, seed=21)
    z = np.full(N, np.inf)
    dQ, dK, dV, dz = ora.backward_head(q, k, v, z, dO)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None], is_causal=True)[0]
    out.backward(torch.tensor(dO))
    np.testing.assert_allclose(dQ, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dK, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dV, tv.grad.numpy(), atol=1e-12)
    np.testing.assert_array_equal(dz, 0.0)


def test_batched_backward_is_per_head():
    B, N, H, d = 2, 10, 2, 4
    r = np.random.default_rng(4)
    q, k, v, dO = (r.standard_normal((B, N, H, d)) for _ in range(4))
    z = r.normal(1.0, 1.0, (B, N, H))
    dQ, dK, dV, dz = ora.backward(q, k, v, z, dO)
    for b in range(B):
        for h in range(H):
            g = ora.backward_head(q[b, :, h], k[b, :, h], v[b, :, h], z[b, :, h], dO[b, :, h])
            for full, one in zip((dQ, dK, dV, dz), g):
                np.testing.assert_array_equal(full[b, :, h], one)


# ------------------------------------------------- non-causal ("encoder") mode


def test_noncausal_open_gate_is_plain_softmax_attention():
    N, d = 40, 8
    q, k, v, _, _ = _rand_head(N, d, seed=61)
    z = np.full(N, np.inf)
    O, lse = ora.attention_head(q, k, v, z, causal=False)
    tq, tk, tv = (torch.tensor(x)[None, None] for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=False)[0, 0].numpy()
    np.testing.assert_allclose(O, ref, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.tensor(d**-0.5 * q @ k.T), -1).numpy(), atol=1e-12)


def test_noncausal_constant_gate_is_symmetric_alibi_with_sign():
    """Encoder mode keeps the outer difference for every key: a constant gate gives
    -m (i - j) everywhere, i.e. a bonus m (j - i) for keys after the query."""
    N, d, m = 50, 8, 0.3
    q, k, v, _, _ = _rand_head(N, d, seed=62)
    z = np.full(N, -math.log(math.expm1(m)))
    i, j = np.meshgrid(np.arange(N), np.arange(N), indexing="ij")
    bias = torch.tensor(-m * (i - j).astype(np.float64))
    O, lse = ora.attention_head(q, k, v, z, causal=False)
    tq, tk, tv = (torch.tensor(x)[None, None] for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=bias[None, None])[0, 0].numpy()
    np.testing.assert_allclose(O, ref, atol=1e-11)


@pytest.mark.parametrize("from_j", [False, True])
def test_noncausal_backward_matches_central_differences(from_j):
    N, d = 9, 3
    q, k, v, z, dO = _rand_head(N, d, gate_mu=0.5, gate_sigma=1.5, seed=63)
    g = ora.backward_head(q, k, v, z, dO, bias_from_j=from_j, causal=False)

    def loss(qq, kk, vv, zz):
        O, _ = ora.attention_head(qq, kk, vv, zz, bias_from_j=from_j, causal=False)
        return float((O * dO).sum())

    h = 1e-6
    for n, x in enumerate((q, k, v, z)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v, z]
            args_m = [q, k, v, z]
            args_p[n], args_m[n] = xp, xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.linalg.norm(num - g[n]) <= 1e-6 * np.linalg.norm(num) + 1e-8


@pytest.mark.parametrize("from_j", [False, True])
def test_noncausal_gate_grad_suffix_equals_signed_double_sum(from_j):
    N, d = 30, 6
    q, k, v, z, dO = _rand_head(N, d, seed=64)
    _, _, _, _, ex = ora.backward_head(q, k, v, z, dO, bias_from_j=from_j, return_sums=True, causal=False)
    np.testing.assert_allclose(ex["da"], ora.gate_grad_bruteforce(ex["dS"], from_j), atol=1e-12)


def test_noncausal_rows_variant_matches_whole_head():
    N, d = 140, 16
    q, k, v, z, _ = _rand_head(N, d, seed=65)
    O, lse = ora.attention_head(q, k, v, z, causal=False)
    rows = [0, 70, 139]
    Or, lr = ora.attention_rows(q, k, v, z, rows, causal=False)
    np.testing.assert_allclose(Or, O[rows], atol=1e-12)
    np.testing.assert_allclose(lr, lse[rows], atol=1e-12)


@pytest.mark.parametrize("from_j", [False, True])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("block", [1, 64, 128, 1000])
def test_row_blocked_forward_matches_whole_head(from_j, causal, block):
    """The row-blocked forward (used where S does not fit whole) against the whole-head
    definition: blocks of 1 row, ragged blocks and one block over everything."""
    N, d = 300, 16
    q, k, v, z, _ = _rand_head(N, d, gate_mu=0.5, gate_sigma=1.5, seed=71)
    O, lse = ora.attention_head(q, k, v, z, scale=0.3, bias_from_j=from_j, causal=causal)
    Ob, lb = ora.attention_head_blocked(q, k, v, z, scale=0.3, bias_from_j=from_j, causal=causal, block=block)
    np.testing.assert_allclose(Ob, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lb, lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("from_j", [False, True])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("block", [1, 64, 1000])
def test_row_blocked_backward_matches_whole_head(from_j, causal, block):
    """The row-blocked backward against backward_head (itself pinned to finite differences,
    the double-sum gate gradient and autograd through SDPA): every gradient, and the row
    and column sums of dS that the gate gradient is formed from."""
    N, d = 300, 16
    q, k, v, z, dO = _rand_head(N, d, gate_mu=0.5, gate_sigma=1.5, seed=72)
    ref = ora.backward_head(q, k, v, z, dO, scale=0.3, bias_from_j=from_j, causal=causal, return_sums=True)
    got = ora.backward_head_blocked(q, k, v, z, dO, scale=0.3, bias_from_j=from_j, causal=causal, block=block,
                                    return_sums=True)
    for n, r, g in zip(("dQ", "dK", "dV", "dz"), ref[:4], got[:4]):
        np.testing.assert_allclose(g, r, rtol=0, atol=1e-11 * max(1.0, np.abs(r).max()), err_msg=n)
    np.testing.assert_allclose(got[4]["R"], ref[4]["R"], rtol=0, atol=1e-11)
    np.testing.assert_allclose(got[4]["C"], ref[4]["C"], rtol=0, atol=1e-11)


def test_row_blocked_open_gate_backward_matches_torch_autograd_sdpa():
    """The row-blocked backward pinned directly to a library routine: with f = 1 it is
    autograd through causal SDPA (dz = 0)."""
    N, d = 200, 8
    q, k, v, _, dO = _rand_head(N, d, seed=73)
    z = np.full(N, np.inf)
    dQ, dK, dV, dz = ora.backward_head_blocked(q, k, v, z, dO, block=48)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None], is_causal=True)[0]
    out.backward(torch.tensor(dO))
    np.testing.assert_allclose(dQ, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dK, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dV, tv.grad.numpy(), atol=1e-12)
    np.testing.assert_array_equal(dz, 0.0)


@pytest.mark.parametrize("from_j", [False, True])
@pytest.mark.parametrize("causal", [True, False])
def test_delta_is_the_row_sum_of_p_times_dp(from_j, causal):
    """Delta_i = dO_i . O_i equals sum_j P_ij dP_ij with dP_ij = dO_i . v_j (O_i = sum_j P_ij v_j):
    the identity the non-causal backward's Delta pass uses to form Delta without O."""
    N, d = 40, 8
    q, k, v, z, dO = _rand_head(N, d, gate_mu=0.5, gate_sigma=1.5, seed=66)
    O, _, P = ora.attention_head(q, k, v, z, bias_from_j=from_j, return_p=True, causal=causal)
    delta_from_o = (dO * O).sum(axis=1)
    delta_from_p = (P * (dO @ v.T)).sum(axis=1)
    np.testing.assert_allclose(delta_from_p, delta_from_o, rtol=0, atol=1e-12)
    # and dS = P (dP - Delta) has zero row sums with it (row-shift invariance of the softmax)
    dS = P * ((dO @ v.T) - delta_from_p[:, None])
    np.testing.assert_allclose(dS.sum(axis=1), 0.0, atol=1e-12)


# ----------------------------------------------------------------- gate projection
def test_gate_projection_is_torch_linear():
    """z = f_proj(x) with f_proj = nn.Linear(hidden, H, bias=True): the library routine in fp64."""
    rng = np.random.default_rng(40)
    x = rng.standard_normal((2, 7, 48))
    w = rng.standard_normal((5, 48))
    b = rng.standard_normal(5)
    ref = torch.nn.functional.linear(torch.tensor(x), torch.tensor(w), torch.tensor(b)).numpy()
    np.testing.assert_allclose(ora.gate_projection(x, w, b), ref, rtol=1e-13, atol=1e-13)


def test_gate_projection_special_inputs():
    """One-hot rows pick weight columns (so the weight layout is [H, hidden], not its
    transpose); x = 0 gives the bias alone."""
    rng = np.random.default_rng(41)
    hidden, H = 12, 3
    w = rng.standard_normal((H, hidden))
    b = rng.standard_normal(H)
    x = np.eye(hidden)[None]
    np.testing.assert_array_equal(ora.gate_projection(x, w, b)[0], w.T + b)
    np.testing.assert_array_equal(ora.gate_projection(np.zeros((1, 4, hidden)), w, b)[0], np.tile(b, (4, 1)))
