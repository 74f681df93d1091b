"""Epsilon-effective window: the CUDA kernels (through the C ABI) against the
oracle's first-passage loop, integer for integer. Both decide the comparison
with L in fp64; rows whose passage sum lies within 1e-9 of L (where the two
summation orders may round differently) accept either neighbouring answer."""
import math

import numpy as np
import pytest

import workloads as wl
from oracle import fox_oracle as ora

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import forget_gated_softmax_gb300 as fox

    fox.lib()


def gpu_window(z, eps):
    import forget_gated_softmax_gb300 as fox

    w = fox.fox_window(torch.from_numpy(z).cuda(), eps)
    torch.cuda.synchronize()
    return w.cpu().numpy()


def near_tie(z_head, i, n, L):
    """True when the walk sum at n (or n-1) of row i is within 1e-9 of L."""
    X = -ora.log_forget_gate(z_head)
    sums = np.cumsum(X[: i + 1][::-1])
    for k in (n - 1, n):
        if 1 <= k <= i + 1 and abs(sums[k - 1] - L) < 1e-9 * max(1.0, L):
            return True
    return False


def compare(z, eps, rows=None):
    B, N, H = z.shape
    got = gpu_window(z, eps)
    L = math.log(1 / eps)
    for b in range(B):
        for h in range(H):
            idx = list(range(N)) if rows is None else list(rows)
            ref = ora.effective_window(z[b, :, h].astype(np.float64), eps, rows=idx)
            for i, r in zip(idx, ref):
                if got[b, i, h] != r:
                    assert near_tie(z[b, :, h].astype(np.float64), i, int(r), L), (b, i, h, got[b, i, h], r)


@pytest.mark.parametrize("N", [1, 7, 128, 300, 2049])
@pytest.mark.parametrize("eps", [0.5, 1e-3])
def test_random_gates(N, eps):
    w = wl.Workload("win", 2, N, 3, 64, "bf16", seed=N + 5, gate="head_uniform", lo=-1.0, hi=4.0)
    compare(wl.gate_logits(w), eps)


def test_alibi_limit_on_gpu():
    z = wl.gate_logits(wl.ALIBI_BF16)  # m_h = 2^(-(h+1)/2)
    got = gpu_window(z, 1e-3)
    L = math.log(1000.0)
    m = 1.0 / (1.0 + np.exp(-z[0, 0].astype(np.float64)))  # f_h
    for h in range(z.shape[2]):
        expect = math.floor(L / -math.log(m[h])) + 1
        i = np.arange(z.shape[1])
        np.testing.assert_array_equal(got[0, i >= expect - 1, h], expect)
        np.testing.assert_array_equal(got[0, i < expect - 1, h], -1)


def test_open_gates_never_pass():
    z = np.full((1, 100, 2), np.inf, dtype=np.float32)
    assert np.all(gpu_window(z, 1e-3) == -1)


def test_long_workload_sampled_rows():
    z = wl.gate_logits(wl.LONG_BF16)
    compare(z, 1e-3, rows=[0, 1, 127, 128, 5000, 16383])
