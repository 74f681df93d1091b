"""The standalone gate steps through the C ABI against the oracle: the prefix scan of the
log forget gate (fox_gate_scan's cumulative output) and the gate gradient from the row and
column sums of dS (fox_gate_bwd)."""
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


def _gates(B, N, H, seed):
    w = wl.Workload("gate", B, N, H, 64, "bf16", seed=seed, gate="head_uniform", lo=-3.0, hi=6.0)
    z = wl.draw(w)["z"]
    z[0, min(3, N - 1), 0] = np.inf  # f = 1 exactly: log f = 0
    return z


@pytest.mark.parametrize("N", [1, 7, 128, 129, 300, 2049, 16384])
@pytest.mark.parametrize("from_j", [False, True])
def test_gate_scan_cumulative(N, from_j):
    import forget_gated_softmax_gb300 as fox

    B, H = (2, 3) if N <= 2049 else (1, 2)
    z = _gates(B, N, H, seed=N)
    c = fox.fox_gate_scan(torch.from_numpy(z).cuda(), bias_from_j=from_j)
    torch.cuda.synchronize()
    got = c.cpu().numpy().astype(np.float64)
    for b in range(B):
        for h in range(H):
            ref = ora.cumulative_log_gate(ora.log_forget_gate(z[b, :, h].astype(np.float64)))
            err = np.abs(got[b, :, h] - ref)
            # fp32 tile-local sums of fp32 log-sigmoid values, fp64 tile bases
            assert np.all(err <= 3e-5 + 2e-6 * np.abs(ref)), (b, h, float(err.max()))


def test_gate_scan_workspace_only():
    """Without the cumulative output the call only forms the workspace's gate terms."""
    import forget_gated_softmax_gb300 as fox

    z = torch.from_numpy(_gates(1, 300, 2, seed=5)).cuda()
    assert fox.fox_gate_scan(z, want_c=False) is None
    torch.cuda.synchronize()


@pytest.mark.parametrize("B,N,H", [(2, 1, 3), (2, 5, 3), (2, 1023, 3), (2, 1024, 3), (2, 1025, 3), (2, 3000, 3),
                                   (3, 8193, 40), (1, 16384, 32)])
@pytest.mark.parametrize("from_j", [False, True])
def test_gate_bwd_from_sums(B, N, H, from_j):
    """One pass with a look-back across 128-token blocks: up to 128 blocks (four rounds of
    32), head groups of 32 with a partial one (H = 40), several batches."""
    import forget_gated_softmax_gb300 as fox

    r = np.random.default_rng(1000 + N + from_j)
    z = _gates(B, N, H, seed=N + 17)
    R = r.standard_normal((B, H, N)).astype(np.float32)
    C = r.standard_normal((B, H, N)).astype(np.float32)
    dz = fox.fox_gate_bwd(torch.from_numpy(z).cuda(), torch.from_numpy(R).cuda(), torch.from_numpy(C).cuda(),
                          bias_from_j=from_j)
    torch.cuda.synchronize()
    got = dz.cpu().numpy().astype(np.float64)
    for b in range(B):
        for h in range(H):
            ref = ora.gate_grad_from_sums(R[b, h], C[b, h], z[b, :, h], from_j)
            g = got[b, :, h]
            # fp32 suffix sums over up to N terms of size ~1
            assert np.linalg.norm(g - ref) <= 1e-5 * max(np.linalg.norm(ref), 1e-30), (b, h)
            assert np.all(g[np.isinf(z[b, :, h])] == 0.0)


@pytest.mark.parametrize("B,N,H", [(64, 520, 32), (160, 200, 8), (80, 1000, 12), (40, 4096, 32)])
@pytest.mark.parametrize("from_j", [False, True])
def test_gate_bwd_one_sequence_per_cta(B, N, H, from_j):
    """Shapes with at least one (b, 4-head group) sequence per SM take the kernel that walks
    each sequence in one CTA (no look-back): fewer blocks than pipeline stages (N = 200), three
    head groups (H = 12), a ragged last block, and 32 blocks. Every head is checked."""
    import forget_gated_softmax_gb300 as fox

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert B * ((H + 3) // 4) >= sms and N % 4 == 0 and H % 4 == 0  # the shape qualifies
    r = np.random.default_rng(2000 + N + from_j)
    z = _gates(B, N, H, seed=N + 29)
    R = r.standard_normal((B, H, N)).astype(np.float32)
    C = r.standard_normal((B, H, N)).astype(np.float32)
    dz = fox.fox_gate_bwd(torch.from_numpy(z).cuda(), torch.from_numpy(R).cuda(), torch.from_numpy(C).cuda(),
                          bias_from_j=from_j)
    torch.cuda.synchronize()
    got = dz.cpu().numpy().astype(np.float64)
    for b in range(B):
        for h in range(H):
            ref = ora.gate_grad_from_sums(R[b, h], C[b, h], z[b, :, h], from_j)
            g = got[b, :, h]
            assert np.linalg.norm(g - ref) <= 1e-5 * max(np.linalg.norm(ref), 1e-30), (b, h)
            assert np.all(g[np.isinf(z[b, :, h])] == 0.0)
