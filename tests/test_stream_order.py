"""Back-to-back calls on one stream and one workspace.

Each call's kernels are launched as programmatic dependents of the kernel before them, so a
kernel may start while its predecessor still runs and must read nothing of the predecessor's
output before the grid-dependency wait. A call that followed another on the same workspace
would see the earlier call's gate terms, row sums or status words if that wait were missing or
misplaced; these tests run different problems back to back, without a synchronisation between
them, and compare every output with the same call made on its own."""
import pytest

import workloads as wl

from foxtest import to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import forget_gated_softmax_gb300 as fox

    fox.lib()


def _inputs(seed, lo, hi, B=2, N=1500, H=4, d=128):
    w = wl.Workload(f"so{seed}", B, N, H, d, "bf16", seed=seed, gate="head_uniform", lo=lo, hi=hi, backward=True)
    return w, to_torch(wl.draw(w), "bf16")


def _same(a, b):
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_forward_calls_back_to_back_on_one_workspace():
    import forget_gated_softmax_gb300 as fox

    w, t1 = _inputs(101, 0.0, 3.0)
    _, t2 = _inputs(102, 4.0, 8.0)  # other gates: other gate terms in the workspace
    p = fox.make_params(w.B, w.N, w.H, w.d)
    ws = fox.workspace(fox.fox_fwd_workspace_bytes(p), "cuda")
    ref1 = fox.fox_fwd(t1["q"], t1["k"], t1["v"], t1["z"])
    ref2 = fox.fox_fwd(t2["q"], t2["k"], t2["v"], t2["z"])
    torch.cuda.synchronize()
    outs = []
    for _ in range(3):  # alternate, nothing in between
        outs.append(fox.fox_fwd(t1["q"], t1["k"], t1["v"], t1["z"], ws=ws))
        outs.append(fox.fox_fwd(t2["q"], t2["k"], t2["v"], t2["z"], ws=ws))
    torch.cuda.synchronize()
    assert fox.fox_check_error(ws) == 0
    for n, (o, lse) in enumerate(outs):
        ro, rl = ref1 if n % 2 == 0 else ref2
        assert _same(o, ro) and _same(lse, rl), n


def test_steps_back_to_back_with_gate_reuse():
    """Forward then backward (gate_ready) of one problem, then of another, on one workspace:
    dK and dV bit for bit as in isolated calls, dQ and dz up to the order of their fp32 sums."""
    import forget_gated_softmax_gb300 as fox

    w, t1 = _inputs(103, 0.0, 2.0)
    _, t2 = _inputs(104, 3.0, 7.0)
    p = fox.make_params(w.B, w.N, w.H, w.d)
    ws = fox.workspace(max(fox.fox_fwd_workspace_bytes(p), fox.fox_bwd_workspace_bytes(p)), "cuda")

    def alone(t):
        o, lse = fox.fox_fwd(t["q"], t["k"], t["v"], t["z"])
        return fox.fox_bwd(t["q"], t["k"], t["v"], t["z"], o, lse, t["dO"])

    refs = [alone(t1), alone(t2)]
    torch.cuda.synchronize()
    got = []
    for t in (t1, t2, t1, t2):
        o, lse = fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], ws=ws)
        got.append(fox.fox_bwd(t["q"], t["k"], t["v"], t["z"], o, lse, t["dO"], ws=ws, gate_ready=True))
    torch.cuda.synchronize()
    assert fox.fox_check_error(ws) == 0
    for n, g in enumerate(got):
        r = refs[n % 2]
        assert _same(g[1], r[1]) and _same(g[2], r[2]), n  # dK, dV
        for a, b in ((g[0], r[0]), (g[3], r[3])):  # dQ, dz
            a, b = a.double(), b.double()
            assert (torch.linalg.norm(a - b) / torch.linalg.norm(b)).item() < 1e-5, n
