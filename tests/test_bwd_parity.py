"""Backward parity: dQ, dK, dV and dz from the CUDA path (through the C ABI)
against the CPU fp64 oracle's chain-rule gradients on the same seeded inputs.
The bar is the relative Frobenius error ||g - g_ref|| / ||g_ref|| <= 2e-2 per
gradient; small cases are compared whole, the full-size training workload on
whole sampled heads (every (b, h) is independent)."""
import numpy as np
import pytest

import workloads as wl
from oracle import fox_oracle as ora

from foxtest import TOL_GRAD_REL, exact, tensor_f64, to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import forget_gated_softmax_gb300 as fox

    fox.lib()


def run_fwd_bwd(w: wl.Workload, scale=0.0, arrays=None, non_causal=False):
    import forget_gated_softmax_gb300 as fox

    arrays = arrays if arrays is not None else wl.draw(w, with_dO=True)
    t = to_torch(arrays, "bf16")
    o, lse = fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], scale=scale, bias_from_j=w.bias_from_j,
                         non_causal=non_causal)
    params = fox.make_params(w.B, w.N, w.H, w.d, 0, scale, w.bias_from_j, non_causal)
    ws = fox.workspace(fox.fox_bwd_workspace_bytes(params), "cuda")
    grads = fox.fox_bwd(t["q"], t["k"], t["v"], t["z"], o, lse, t["dO"], scale=scale, bias_from_j=w.bias_from_j,
                        non_causal=non_causal, ws=ws)
    assert fox.fox_check_error(ws) == 0
    torch.cuda.synchronize()
    return arrays, [tensor_f64(g) for g in grads]


def rel(g, r):
    n = np.linalg.norm(r)
    return np.linalg.norm(g - r) / n if n > 0 else np.linalg.norm(g)


def check_heads(w: wl.Workload, heads=None, scale=0.0, non_causal=False):
    arrays, (dq, dk, dv, dz) = run_fwd_bwd(w, scale, non_causal=non_causal)
    for g in (dq, dk, dv, dz):
        assert np.isfinite(g).all()
    x = exact(arrays, "bf16")
    heads = heads if heads is not None else [(b, h) for b in range(w.B) for h in range(w.H)]
    ref = {n: [] for n in ("dq", "dk", "dv", "dz")}
    got = {n: [] for n in ref}
    for b, h in heads:
        r = ora.backward_head(x["q"][b, :, h], x["k"][b, :, h], x["v"][b, :, h], x["z"][b, :, h], x["dO"][b, :, h],
                              scale=scale or None, bias_from_j=w.bias_from_j, causal=not non_causal)
        for n, rr, gg in zip(("dq", "dk", "dv", "dz"), r, (dq, dk, dv, dz)):
            ref[n].append(rr)
            got[n].append(gg[b, :, h])
    errs = {n: rel(np.stack(got[n]), np.stack(ref[n])) for n in ref}
    for n, e in errs.items():
        assert e <= TOL_GRAD_REL, (w.name, n, e, errs)
    return errs


SMALL = [
    (1, 1, 1, 64),
    (1, 5, 2, 128),
    (2, 127, 2, 64),
    (1, 128, 2, 128),
    (2, 129, 3, 64),
    (1, 300, 2, 128),
    (1, 640, 2, 64),
    (2, 1000, 1, 128),
]


@pytest.mark.parametrize("B,N,H,d", SMALL)
@pytest.mark.parametrize("from_j", [False, True])
def test_small_shapes(B, N, H, d, from_j):
    w = wl.Workload(f"b{B}x{N}x{H}x{d}", B, N, H, d, "bf16", seed=N * 3 + d, gate="head_uniform", lo=0.0, hi=5.0,
                    bias_from_j=from_j, backward=True)
    check_heads(w)


def test_head_groups_with_remainder():
    """13 heads: key tiles are scheduled in groups of 8 heads, so this covers one full group
    and a remainder group of 5."""
    w = wl.Workload("bgroups", 1, 700, 13, 64, "bf16", seed=77, gate="head_linspace", lo=0.0, hi=5.0, sigma=0.5,
                    backward=True)
    check_heads(w)


def test_custom_scale():
    w = wl.Workload("bscale", 1, 384, 2, 128, "bf16", seed=17, gate="normal", lo=1.0, backward=True)
    check_heads(w, scale=0.2)


def test_open_gate_has_zero_gate_gradient():
    w = wl.Workload("bopen", 1, 300, 2, 64, "bf16", seed=4, gate="open", backward=True)
    arrays, (dq, dk, dv, dz) = run_fwd_bwd(w)
    assert np.all(dz == 0.0)
    x = exact(arrays, "bf16")
    r = ora.backward_head(x["q"][0, :, 0], x["k"][0, :, 0], x["v"][0, :, 0], x["z"][0, :, 0], x["dO"][0, :, 0])
    assert rel(dq[0, :, 0], r[0]) <= TOL_GRAD_REL and rel(dv[0, :, 0], r[2]) <= TOL_GRAD_REL


def test_train_workload_sampled_heads():
    w = wl.TRAIN_BF16
    check_heads(w, heads=[(0, 0), (0, 15), (3, 7), (5, 2), (7, 15)])


def test_backward_determinism():
    """dK and dV are written without atomics and repeat bit for bit; dQ and dz
    take fp32 atomic reductions across key tiles and repeat within rounding."""
    w = wl.Workload("bdet", 2, 700, 2, 128, "bf16", seed=21, gate="head_uniform", lo=0.5, hi=4.0, backward=True)
    a, g1 = run_fwd_bwd(w)
    _, g2 = run_fwd_bwd(w, arrays=a)
    for n in (1, 2):
        np.testing.assert_array_equal(g1[n], g2[n])
    assert rel(g1[0], g2[0]) < 1e-3 and rel(g1[3], g2[3]) < 1e-3


@pytest.mark.parametrize("B,N,H,d", [(1, 5, 2, 128), (2, 129, 2, 64), (1, 300, 2, 128), (1, 640, 1, 64)])
@pytest.mark.parametrize("from_j", [False, True])
def test_noncausal_backward(B, N, H, d, from_j):
    w = wl.Workload(f"bnc{B}x{N}x{H}x{d}", B, N, H, d, "bf16", seed=N * 5 + d, gate="head_uniform", lo=1.0,
                    hi=5.0, bias_from_j=from_j, backward=True)
    check_heads(w, non_causal=True)
