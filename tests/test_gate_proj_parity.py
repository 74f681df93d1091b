"""Gate projection on the GPU (fox_gate_proj, fox_fwd_xgate), through the C ABI,
against the oracle's gate_projection (fp64 on the exact bf16 inputs).

z tolerance, from the arithmetic. The tensor core forms each z as a sum of
`hidden` exact bf16 x bf16 products plus the bias, in fp32, and the
summation order is unknown. So |z - z_ref| <= gamma * (sum_e |x_e w_e| + |b|)
with gamma = (hidden + 2) u and u = 2^-24 (the standard worst-case bound for
a recursive fp32 sum).

The fused kernel feeds the same fp32 z values to the same gate scan that
fox_fwd uses. fox_fwd_xgate is therefore bit-identical to fox_fwd on the z
that fox_gate_proj returns."""
import numpy as np
import pytest

import workloads as wl
from oracle import fox_oracle as ora

from foxtest import TOL_LSE_BF16, exact, assert_o, sample_rows, tensor_f64, to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import forget_gated_softmax_gb300 as fox

    fox.lib()


def _fox():
    import forget_gated_softmax_gb300 as fox

    return fox


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def proj_inputs(w, hidden):
    g = wl.draw_gate_projection(w, hidden)
    dev = {"x": _bf16(g["x"]), "w_f": _bf16(g["w_f"]), "b_f": torch.from_numpy(g["b_f"]).cuda()}
    ex = {"x": wl.bf16_bits_to_f64(g["x"]), "w_f": wl.bf16_bits_to_f64(g["w_f"]), "b_f": g["b_f"].astype(np.float64)}
    return dev, ex


def check_z(z_gpu, ex, rows=None):
    x = ex["x"] if rows is None else ex["x"][:, rows]
    ref = ora.gate_projection(x, ex["w_f"], ex["b_f"])
    mag = np.abs(x) @ np.abs(ex["w_f"]).T + np.abs(ex["b_f"])
    gamma = (x.shape[-1] + 2) * 2.0**-24
    got = z_gpu if rows is None else z_gpu[:, rows]
    err = np.abs(got - ref)
    assert np.all(err <= gamma * mag), float((err / (gamma * mag)).max())
    return float(err.max())


def gate_workload(name, B, N, H, seed):
    return wl.Workload(name, B, N, H, 64, "bf16", seed=seed, gate="head_linspace", lo=0.0, hi=5.0, sigma=0.5)


@pytest.mark.parametrize("B,N,H,hidden", [(1, 1, 1, 8), (1, 5, 3, 64), (2, 300, 5, 200), (1, 129, 16, 1024),
                                          (2, 257, 32, 4096), (1, 200, 48, 520), (1, 130, 256, 256)])
def test_gate_projection_matches_oracle(B, N, H, hidden):
    fox = _fox()
    w = gate_workload(f"proj{N}", B, N, H, seed=N + H + hidden)
    dev, ex = proj_inputs(w, hidden)
    z = fox.fox_gate_proj(dev["x"], dev["w_f"], dev["b_f"])
    torch.cuda.synchronize()
    check_z(tensor_f64(z), ex)


@pytest.mark.parametrize("B,N,H,d,hidden,from_j", [(1, 300, 4, 64, 256, False), (2, 640, 3, 128, 384, True),
                                                   (1, 1000, 8, 128, 1024, False)])
def test_fwd_xgate_equals_fwd_on_projected_z(B, N, H, d, hidden, from_j):
    fox = _fox()
    w = wl.Workload(f"xg{N}", B, N, H, d, "bf16", seed=N * 3 + hidden, gate="head_linspace", lo=0.0, hi=5.0,
                    sigma=0.5, bias_from_j=from_j)
    arrays = wl.draw(w, with_dO=False)
    t = to_torch(arrays, "bf16")
    dev, ex = proj_inputs(w, hidden)
    o1, l1, z1 = fox.fox_fwd_xgate(t["q"], t["k"], t["v"], dev["x"], dev["w_f"], dev["b_f"], bias_from_j=from_j)
    z0 = fox.fox_gate_proj(dev["x"], dev["w_f"], dev["b_f"])
    o0, l0 = fox.fox_fwd(t["q"], t["k"], t["v"], z0, bias_from_j=from_j)
    torch.cuda.synchronize()
    assert torch.equal(z0.view(torch.int32), z1.view(torch.int32))
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l0.view(torch.int32), l1.view(torch.int32))
    # and the whole chain against the oracle: z from the projection, then attention
    check_z(tensor_f64(z1), ex)
    x = exact(arrays, "bf16")
    z_ref = ora.gate_projection(ex["x"], ex["w_f"], ex["b_f"])
    O_ref, L_ref = ora.forward(x["q"], x["k"], x["v"], z_ref, bias_from_j=from_j)
    assert_o(tensor_f64(o1), O_ref, "bf16", "xgate small")
    assert np.abs(tensor_f64(l1) - L_ref).max() <= TOL_LSE_BF16


def test_long_workload_xgate_sampled():
    """The long-context shape (B1 H32 N16384 d128) with hidden = H d = 4096: z checked on
    sampled tokens, O and LSE on sampled rows of three heads (oracle fed its own z)."""
    fox = _fox()
    w = wl.LONG_BF16
    hidden = w.H * w.d
    arrays = wl.draw(w, with_dO=False)
    t = to_torch(arrays, "bf16")
    dev, ex = proj_inputs(w, hidden)
    o, lse, z = fox.fox_fwd_xgate(t["q"], t["k"], t["v"], dev["x"], dev["w_f"], dev["b_f"], tile_skip=True)
    torch.cuda.synchronize()
    zg = tensor_f64(z)
    check_z(zg, ex, rows=sample_rows(w.N, 64, 5))
    x = exact(arrays, "bf16")
    O, L = tensor_f64(o), tensor_f64(lse)
    z_ref = ora.gate_projection(ex["x"][0], ex["w_f"], ex["b_f"])  # [N, H]
    for h in (0, 13, 31):
        rows = sample_rows(w.N, 10, h)
        Or, Lr = ora.attention_rows(x["q"][0, :, h], x["k"][0, :, h], x["v"][0, :, h], z_ref[:, h], rows)
        assert_o(O[0, rows, h], Or, "bf16", "xgate long sampled rows")
        assert np.abs(L[0, rows, h] - Lr).max() <= TOL_LSE_BF16


def test_projection_argument_errors():
    fox = _fox()
    w = gate_workload("perr", 1, 64, 4, seed=3)
    dev, _ = proj_inputs(w, 64)
    with pytest.raises(fox.FoxError, match="INVALID_ARG"):
        fox.fox_gate_proj(dev["x"][..., :60].contiguous(), dev["w_f"][:, :60].contiguous(), dev["b_f"])
    big = gate_workload("pbig", 1, 64, 257, seed=3)
    dv, _ = proj_inputs(big, 64)
    with pytest.raises(fox.FoxError, match="UNSUPPORTED"):
        fox.fox_gate_proj(dv["x"], dv["w_f"], dv["b_f"])
