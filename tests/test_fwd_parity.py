"""Forward parity: the CUDA path (through the C ABI) against the CPU fp64
oracle on the same seeded inputs, element by element.

Small cases span several 128-row tiles and ragged tails; they and every named
workload are compared on every head and every row (the long ones through the
oracle's row-blocked forward, heads in a thread pool). The O bound is the plain
max |O_gpu - O_ref| <= 1e-2, with the bf16-neighbour rule only where |O_ref| >= 4."""
import numpy as np
import pytest

import workloads as wl
from oracle import fox_oracle as ora

from foxtest import TOL_LSE_BF16, TOL_LSE_F32, assert_o, exact, map_heads, tensor_f64, to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import forget_gated_softmax_gb300 as fox

    fox.lib()  # fails loudly if the library is missing


def run_fwd(w: wl.Workload, scale=0.0, arrays=None, non_causal=False):
    import forget_gated_softmax_gb300 as fox

    arrays = arrays if arrays is not None else wl.draw(w, with_dO=False)
    t = to_torch(arrays, w.dtype)
    ws = fox.workspace(fox.fox_fwd_workspace_bytes(fox.make_params(w.B, w.N, w.H, w.d, 0 if w.dtype == "bf16" else 1,
                                                                   scale, w.bias_from_j, non_causal)), "cuda")
    o, lse = fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], scale=scale, bias_from_j=w.bias_from_j,
                         non_causal=non_causal, ws=ws)
    assert fox.fox_check_error(ws) == 0
    torch.cuda.synchronize()
    return arrays, o, lse


def check_full(w: wl.Workload, scale=0.0, arrays=None, non_causal=False):
    arrays, o, lse = run_fwd(w, scale, arrays, non_causal)
    x = exact(arrays, w.dtype)
    O_ref, L_ref = ora.forward(x["q"], x["k"], x["v"], x["z"], scale=scale or None, bias_from_j=w.bias_from_j,
                               causal=not non_causal)
    tol_l = TOL_LSE_BF16 if w.dtype == "bf16" else TOL_LSE_F32
    res = assert_o(tensor_f64(o), O_ref, w.dtype, f"fwd {w.name}{' non-causal' if non_causal else ''}")
    L = tensor_f64(lse)
    err_l = np.abs(L - L_ref).max()
    assert np.isfinite(L).all()
    assert err_l <= tol_l, (w.name, "LSE", err_l)
    return res["max_abs"], err_l


def check_all_rows(w: wl.Workload, block=512):
    """Every head and every row of a full-size workload, through the row-blocked oracle."""
    arrays, o, lse = run_fwd(w)
    x = exact(arrays, w.dtype)
    O = tensor_f64(o)
    L = tensor_f64(lse)

    def one(bh):
        b, h = bh
        Or, Lr = ora.attention_head_blocked(x["q"][b, :, h], x["k"][b, :, h], x["v"][b, :, h], x["z"][b, :, h],
                                            bias_from_j=w.bias_from_j, block=block)
        return Or, Lr

    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    O_ref = np.empty_like(O)
    L_ref = np.empty_like(L)
    for (b, h), (Or, Lr) in zip(heads, map_heads(one, heads)):
        O_ref[b, :, h] = Or
        L_ref[b, :, h] = Lr
    res = assert_o(O, O_ref, w.dtype, f"fwd {w.name} (all rows)")
    err_l = np.abs(L - L_ref).max()
    assert np.isfinite(L).all()
    assert err_l <= TOL_LSE_BF16, (w.name, "LSE", err_l)
    return res["max_abs"], err_l


SMALL = [
    (1, 1, 1, 64),
    (1, 2, 2, 64),
    (2, 127, 3, 64),
    (1, 128, 2, 128),
    (2, 129, 2, 128),
    (1, 255, 1, 64),
    (1, 256, 2, 128),
    (2, 300, 3, 128),
    (1, 513, 2, 64),
    (1, 1000, 2, 128),
]


@pytest.mark.parametrize("B,N,H,d", SMALL)
@pytest.mark.parametrize("from_j", [False, True])
def test_small_shapes_bf16(B, N, H, d, from_j):
    w = wl.Workload(f"s{B}x{N}x{H}x{d}", B, N, H, d, "bf16", seed=N * 7 + d, gate="head_uniform", lo=-1.0,
                    hi=5.0, bias_from_j=from_j)
    check_full(w)


@pytest.mark.parametrize("B,N,H,d", [(1, 700, 13, 128), (1, 520, 21, 64)])
def test_head_groups_with_remainder(B, N, H, d):
    """Query blocks are scheduled in groups of 8 heads at d = 128 and 16 at d = 64: 13 and 21
    heads cover one full group and a remainder group of 5, every row checked."""
    w = wl.Workload(f"fgroups{H}x{d}", B, N, H, d, "bf16", seed=N + H, gate="head_linspace", lo=0.0, hi=5.0,
                    sigma=0.5)
    check_full(w)


@pytest.mark.parametrize("scale", [0.05, 0.3])
def test_custom_scale(scale):
    w = wl.Workload("scale", 1, 300, 2, 64, "bf16", seed=11, gate="normal", lo=1.0)
    check_full(w, scale=scale)


def test_open_gate_and_closing_gates():
    w = wl.Workload("open", 1, 384, 2, 128, "bf16", seed=5, gate="open")
    check_full(w)
    w2 = wl.Workload("fast", 1, 384, 2, 128, "bf16", seed=6, gate="normal", lo=-30.0, sigma=1.0)
    check_full(w2)


@pytest.mark.parametrize("B,N,H,d", [(1, 256, 2, 64), (1, 300, 3, 128), (2, 129, 1, 64)])
def test_fp32_path(B, N, H, d):
    w = wl.Workload("f32", B, N, H, d, "f32", seed=3, gate="normal", lo=2.0)
    check_full(w)


def test_tiny_f32_workload():
    check_full(wl.TINY_F32)


def test_mid_bf16_workload_full():
    check_full(wl.MID_BF16)


def test_long_bf16_workload_all_rows():
    """B1 H32 N16384 d128, fast- to slow-forgetting heads: all 32 heads, all 16384 rows."""
    check_all_rows(wl.LONG_BF16)


@pytest.mark.parametrize("w", [wl.ALIBI_BF16, wl.OPEN_BF16], ids=["alibi", "open"])
def test_limit_workloads_all_rows(w):
    check_all_rows(w)


def test_train_workload_forward_all_rows():
    check_all_rows(wl.TRAIN_BF16)


@pytest.mark.parametrize("gate", ["open", "slow"])
def test_row_maximum_growing_on_a_far_tile(gate):
    """Keys 0..127 scaled by 8: their scores dwarf those near the diagonal, so for most rows the
    maximum sits in the last key tile visited (tile 0; tiles are visited from the diagonal back)
    and exceeds the running maximum by far more than the rescale threshold, so O and the row sum
    are rescaled late in the row. Open gates (f = 1) and slowly forgetting ones (z ~ N(6, 1))."""
    w = wl.Workload(f"grow_{gate}", 1, 900, 2, 128, "bf16", seed=71, gate="open" if gate == "open" else "normal",
                    lo=6.0)
    arrays = wl.draw(w)
    k = wl.bf16_bits_to_f64(arrays["k"]).astype(np.float32)
    k[:, :128] *= 8.0
    arrays["k"] = wl.f32_to_bf16_bits(k).reshape(arrays["k"].shape)
    check_full(w, arrays=arrays)


def test_forward_is_deterministic():
    w = wl.Workload("det", 2, 700, 3, 128, "bf16", seed=9, gate="head_uniform", lo=0.0, hi=4.0)
    a, o1, l1 = run_fwd(w)
    _, o2, l2 = run_fwd(w, arrays=a)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_outputs_leave_neighbours_untouched():
    """Guard bands around O and LSE keep their NaN fill: no write past the ends."""
    import forget_gated_softmax_gb300 as fox

    w = wl.Workload("guard", 1, 200, 3, 64, "bf16", seed=2, gate="normal", lo=1.0)
    arrays = wl.draw(w)
    t = to_torch(arrays, "bf16")
    G = 4096
    obuf = torch.full((G + w.B * w.N * w.H * w.d + G,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((G + w.B * w.N * w.H + G,), float("nan"), dtype=torch.float32, device="cuda")
    o = obuf[G : G + w.B * w.N * w.H * w.d].view(w.B, w.N, w.H, w.d)
    lse = lbuf[G : G + w.B * w.N * w.H].view(w.B, w.N, w.H)
    fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], o=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.isnan(obuf[:G]).all() and torch.isnan(obuf[-G:]).all()
    assert torch.isnan(lbuf[:G]).all() and torch.isnan(lbuf[-G:]).all()
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()


@pytest.mark.parametrize("B,N,H,d", [(1, 1, 1, 64), (2, 129, 2, 128), (1, 300, 3, 64), (1, 700, 2, 128)])
@pytest.mark.parametrize("from_j", [False, True])
def test_noncausal_forward(B, N, H, d, from_j):
    """The module's encoder mode: every key, the outer-difference bias positive for keys after the query."""
    w = wl.Workload(f"nc{B}x{N}x{H}x{d}", B, N, H, d, "bf16", seed=N + 3 * d, gate="head_uniform", lo=0.0,
                    hi=5.0, bias_from_j=from_j)
    check_full(w, non_causal=True)


def test_noncausal_fp32_is_unsupported():
    import forget_gated_softmax_gb300 as fox

    t = to_torch(wl.draw(wl.Workload("ncf", 1, 64, 1, 64, "f32", seed=1)), "f32")
    with pytest.raises(fox.FoxError) as e:
        fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], non_causal=True)
    assert e.value.status == 2
