"""Backward parity: dQ, dK, dV and dz from the CUDA path (through the C ABI)
against the CPU fp64 oracle's chain-rule gradients on the same seeded inputs.
The bar is the relative Frobenius error ||g - g_ref|| / ||g_ref|| <= 2e-2 per
gradient; small cases are compared whole. The full-size shapes are compared on
whole heads through the oracle's row-blocked backward, each head on its own
(every (b, h) is independent): the long-context shape that the benchmark step
times (B1 H32 N16384 d128) on heads 0, 1, 16 and 31 (fastest to slowest
forgetting), and the training workload on 16 heads spread over all 8 batches."""
import numpy as np
import pytest

import workloads as wl
from oracle import fox_oracle as ora

from foxtest import PARITY_LOG, TOL_GRAD_REL, exact, map_heads, tensor_f64, to_torch

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
    """The whole gradient tensors of the listed heads (default: all) against backward_head."""
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


def check_heads_blocked(w: wl.Workload, heads, arrays=None, non_causal=False, block=1024):
    """Whole heads of a full-size shape, each against the row-blocked oracle backward, each
    gradient of each head within the bar on its own; heads run in a thread pool."""
    arrays, (dq, dk, dv, dz) = run_fwd_bwd(w, arrays=arrays, non_causal=non_causal)
    for g in (dq, dk, dv, dz):
        assert np.isfinite(g).all()
    x = exact(arrays, "bf16")

    def one(bh):
        b, h = bh
        return ora.backward_head_blocked(x["q"][b, :, h], x["k"][b, :, h], x["v"][b, :, h], x["z"][b, :, h],
                                         x["dO"][b, :, h], bias_from_j=w.bias_from_j, causal=not non_causal,
                                         block=block)

    worst = {}
    for (b, h), r in zip(heads, map_heads(one, heads, threads=min(8, len(heads)))):
        errs = {n: rel(g[b, :, h], rr) for n, g, rr in zip(("dq", "dk", "dv", "dz"), (dq, dk, dv, dz), r)}
        for n, e in errs.items():
            worst[n] = max(worst.get(n, 0.0), e)
            assert e <= TOL_GRAD_REL, (w.name, (b, h), n, e, errs)
    PARITY_LOG.append((f"bwd {w.name}{' non-causal' if non_causal else ''} worst head rel", worst, len(heads)))
    return worst


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


@pytest.mark.parametrize("d", [64, 128])
def test_head_groups_with_remainder(d):
    """13 heads: key tiles are scheduled in groups of 8 heads, so this covers one full group
    and a remainder group of 5."""
    w = wl.Workload(f"bgroups{d}", 1, 700, 13, d, "bf16", seed=77, gate="head_linspace", lo=0.0, hi=5.0, sigma=0.5,
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


def test_long_shape_backward_heads():
    """The backward the benchmark step times: B1 H32 N16384 d128, b_h = linspace(0, 8, 32),
    dO ~ N(0, 1). Heads 0 and 1 forget fastest (a ~ -0.7 per token), 31 slowest; dz is a
    suffix scan over all 16384 tokens."""
    check_heads_blocked(wl.LONG_BF16, [(0, 0), (0, 1), (0, 16), (0, 31)], arrays=wl.draw(wl.LONG_BF16, with_dO=True))


def test_train_workload_backward_16_heads():
    """B8 H16 N4096 d128: two heads of every batch, 16 distinct heads in all."""
    heads = [(b, h) for b in range(8) for h in ((2 * b) % 16, (2 * b + 9) % 16)]
    assert len({h for _, h in heads}) == 16
    check_heads_blocked(wl.TRAIN_BF16, heads, block=512)


def test_many_heads_take_one_sequence_per_cta_for_the_gate_gradient():
    """B ceil(H / 4) >= the SM count: the backward's gate gradient walks each (b, 4-head)
    sequence in one CTA. N = 260 leaves a ragged last block. Heads from the first, middle and
    last CTAs, at both ends of a head group, are checked."""
    w = wl.Workload("many_heads", 80, 260, 12, 64, "bf16", seed=91, gate="head_uniform", lo=-1.0, hi=6.0,
                    backward=True)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert w.B * ((w.H + 3) // 4) >= sms
    check_heads_blocked(w, [(0, 0), (0, 7), (0, 8), (0, 11), (39, 3), (40, 9), (79, 4), (79, 11)])


@pytest.mark.parametrize("tile_skip", [False, True])
def test_gate_ready_reuses_the_forward_gate_terms(tile_skip):
    """fox_bwd with gate_ready on the workspace the forward wrote: no gate scan, the same results
    (dK, dV bit for bit; dQ and dz up to the order of their fp32 reductions)."""
    import forget_gated_softmax_gb300 as fox

    w = wl.Workload("bready", 2, 900, 3, 128, "bf16", seed=23, gate="head_uniform", lo=0.0, hi=5.0, backward=True)
    arrays = wl.draw(w)
    t = to_torch(arrays, "bf16")
    p = fox.make_params(w.B, w.N, w.H, w.d, tile_skip=tile_skip)
    ws = fox.workspace(max(fox.fox_fwd_workspace_bytes(p), fox.fox_bwd_workspace_bytes(p)), "cuda")
    o, lse = fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], ws=ws, tile_skip=tile_skip)
    g1 = fox.fox_bwd(t["q"], t["k"], t["v"], t["z"], o, lse, t["dO"], ws=ws, gate_ready=True, tile_skip=tile_skip)
    assert fox.fox_check_error(ws) == 0
    g0 = fox.fox_bwd(t["q"], t["k"], t["v"], t["z"], o, lse, t["dO"], tile_skip=tile_skip)
    torch.cuda.synchronize()
    g0, g1 = [tensor_f64(x) for x in g0], [tensor_f64(x) for x in g1]
    np.testing.assert_array_equal(g1[1], g0[1])
    np.testing.assert_array_equal(g1[2], g0[2])
    assert rel(g1[0], g0[0]) < 1e-5 and rel(g1[3], g0[3]) < 1e-5
    x = exact(arrays, "bf16")
    r = ora.backward_head(x["q"][1, :, 2], x["k"][1, :, 2], x["v"][1, :, 2], x["z"][1, :, 2], x["dO"][1, :, 2])
    for n in range(4):
        assert rel(g1[n][1, :, 2], r[n]) <= TOL_GRAD_REL


def test_backward_determinism():
    """dK and dV are written without atomics and repeat bit for bit; dQ and dz
    take fp32 atomic reductions across key tiles and repeat within rounding."""
    w = wl.Workload("bdet", 2, 700, 2, 128, "bf16", seed=21, gate="head_uniform", lo=0.5, hi=4.0, backward=True)
    a, g1 = run_fwd_bwd(w)
    _, g2 = run_fwd_bwd(w, arrays=a)
    for n in (1, 2):
        np.testing.assert_array_equal(g1[n], g2[n])
    assert rel(g1[0], g2[0]) < 1e-3 and rel(g1[3], g2[3]) < 1e-3


@pytest.mark.parametrize("from_j", [False, True])
def test_noncausal_backward_long(from_j):
    """Encoder mode at N = 2048 (16 key tiles per query row), both conventions: the gate
    gradient there is a small difference of large row and column sums over every key."""
    w = wl.Workload(f"bnc_long_j{int(from_j)}", 1, 2048, 2, 128, "bf16", seed=2048 + int(from_j), gate="head_uniform",
                    lo=1.0, hi=5.0, bias_from_j=from_j, backward=True)
    check_heads_blocked(w, [(0, 0), (0, 1)], non_causal=True, block=512)


@pytest.mark.parametrize("B,N,H,d", [(1, 5, 2, 128), (2, 129, 2, 64), (1, 300, 2, 128), (1, 640, 1, 64)])
@pytest.mark.parametrize("from_j", [False, True])
def test_noncausal_backward(B, N, H, d, from_j):
    w = wl.Workload(f"bnc{B}x{N}x{H}x{d}", B, N, H, d, "bf16", seed=N * 5 + d, gate="head_uniform", lo=1.0,
                    hi=5.0, bias_from_j=from_j, backward=True)
    check_heads(w, non_causal=True)
