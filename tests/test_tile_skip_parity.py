"""Decay-aware tile skipping on the GPU (tile_skip = 1), through the C ABI.

* The tile spans fox_tile_span returns equal the oracle's tile_span, and every
  pair they leave out is negligible by the exact brute-force excess.
* Skipping changes no output bit of the forward, dK or dV, and leaves dQ and
  dz equal up to the order of their fp32 atomic sums, so the skipped path
  keeps the oracle parity of the full path. This is checked at small sizes and
  on the full-size long-context workload, whose fast-forgetting heads skip most
  pairs.
* Non-causal and fp32 requests are refused."""
import numpy as np
import pytest

import workloads as wl
from oracle import fox_oracle as ora

from foxtest import TOL_GRAD_REL, TOL_LSE_BF16, exact, assert_o, sample_rows, tensor_f64, to_torch

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


def fast_decay(name, B, N, H, d, seed, from_j=False, backward=False):
    """Heads from fast to slow forgetting (b_h evenly in [-1, 6]), as in the long-context recipe."""
    return wl.Workload(name, B, N, H, d, "bf16", seed=seed, gate="head_linspace", lo=-1.0, hi=6.0, sigma=0.5,
                       bias_from_j=from_j, backward=backward)


@pytest.mark.parametrize("B,N,H,d,from_j", [(1, 2000, 4, 64, False), (2, 1500, 3, 128, True),
                                            (1, 4096, 8, 128, False)])
def test_spans_match_oracle(B, N, H, d, from_j):
    fox = _fox()
    w = fast_decay(f"span{N}", B, N, H, d, seed=N + d, from_j=from_j)
    arrays = wl.draw(w, with_dO=False)
    t = to_torch(arrays, "bf16")
    jmin, imax = fox.fox_tile_span(t["q"], t["k"], t["z"], bias_from_j=from_j)
    jmin, imax = jmin.cpu().numpy(), imax.cpu().numpy()
    x = exact(arrays, "bf16")
    # The GPU forms the bound from fp32 norms and gate sums, the oracle in fp64: a decision
    # may differ only where the oracle's bound lies within DELTA of the threshold, so the
    # GPU's spans must sit between the oracle's at threshold +- DELTA (equal almost always).
    DELTA = 1e-3
    skipped = exact_hits = 0
    for b in range(B):
        for h in range(H):
            args = (x["q"][b, :, h], x["k"][b, :, h], x["z"][b, :, h])
            jr, ir = ora.tile_span(*args, bias_from_j=from_j)
            j_hi, i_lo = ora.tile_span(*args, bias_from_j=from_j, threshold=ora.SKIP_THRESHOLD_LOG2 - DELTA)
            j_lo, i_hi = ora.tile_span(*args, bias_from_j=from_j, threshold=ora.SKIP_THRESHOLD_LOG2 + DELTA)
            jg, ig = jmin[b * H + h], imax[b * H + h]
            assert np.all((j_lo <= jg) & (jg <= j_hi)), (b, h, jg, jr)
            assert np.all((i_lo <= ig) & (ig <= i_hi)), (b, h, ig, ir)
            exact_hits += int(np.array_equal(jg, jr) and np.array_equal(ig, ir))
            skipped += int(jr.sum())
    assert skipped > 0  # the fast heads do skip
    assert exact_hits >= B * H - 1


def test_skipped_pairs_are_negligible_exactly():
    """Brute force over the full fp64 logits: every pair left out has all weights < 2^-150."""
    fox = _fox()
    w = fast_decay("spanexact", 1, 1200, 3, 64, seed=9)
    arrays = wl.draw(w, with_dO=False)
    t = to_torch(arrays, "bf16")
    jmin, _ = fox.fox_tile_span(t["q"], t["k"], t["z"])
    jmin = jmin.cpu().numpy()
    x = exact(arrays, "bf16")
    for h in range(w.H):
        E = ora.tile_pair_excess(x["q"][0, :, h], x["k"][0, :, h], x["z"][0, :, h])
        for I in range(E.shape[0]):
            for J in range(int(jmin[h, I])):
                assert E[I, J] < -ora.SKIP_THRESHOLD_LOG2, (h, I, J, E[I, J])


def _fwd(t, w, skip):
    fox = _fox()
    params = fox.make_params(w.B, w.N, w.H, w.d, 0, 0.0, w.bias_from_j, tile_skip=skip)
    ws = fox.workspace(fox.fox_fwd_workspace_bytes(params), "cuda")
    o, lse = fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], bias_from_j=w.bias_from_j, tile_skip=skip, ws=ws)
    assert fox.fox_check_error(ws) == 0
    return o, lse


@pytest.mark.parametrize("B,N,H,d,from_j", [(1, 3000, 4, 64, False), (2, 2100, 3, 128, True),
                                            (1, 129, 2, 128, False)])
def test_forward_bit_identical_and_oracle(B, N, H, d, from_j):
    w = fast_decay(f"fskip{N}", B, N, H, d, seed=N * 7 + d, from_j=from_j)
    arrays = wl.draw(w, with_dO=False)
    t = to_torch(arrays, "bf16")
    o0, l0 = _fwd(t, w, False)
    o1, l1 = _fwd(t, w, True)
    torch.cuda.synchronize()
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l0.view(torch.int32), l1.view(torch.int32))
    x = exact(arrays, "bf16")
    O_ref, L_ref = ora.forward(x["q"], x["k"], x["v"], x["z"], bias_from_j=from_j)
    assert_o(tensor_f64(o1), O_ref, "bf16", f"tile_skip {w.name}")
    assert np.abs(tensor_f64(l1) - L_ref).max() <= TOL_LSE_BF16


def _bwd(t, o, lse, w, skip):
    fox = _fox()
    params = fox.make_params(w.B, w.N, w.H, w.d, 0, 0.0, w.bias_from_j, tile_skip=skip)
    ws = fox.workspace(fox.fox_bwd_workspace_bytes(params), "cuda")
    g = fox.fox_bwd(t["q"], t["k"], t["v"], t["z"], o, lse, t["dO"], bias_from_j=w.bias_from_j, tile_skip=skip,
                    ws=ws)
    assert fox.fox_check_error(ws) == 0
    return g


def _rel(a, b):
    n = np.linalg.norm(b)
    return np.linalg.norm(a - b) / n if n > 0 else np.linalg.norm(a)


@pytest.mark.parametrize("B,N,H,d,from_j", [(1, 3000, 4, 64, False), (2, 2100, 3, 128, True)])
def test_backward_matches_unskipped_and_oracle(B, N, H, d, from_j):
    w = fast_decay(f"bskip{N}", B, N, H, d, seed=N * 11 + d, from_j=from_j, backward=True)
    arrays = wl.draw(w, with_dO=True)
    t = to_torch(arrays, "bf16")
    o, lse = _fwd(t, w, False)
    g0 = [tensor_f64(x) for x in _bwd(t, o, lse, w, False)]
    g1 = [tensor_f64(x) for x in _bwd(t, o, lse, w, True)]
    np.testing.assert_array_equal(g0[1], g1[1])  # dK
    np.testing.assert_array_equal(g0[2], g1[2])  # dV
    assert _rel(g1[0], g0[0]) < 1e-5 and _rel(g1[3], g0[3]) < 1e-5  # dQ, dz: atomic-sum order only
    x = exact(arrays, "bf16")
    for b, h in [(0, 0), (B - 1, H - 1)]:
        r = ora.backward_head(x["q"][b, :, h], x["k"][b, :, h], x["v"][b, :, h], x["z"][b, :, h],
                              x["dO"][b, :, h], bias_from_j=from_j)
        for n in range(4):
            assert _rel(g1[n][b, :, h], r[n]) <= TOL_GRAD_REL, (b, h, n)


def test_long_workload_forward_bit_identical():
    """The long-context recipe at full size (B1 H32 N16384 d128): most pairs of the fast
    heads are skipped, no output bit changes; sampled rows still meet the oracle."""
    fox = _fox()
    w = wl.LONG_BF16
    arrays = wl.draw(w, with_dO=False)
    t = to_torch(arrays, "bf16")
    o0, l0 = _fwd(t, w, False)
    o1, l1 = _fwd(t, w, True)
    jmin, _ = fox.fox_tile_span(t["q"], t["k"], t["z"])
    torch.cuda.synchronize()
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l0.view(torch.int32), l1.view(torch.int32))
    nT = jmin.shape[1]
    visited = (torch.arange(nT, device="cuda")[None, :] - jmin + 1).sum().item()
    assert visited < 0.8 * w.H * nT * (nT + 1) // 2
    x = exact(arrays, "bf16")
    O, L = tensor_f64(o1), tensor_f64(l1)
    for h in (0, 5, 31):
        rows = sample_rows(w.N, 12, h)
        Or, Lr = ora.attention_rows(x["q"][0, :, h], x["k"][0, :, h], x["v"][0, :, h], x["z"][0, :, h], rows)
        assert_o(O[0, rows, h], Or, "bf16", "tile_skip long sampled rows")
        assert np.abs(L[0, rows, h] - Lr).max() <= TOL_LSE_BF16


def test_train_workload_backward_with_skip():
    """The training workload (B8 H16 N4096 d128, b_h ~ U[1, 6]): dK, dV bit-identical with skipping."""
    w = wl.TRAIN_BF16
    arrays = wl.draw(w, with_dO=True)
    t = to_torch(arrays, "bf16")
    o, lse = _fwd(t, w, False)
    g0 = _bwd(t, o, lse, w, False)
    g1 = _bwd(t, o, lse, w, True)
    torch.cuda.synchronize()
    assert torch.equal(g0[1].view(torch.int16), g1[1].view(torch.int16))
    assert torch.equal(g0[2].view(torch.int16), g1[2].view(torch.int16))
    for a, b in ((g0[0], g1[0]), (g0[3], g1[3])):
        a, b = a.double(), b.double()
        assert (torch.linalg.norm(a - b) / torch.linalg.norm(a)).item() < 1e-5


def test_unsupported_combinations():
    fox = _fox()
    w = fast_decay("unsup", 1, 256, 2, 64, seed=1)
    arrays = wl.draw(w, with_dO=False)
    t = to_torch(arrays, "bf16")
    with pytest.raises(fox.FoxError, match="UNSUPPORTED"):
        fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], non_causal=True, tile_skip=True)
    tf = to_torch(wl.draw(wl.Workload("unsup32", 1, 256, 2, 64, "f32", seed=1), with_dO=False), "f32")
    with pytest.raises(fox.FoxError, match="UNSUPPORTED"):
        fox.fox_fwd(tf["q"], tf["k"], tf["v"], tf["z"], tile_skip=True)
