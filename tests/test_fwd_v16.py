"""The forward's two ways to an fp16 V for P V.

With a workspace of fox_fwd_workspace_bytes, a conversion kernel writes an fp16 copy of V
once and the attention kernel loads it; with less (down to fox_fwd_min_workspace_bytes,
the gate terms alone) the attention kernel converts each V tile it loads, in shared memory.
Both convert every element the same way and feed the same MMAs, so O and LSE must agree
bit for bit. The parity tests check the first path against the oracle; here the second is
checked against the first on every feature that reaches the attention kernel."""
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


CASES = [
    # name, B, N, H, d, gate, lo, hi, options
    ("causal d128 ragged", 2, 700, 3, 128, "head_uniform", 0.0, 5.0, {}),
    ("causal d64 j-convention", 1, 300, 2, 64, "normal", 1.0, 0.0, {"bias_from_j": True}),
    ("non-causal d128", 1, 513, 2, 128, "head_uniform", 2.0, 6.0, {"non_causal": True}),
    ("tile skip d128", 1, 1500, 2, 128, "head_uniform", -2.0, 0.0, {"tile_skip": True}),
    ("causal d64 many heads", 3, 1100, 6, 64, "head_uniform", 0.0, 8.0, {}),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_on_chip_conversion_matches_the_fp16_copy(case):
    import forget_gated_softmax_gb300 as fox

    name, B, N, H, d, gate, lo, hi, opts = case
    w = wl.Workload(name.replace(" ", "_"), B, N, H, d, "bf16", seed=77, gate=gate, lo=lo, hi=hi,
                    bias_from_j=opts.get("bias_from_j", False))
    t = to_torch(wl.draw(w), "bf16")
    p = fox.make_params(B, N, H, d, 0, 0.0, opts.get("bias_from_j", False), opts.get("non_causal", False),
                        opts.get("tile_skip", False))
    full, least = fox.fox_fwd_workspace_bytes(p), fox.fox_fwd_min_workspace_bytes(p)
    assert full - least == B * N * H * d * 2
    outs = []
    for nbytes in (full, least):
        ws = fox.workspace(nbytes, "cuda")[:nbytes]
        outs.append(fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], ws=ws, **opts))
        torch.cuda.synchronize()
        assert fox.fox_check_error(ws) == 0
    (o1, l1), (o2, l2) = outs
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_fp16_copy_leaves_v_and_the_gate_terms_alone():
    """The copy goes after the gate terms: a backward that reuses the forward's gate terms
    (gate_ready) on the same workspace gets the same gradients as one that recomputes them,
    and V is unchanged."""
    import forget_gated_softmax_gb300 as fox

    w = wl.Workload("v16ws", 2, 900, 4, 128, "bf16", seed=78, gate="head_uniform", lo=0.0, hi=6.0, backward=True)
    t = to_torch(wl.draw(w), "bf16")
    v0 = t["v"].clone()
    p = fox.make_params(w.B, w.N, w.H, w.d)
    ws = fox.workspace(max(fox.fox_fwd_workspace_bytes(p), fox.fox_bwd_workspace_bytes(p)), "cuda")
    o, lse = fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], ws=ws)
    g1 = fox.fox_bwd(t["q"], t["k"], t["v"], t["z"], o, lse, t["dO"], ws=ws, gate_ready=True)
    g0 = fox.fox_bwd(t["q"], t["k"], t["v"], t["z"], o, lse, t["dO"])
    torch.cuda.synchronize()
    assert fox.fox_check_error(ws) == 0
    assert torch.equal(t["v"].view(torch.int16), v0.view(torch.int16))
    assert torch.equal(g1[1].view(torch.int16), g0[1].view(torch.int16))  # dK
    assert torch.equal(g1[2].view(torch.int16), g0[2].view(torch.int16))  # dV
    for a, b in ((g1[0], g0[0]), (g1[3], g0[3])):  # dQ, dz: fp32 sums in any order
        a, b = a.double(), b.double()
        assert (torch.linalg.norm(a - b) / torch.linalg.norm(b)).item() < 1e-5
