"""The device-side error path, on the GPU, without a fault: a bounded wait that runs out
(an mbarrier nothing arrives at, 1 ms limit) must set the timeout bit in the workspace's
error word, release the CTA's other wait through the abort flag, and leave the context
usable; fox_check_error must report FOX_ERR_TIMEOUT once and then FOX_OK."""
import pytest

import workloads as wl

from foxtest import to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

FOX_ERR_TIMEOUT = 5
DEV_ERR_TIMEOUT_SYNC = 1 << 2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import forget_gated_softmax_gb300 as fox

    fox.lib()


def test_bounded_wait_timeout_is_reported_and_cleared():
    import forget_gated_softmax_gb300 as fox

    ws = fox.workspace(4096, "cuda")
    fox.fox_selftest_wait_timeout(1000, ws)
    torch.cuda.synchronize()
    words = ws[:12].view(torch.int32).cpu().tolist()
    assert words[0] == DEV_ERR_TIMEOUT_SYNC, words  # only the wait that ran out set its bit
    assert words[1] == 0 and words[2] == 0, words   # both waits gave up; the second by the abort flag
    assert fox.fox_check_error(ws) == FOX_ERR_TIMEOUT
    assert fox.fox_check_error(ws) == 0             # the word was cleared


def test_context_stays_usable_after_a_timeout():
    """The same workspace, after the self-test, serves a forward bit-identical to one on a fresh workspace."""
    import forget_gated_softmax_gb300 as fox

    w = wl.Workload("errctx", 1, 700, 2, 128, "bf16", seed=5, gate="head_uniform", lo=0.0, hi=4.0)
    t = to_torch(wl.draw(w), "bf16")
    p = fox.make_params(w.B, w.N, w.H, w.d)
    ws = fox.workspace(fox.fox_fwd_workspace_bytes(p), "cuda")
    fox.fox_selftest_wait_timeout(500, ws)
    assert fox.fox_check_error(ws) == FOX_ERR_TIMEOUT
    o1, l1 = fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], ws=ws)
    assert fox.fox_check_error(ws) == 0
    o0, l0 = fox.fox_fwd(t["q"], t["k"], t["v"], t["z"])
    torch.cuda.synchronize()
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l0.view(torch.int32), l1.view(torch.int32))


@pytest.mark.parametrize("path", ["fp16 copy", "on chip"])
def test_v_outside_fp16_range_is_reported(path):
    """The forward's P V runs in fp16: a V value of magnitude 65536 or more cannot be held
    there, and the conversion reports it as FOX_ERR_DEVICE (the other outputs are then not
    meaningful; nothing faults), whether V is converted into the workspace (a workspace of
    fox_fwd_workspace_bytes) or tile by tile in the attention kernel (the minimum workspace)."""
    import forget_gated_softmax_gb300 as fox

    w = wl.Workload("vrange", 1, 300, 2, 64, "bf16", seed=6, gate="normal", lo=1.0)
    t = to_torch(wl.draw(w), "bf16")
    p = fox.make_params(w.B, w.N, w.H, w.d)
    nbytes = fox.fox_fwd_workspace_bytes(p) if path == "fp16 copy" else fox.fox_fwd_min_workspace_bytes(p)
    ws = fox.workspace(nbytes, "cuda")[:nbytes]
    fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], ws=ws)
    assert fox.fox_check_error(ws) == 0
    v = t["v"].clone()
    v[0, 137, 1, 5] = 1.0e6
    fox.fox_fwd(t["q"], t["k"], v, t["z"], ws=ws)
    assert fox.fox_check_error(ws) == 6  # FOX_ERR_DEVICE
    v[0, 137, 1, 5] = 65280.0  # the largest bf16 value below 65536 still converts exactly
    fox.fox_fwd(t["q"], t["k"], v, t["z"], ws=ws)
    assert fox.fox_check_error(ws) == 0
