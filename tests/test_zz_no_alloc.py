"""fox_fwd_noalloc, the forward for callers that cannot allocate device memory
(it uses a fixed scratch array compiled into the library instead of a
workspace), checked against fox_fwd through the C ABI on two calls in a row.
Both run the same deterministic kernels on the same inputs, so O and LSE must
match bit for bit. Collected last so that a stop-at-first-failure run has
already run the rest."""
import ctypes

import numpy as np
import pytest

import workloads as wl

from foxtest import to_torch

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _lib():
    import forget_gated_softmax_gb300 as fox

    return fox, fox.lib()


def test_noalloc_forward_matches_fox_fwd_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fox, L = _lib()
    cases = [
        wl.Workload("na1", 2, 700, 3, 128, "bf16", seed=31, gate="head_uniform", lo=0.0, hi=5.0),
        wl.Workload("na2", 1, 300, 2, 64, "bf16", seed=32, gate="normal", lo=1.0, bias_from_j=True),
    ]
    for w in cases:  # two calls in a row per case; the second case also follows the first's contents
        t = to_torch(wl.draw(w), "bf16")
        o_ref, l_ref = fox.fox_fwd(t["q"], t["k"], t["v"], t["z"], bias_from_j=w.bias_from_j)
        p = fox.make_params(w.B, w.N, w.H, w.d, 0, 0.0, w.bias_from_j)
        stream = torch.cuda.current_stream().cuda_stream
        for _ in range(2):
            o = torch.full_like(o_ref, float("nan"))
            lse = torch.full_like(l_ref, float("nan"))
            st = L.fox_fwd_noalloc(ctypes.byref(p), t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(),
                                   t["z"].data_ptr(), o.data_ptr(), lse.data_ptr(), stream)
            assert st == 0, fox.fox_status_string(st)
            assert L.fox_noalloc_check_error(stream) == 0
            torch.cuda.synchronize()
            assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)), w.name
            assert torch.equal(lse.view(torch.int32), l_ref.view(torch.int32)), w.name


def test_noalloc_rejects_problems_larger_than_its_scratch():
    fox, L = _lib()
    limit = L.fox_noalloc_scratch_bytes()
    assert limit == 16 << 20
    big = fox.make_params(4, 65536, 32, 128, 0, 0.0, False)
    assert fox.fox_fwd_workspace_bytes(big) > limit
    fake = 0x10000  # never dereferenced: the size check comes first
    assert L.fox_fwd_noalloc(ctypes.byref(big), fake, fake, fake, fake, fake, fake, None) == 3
    bad = fox.make_params(1, 10, 1, 96, 0, 0.0, False)
    assert L.fox_fwd_noalloc(ctypes.byref(bad), fake, fake, fake, fake, fake, fake, None) == 2
