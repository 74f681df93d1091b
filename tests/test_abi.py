"""The C ABI library without a GPU: it loads, exports every entry point the
header declares, and rejects bad arguments on the host with the documented
status codes before touching the device."""
import ctypes
import os
import re

import pytest

import forget_gated_softmax_gb300 as fox
from forget_gated_softmax_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    fbuild.build()
    return fox.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "fox.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fox_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert set(header_functions()) >= {
        "fox_fwd",
        "fox_bwd",
        "fox_fwd_workspace_bytes",
        "fox_bwd_workspace_bytes",
        "fox_check_error",
        "fox_status_string",
    }


def test_library_exports_every_declared_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), name
    for name in fox.EXPORTS:
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert L.fox_version() >= 100
    for code, name in fox.STATUS_NAMES.items():
        assert fox.fox_status_string(code).startswith(name)


def _p(**kw):
    base = dict(B=1, N=256, H=2, d=64, dtype=0, scale=0.0, bias_from_j=False)
    base.update(kw)
    return fox.make_params(**base)


def test_workspace_queries(L):
    ws = fox.fox_fwd_workspace_bytes(_p())
    assert ws >= 256 + 2 * 256 * 4
    assert fox.fox_bwd_workspace_bytes(_p()) > ws
    big = fox.fox_fwd_workspace_bytes(_p(B=1, H=32, N=16384, d=128))
    assert big >= 32 * 16384 * 4 * 2
    assert fox.fox_fwd_workspace_bytes(_p(d=96)) == 0
    assert fox.fox_fwd_workspace_bytes(_p(N=-1)) == 0
    assert fox.fox_fwd_min_workspace_bytes(_p(d=96)) == 0


def test_forward_workspace_holds_the_gate_terms_then_an_fp16_copy_of_v(L):
    for kw in (dict(), dict(B=3, N=700, H=5, d=128), dict(B=1, H=32, N=16384, d=128)):
        p = _p(**kw)
        lo, hi = fox.fox_fwd_min_workspace_bytes(p), fox.fox_fwd_workspace_bytes(p)
        assert lo % 256 == 0 and hi - lo == p.B * p.N * p.H * p.d * 2
    p = _p(dtype=1)  # the fp32 forward has no fp16 copy
    assert fox.fox_fwd_min_workspace_bytes(p) == fox.fox_fwd_workspace_bytes(p) > 0
    assert _fwd(L, _p(), nbytes=fox.fox_fwd_min_workspace_bytes(_p()) - 1) == 3


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _fwd(L, params, q=FAKE, k=FAKE, v=FAKE, z=FAKE, o=FAKE, lse=FAKE, ws=FAKE, nbytes=1 << 30):
    return L.fox_fwd(ctypes.byref(params), q, k, v, z, o, lse, ws, nbytes, None)


def test_fwd_rejects_bad_arguments_on_host(L):
    assert L.fox_fwd(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == 1
    assert _fwd(L, _p(d=96)) == 2
    assert _fwd(L, _p(d=0)) == 1
    assert _fwd(L, _p(B=-1)) == 1
    assert _fwd(L, _p(dtype=7)) == 1
    assert _fwd(L, fox.fox_params(1, 256, 2, 64, 0, -1.0, 0)) == 1
    assert _fwd(L, fox.fox_params(1, 256, 2, 64, 0, float("nan"), 0)) == 1
    assert _fwd(L, fox.fox_params(1, 256, 2, 64, 0, 0.0, 2)) == 1
    assert _fwd(L, fox.fox_params(1, 256, 2, 64, 0, 0.0, 0, 0, 0, 2)) == 1  # gate_ready must be 0 or 1
    assert _fwd(L, _p(), q=None) == 1
    assert _fwd(L, _p(), lse=None) == 1
    assert _fwd(L, _p(), q=FAKE + 8) == 1  # TMA needs 16-byte aligned operands
    assert _fwd(L, _p(), z=FAKE + 2) == 1
    assert _fwd(L, _p(), ws=None) == 3
    assert _fwd(L, _p(), ws=FAKE + 128) == 3
    assert _fwd(L, _p(), nbytes=100) == 3


def test_empty_problems_are_no_ops(L):
    for kw in (dict(N=0), dict(B=0), dict(H=0)):
        assert _fwd(L, _p(**kw), q=None, k=None, v=None, z=None, o=None, lse=None, ws=None, nbytes=0) == 0


def test_bwd_rejects_bad_arguments_on_host(L):
    p = _p()
    args = [FAKE] * 11
    assert L.fox_bwd(ctypes.byref(_p(d=96)), *args, FAKE, 1 << 30, None) == 2
    assert L.fox_bwd(ctypes.byref(_p(dtype=1)), *args, FAKE, 1 << 30, None) == 2
    bad = list(args)
    bad[6] = None  # dO
    assert L.fox_bwd(ctypes.byref(p), *bad, FAKE, 1 << 30, None) == 1
    assert L.fox_bwd(ctypes.byref(p), *args, None, 1 << 30, None) == 3


def test_check_error_rejects_bad_workspace(L):
    assert L.fox_check_error(None, None) == 3
    assert L.fox_check_error(FAKE + 4, None) == 3


def test_selftest_rejects_bad_arguments_on_host(L):
    assert L.fox_selftest_wait_timeout(0, FAKE, 256, None) == 1
    assert L.fox_selftest_wait_timeout(100001, FAKE, 256, None) == 1
    assert L.fox_selftest_wait_timeout(1000, None, 256, None) == 3
    assert L.fox_selftest_wait_timeout(1000, FAKE + 16, 256, None) == 3
    assert L.fox_selftest_wait_timeout(1000, FAKE, 255, None) == 3


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fox, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(fox, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        fox.lib()
