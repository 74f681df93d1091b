"""Python binding of libfox.so: forget-gated causal softmax attention (FoX) on sm_103a.

Argument marshalling only. Every step of the computation runs in the CUDA
kernels behind the C ABI in include/fox.h; this module turns torch tensors
into pointers, allocates outputs and workspaces when the caller does not pass
them, and raises FoxError on a non-OK status. There is no CPU fallback: if the
library has not been built, every call fails with an error saying so.

Names follow the C ABI: fox_fwd, fox_bwd, fox_fwd_workspace_bytes,
fox_bwd_workspace_bytes, fox_check_error, fox_status_string.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfox.so")

FOX_DTYPE_BF16 = 0
FOX_DTYPE_F32 = 1

STATUS_NAMES = {
    0: "FOX_OK",
    1: "FOX_ERR_INVALID_ARG",
    2: "FOX_ERR_UNSUPPORTED",
    3: "FOX_ERR_WORKSPACE",
    4: "FOX_ERR_CUDA",
    5: "FOX_ERR_TIMEOUT",
    6: "FOX_ERR_DEVICE",
}

# Exported symbols of libfox.so (the entry points include/fox.h declares).
EXPORTS = (
    "fox_fwd",
    "fox_bwd",
    "fox_fwd_workspace_bytes",
    "fox_fwd_min_workspace_bytes",
    "fox_bwd_workspace_bytes",
    "fox_check_error",
    "fox_status_string",
    "fox_version",
    "fox_trace_begin",
    "fox_trace_end",
    "fox_fwd_noalloc",
    "fox_noalloc_check_error",
    "fox_selftest_wait_timeout",
    "fox_noalloc_scratch_bytes",
    "fox_window",
    "fox_window_workspace_bytes",
    "fox_tile_span",
    "fox_gate_proj",
    "fox_fwd_xgate",
    "fox_gate_scan",
    "fox_gate_scan_workspace_bytes",
    "fox_gate_bwd",
    "fox_gate_bwd_workspace_bytes",
)


class FoxError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fox_status_string(status)}")


class fox_params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int),
        ("N", ctypes.c_int),
        ("H", ctypes.c_int),
        ("d", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("bias_from_j", ctypes.c_int),
        ("non_causal", ctypes.c_int),
        ("tile_skip", ctypes.c_int),
        ("gate_ready", ctypes.c_int),
    ]


class fox_trace_record(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_char_p), ("ms", ctypes.c_float)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libfox.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libfox.so is not built ({LIB_PATH} missing); run "
                "`python -m forget_gated_softmax_gb300.build` (needs nvcc)"
            )
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        pp = ctypes.POINTER(fox_params)
        L.fox_fwd.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.fox_fwd.restype = i
        L.fox_bwd.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.fox_bwd.restype = i
        L.fox_fwd_workspace_bytes.argtypes = [pp]
        L.fox_fwd_workspace_bytes.restype = sz
        L.fox_fwd_min_workspace_bytes.argtypes = [pp]
        L.fox_fwd_min_workspace_bytes.restype = sz
        L.fox_bwd_workspace_bytes.argtypes = [pp]
        L.fox_bwd_workspace_bytes.restype = sz
        L.fox_check_error.argtypes = [vp, vp]
        L.fox_check_error.restype = i
        L.fox_status_string.argtypes = [i]
        L.fox_status_string.restype = ctypes.c_char_p
        L.fox_version.argtypes = []
        L.fox_version.restype = i
        L.fox_window_workspace_bytes.argtypes = [pp]
        L.fox_window_workspace_bytes.restype = sz
        L.fox_window.argtypes = [pp, vp, ctypes.c_double, vp, vp, sz, vp]
        L.fox_window.restype = i
        L.fox_gate_proj.argtypes = [pp, i, vp, vp, vp, vp, vp, sz, vp]
        L.fox_gate_proj.restype = i
        L.fox_fwd_xgate.argtypes = [pp, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.fox_fwd_xgate.restype = i
        L.fox_tile_span.argtypes = [pp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.fox_tile_span.restype = i
        L.fox_fwd_noalloc.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp]
        L.fox_fwd_noalloc.restype = i
        L.fox_noalloc_scratch_bytes.argtypes = []
        L.fox_noalloc_scratch_bytes.restype = sz
        L.fox_noalloc_check_error.argtypes = [vp]
        L.fox_noalloc_check_error.restype = i
        L.fox_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp, sz, vp]
        L.fox_selftest_wait_timeout.restype = i
        L.fox_gate_scan_workspace_bytes.argtypes = [pp]
        L.fox_gate_scan_workspace_bytes.restype = sz
        L.fox_gate_scan.argtypes = [pp, vp, vp, vp, sz, vp]
        L.fox_gate_scan.restype = i
        L.fox_gate_bwd_workspace_bytes.argtypes = [pp]
        L.fox_gate_bwd_workspace_bytes.restype = sz
        L.fox_gate_bwd.argtypes = [pp, vp, vp, vp, vp, vp, sz, vp]
        L.fox_gate_bwd.restype = i
        L.fox_trace_begin.argtypes = []
        L.fox_trace_begin.restype = i
        L.fox_trace_end.argtypes = [ctypes.POINTER(fox_trace_record), i]
        L.fox_trace_end.restype = i
        _lib = L
    return _lib


def fox_status_string(status: int) -> str:
    try:
        return lib().fox_status_string(int(status)).decode()
    except RuntimeError:
        return STATUS_NAMES.get(int(status), f"status {status}")


def make_params(B, N, H, d, dtype=FOX_DTYPE_BF16, scale=0.0, bias_from_j=False, non_causal=False,
                tile_skip=False, gate_ready=False) -> fox_params:
    return fox_params(int(B), int(N), int(H), int(d), int(dtype), float(scale), int(bool(bias_from_j)),
                      int(bool(non_causal)), int(bool(tile_skip)), int(bool(gate_ready)))


def fox_fwd_workspace_bytes(params: fox_params) -> int:
    return int(lib().fox_fwd_workspace_bytes(ctypes.byref(params)))


def fox_fwd_min_workspace_bytes(params: fox_params) -> int:
    return int(lib().fox_fwd_min_workspace_bytes(ctypes.byref(params)))


def fox_bwd_workspace_bytes(params: fox_params) -> int:
    return int(lib().fox_bwd_workspace_bytes(ctypes.byref(params)))


def _torch():
    import torch

    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return FOX_DTYPE_BF16
    if t.dtype == torch.float32:
        return FOX_DTYPE_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def workspace(nbytes: int, device):
    """A 256-byte aligned device workspace of at least nbytes (torch allocation)."""
    torch = _torch()
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def fox_fwd(
    q,
    k,
    v,
    z,
    *,
    scale: float = 0.0,
    bias_from_j: bool = False,
    non_causal: bool = False,
    tile_skip: bool = False,
    o=None,
    lse=None,
    ws=None,
    stream=None,
) -> Tuple[object, object]:
    """Forward: q, k, v [B, N, H, d] (bf16 or fp32), z [B, N, H] fp32 -> (O, LSE).

    O has q's dtype and layout; LSE is fp32 [B, N, H] (natural log). All
    tensors must be contiguous on the current CUDA device.
    """
    torch = _torch()
    B, N, H, d = q.shape
    params = make_params(B, N, H, d, _dtype_code(q), scale, bias_from_j, non_causal, tile_skip)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, N, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(fox_fwd_workspace_bytes(params), q.device)
    for t in (q, k, v, z, o, lse):
        if not t.is_contiguous():
            raise ValueError("fox_fwd needs contiguous tensors")
    st = lib().fox_fwd(
        ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
        _stream_handle(stream),
    )
    if st != 0:
        raise FoxError(st, "fox_fwd")
    return o, lse


def fox_bwd(
    q,
    k,
    v,
    z,
    o,
    lse,
    dO,
    *,
    scale: float = 0.0,
    bias_from_j: bool = False,
    non_causal: bool = False,
    tile_skip: bool = False,
    gate_ready: bool = False,
    dq=None,
    dk=None,
    dv=None,
    dz=None,
    ws=None,
    stream=None,
):
    """Backward (bf16): returns (dQ, dK, dV, dz); dz is fp32 [B, N, H]. gate_ready: `ws` holds the
    gate terms of z from a forward on the same workspace (see fox_params.gate_ready)."""
    torch = _torch()
    B, N, H, d = q.shape
    params = make_params(B, N, H, d, _dtype_code(q), scale, bias_from_j, non_causal, tile_skip, gate_ready)
    if gate_ready and ws is None:
        raise ValueError("gate_ready needs the workspace the forward wrote its gate terms into")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    dz = torch.empty((B, N, H), dtype=torch.float32, device=q.device) if dz is None else dz
    if ws is None:
        ws = workspace(fox_bwd_workspace_bytes(params), q.device)
    for t in (q, k, v, z, o, lse, dO, dq, dk, dv, dz):
        if not t.is_contiguous():
            raise ValueError("fox_bwd needs contiguous tensors")
    st = lib().fox_bwd(
        ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
        _ptr(dk), _ptr(dv), _ptr(dz), _ptr(ws), ws.numel(), _stream_handle(stream),
    )
    if st != 0:
        raise FoxError(st, "fox_bwd")
    return dq, dk, dv, dz


def fox_fwd_noalloc(q, k, v, z, *, scale: float = 0.0, bias_from_j: bool = False, o=None, lse=None, stream=None):
    """Forward with the library's fixed device scratch instead of a workspace
    (for callers that cannot allocate device memory; see fox_fwd_noalloc in
    include/fox.h). Output tensors are allocated here only when not passed."""
    torch = _torch()
    B, N, H, d = q.shape
    params = make_params(B, N, H, d, _dtype_code(q), scale, bias_from_j)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, N, H), dtype=torch.float32, device=q.device)
    for t in (q, k, v, z, o, lse):
        if not t.is_contiguous():
            raise ValueError("fox_fwd_noalloc needs contiguous tensors")
    st = lib().fox_fwd_noalloc(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(o), _ptr(lse),
                               _stream_handle(stream))
    if st != 0:
        raise FoxError(st, "fox_fwd_noalloc")
    return o, lse


def fox_window_workspace_bytes(params: fox_params) -> int:
    return int(lib().fox_window_workspace_bytes(ctypes.byref(params)))


def fox_window(z, eps: float, *, window=None, ws=None, stream=None):
    """Epsilon-effective window per query row: z [B, N, H] fp32 -> int32 [B, N, H] (-1: not reached)."""
    torch = _torch()
    B, N, H = z.shape
    params = make_params(B, N, H, 64)
    if window is None:
        window = torch.empty((B, N, H), dtype=torch.int32, device=z.device)
    if ws is None:
        ws = workspace(fox_window_workspace_bytes(params), z.device)
    if not z.is_contiguous() or not window.is_contiguous():
        raise ValueError("fox_window needs contiguous tensors")
    st = lib().fox_window(ctypes.byref(params), _ptr(z), float(eps), _ptr(window), _ptr(ws), ws.numel(),
                          _stream_handle(stream))
    if st != 0:
        raise FoxError(st, "fox_window")
    return window


def fox_gate_scan_workspace_bytes(params: fox_params) -> int:
    return int(lib().fox_gate_scan_workspace_bytes(ctypes.byref(params)))


def fox_gate_scan(z, *, bias_from_j: bool = False, c=None, want_c: bool = True, ws=None, stream=None):
    """The gate step alone: z [B, N, H] fp32 -> the cumulative log gate c [B, N, H] fp32
    (c_t = sum_{l<=t} log sigmoid(z_l)); with want_c=False only the workspace's gate terms
    are formed (what fox_fwd does first) and None is returned."""
    torch = _torch()
    B, N, H = z.shape
    params = make_params(B, N, H, 64, FOX_DTYPE_BF16, 0.0, bias_from_j)
    if want_c and c is None:
        c = torch.empty((B, N, H), dtype=torch.float32, device=z.device)
    if ws is None:
        ws = workspace(fox_gate_scan_workspace_bytes(params), z.device)
    if not z.is_contiguous() or (want_c and not c.is_contiguous()):
        raise ValueError("fox_gate_scan needs contiguous tensors")
    st = lib().fox_gate_scan(ctypes.byref(params), _ptr(z), _ptr(c) if want_c else None, _ptr(ws), ws.numel(),
                             _stream_handle(stream))
    if st != 0:
        raise FoxError(st, "fox_gate_scan")
    return c if want_c else None


def fox_gate_bwd_workspace_bytes(params: fox_params) -> int:
    return int(lib().fox_gate_bwd_workspace_bytes(ctypes.byref(params)))


def fox_gate_bwd(z, R, C, *, bias_from_j: bool = False, dz=None, ws=None, stream=None):
    """Gate gradient from the row / column sums of dS: z [B, N, H] fp32, R and C [B, H, N] fp32
    -> dz [B, N, H] fp32 (suffix sums of R - C, plus C under bias_from_j, times sigmoid(-z))."""
    torch = _torch()
    B, N, H = z.shape
    params = make_params(B, N, H, 64, FOX_DTYPE_BF16, 0.0, bias_from_j)
    if tuple(R.shape) != (B, H, N) or tuple(C.shape) != (B, H, N):
        raise ValueError("fox_gate_bwd: R and C must be [B, H, N]")
    if dz is None:
        dz = torch.empty((B, N, H), dtype=torch.float32, device=z.device)
    if ws is None:
        ws = workspace(fox_gate_bwd_workspace_bytes(params), z.device)
    for t in (z, R, C, dz):
        if not t.is_contiguous():
            raise ValueError("fox_gate_bwd needs contiguous tensors")
    st = lib().fox_gate_bwd(ctypes.byref(params), _ptr(z), _ptr(R), _ptr(C), _ptr(dz), _ptr(ws), ws.numel(),
                            _stream_handle(stream))
    if st != 0:
        raise FoxError(st, "fox_gate_bwd")
    return dz


def fox_gate_proj(x, w_f, b_f, *, bias_from_j: bool = False, z=None, ws=None, stream=None):
    """Gate logits z = x W_f^T + b_f: x [B, N, hidden] bf16, W_f [H, hidden] bf16, b_f [H] fp32
    -> z [B, N, H] fp32 (tensor cores; the gate scan runs in the same kernel into `ws`)."""
    torch = _torch()
    B, N, hidden = x.shape
    H = w_f.shape[0]
    params = make_params(B, N, H, 64, FOX_DTYPE_BF16, 0.0, bias_from_j)
    if z is None:
        z = torch.empty((B, N, H), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(fox_fwd_workspace_bytes(params), x.device)
    for t in (x, w_f, b_f, z):
        if not t.is_contiguous():
            raise ValueError("fox_gate_proj needs contiguous tensors")
    st = lib().fox_gate_proj(ctypes.byref(params), int(hidden), _ptr(x), _ptr(w_f), _ptr(b_f), _ptr(z), _ptr(ws),
                             ws.numel(), _stream_handle(stream))
    if st != 0:
        raise FoxError(st, "fox_gate_proj")
    return z


def fox_fwd_xgate(q, k, v, x, w_f, b_f, *, scale: float = 0.0, bias_from_j: bool = False, tile_skip: bool = False,
                  z=None, o=None, lse=None, ws=None, stream=None):
    """Forward from the gate projection: returns (O, LSE, z) with z = x W_f^T + b_f [B, N, H] fp32."""
    torch = _torch()
    B, N, H, d = q.shape
    hidden = x.shape[-1]
    params = make_params(B, N, H, d, _dtype_code(q), scale, bias_from_j, tile_skip=tile_skip)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, N, H), dtype=torch.float32, device=q.device) if lse is None else lse
    z = torch.empty((B, N, H), dtype=torch.float32, device=q.device) if z is None else z
    if ws is None:
        ws = workspace(fox_fwd_workspace_bytes(params), q.device)
    for t in (q, k, v, x, w_f, b_f, z, o, lse):
        if not t.is_contiguous():
            raise ValueError("fox_fwd_xgate needs contiguous tensors")
    st = lib().fox_fwd_xgate(ctypes.byref(params), int(hidden), _ptr(q), _ptr(k), _ptr(v), _ptr(x), _ptr(w_f),
                             _ptr(b_f), _ptr(z), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream_handle(stream))
    if st != 0:
        raise FoxError(st, "fox_fwd_xgate")
    return o, lse, z


def fox_tile_span(q, k, z, *, scale: float = 0.0, bias_from_j: bool = False, ws=None, stream=None):
    """Tile spans of the decay-aware tile skip: (jmin, imax), int32 [B*H, ceil(N/128)] each
    (first key tile of every query tile, last query tile of every key tile)."""
    torch = _torch()
    B, N, H, d = q.shape
    params = make_params(B, N, H, d, _dtype_code(q), scale, bias_from_j, tile_skip=True)
    nT = (N + 127) // 128
    jmin = torch.empty((B * H, nT), dtype=torch.int32, device=q.device)
    imax = torch.empty((B * H, nT), dtype=torch.int32, device=q.device)
    if ws is None:
        ws = workspace(fox_fwd_workspace_bytes(params), q.device)
    for t in (q, k, z):
        if not t.is_contiguous():
            raise ValueError("fox_tile_span needs contiguous tensors")
    st = lib().fox_tile_span(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(z), _ptr(jmin), _ptr(imax), _ptr(ws),
                             ws.numel(), _stream_handle(stream))
    if st != 0:
        raise FoxError(st, "fox_tile_span")
    return jmin, imax


def fox_check_error(ws, stream=None) -> int:
    """Synchronise and read (then clear) the workspace's device error word; returns the status."""
    return int(lib().fox_check_error(_ptr(ws), _stream_handle(stream)))


def fox_noalloc_check_error(stream=None) -> int:
    """fox_check_error for the fixed scratch of fox_fwd_noalloc on the current device."""
    return int(lib().fox_noalloc_check_error(_stream_handle(stream)))


def fox_selftest_wait_timeout(limit_us: int, ws, stream=None) -> None:
    """Enqueue the device error path's self-test (a bounded wait that runs out; see
    fox_selftest_wait_timeout in include/fox.h); read the outcome with fox_check_error(ws)."""
    st = lib().fox_selftest_wait_timeout(int(limit_us), _ptr(ws), ws.numel(), _stream_handle(stream))
    if st != 0:
        raise FoxError(st, "fox_selftest_wait_timeout")


def trace_begin() -> None:
    """Start bracketing every kernel launch of the library with CUDA events (see fox_trace_begin)."""
    st = lib().fox_trace_begin()
    if st != 0:
        raise FoxError(st, "fox_trace_begin")


def trace_end(max_records: int = 1 << 16):
    """Stop tracing; returns [(kernel name, milliseconds)] in launch order."""
    buf = (fox_trace_record * max_records)()
    n = lib().fox_trace_end(buf, max_records)
    if n < 0:
        raise FoxError(4, "fox_trace_end")
    return [(buf[i].kernel.decode(), float(buf[i].ms)) for i in range(min(n, max_records))]
