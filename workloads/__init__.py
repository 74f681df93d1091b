"""Seeded synthetic inputs for forget-gated causal attention workloads.

This module holds only random-number generation and the input recipes
(shapes, value distributions, seeds). It contains none of the attention
arithmetic, so both the CPU oracle and the CUDA path can draw the same inputs
from it without sharing any of the method's code.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the 64-bit finaliser constants as published by
Vigna), used as a counter-based stream: output k of a stream with seed s is
mix(s + (k+1) * 0x9E3779B97F4A7C15). Uniforms take the top 53 bits; normals are
Box-Muller pairs (u1, u2) -> sqrt(-2 ln(1-u1)) * (cos 2*pi*u2, sin 2*pi*u2).
bf16 tensors are drawn in fp32 and rounded to nearest even.

All tensors of one workload come from one stream in a fixed order:
q, k, v, dO (always reserved, drawn only when asked), per-head gate bias b_h,
gate noise. Each block starts at a fixed counter offset, so drawing dO or not
does not change the other tensors.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
from typing import Optional

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the SplitMix64 stream with this seed."""
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + k * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def uniforms(seed: int, start: int, count: int) -> np.ndarray:
    """fp64 uniforms in [0, 1) from outputs start .. start+count-1."""
    return (splitmix64(seed, start, count) >> np.uint64(11)).astype(np.float64) * (2.0**-53)


def normals(seed: int, start: int, count: int) -> np.ndarray:
    """`count` standard normals (fp64); consumes 2*ceil(count/2) outputs from `start`."""
    out = np.empty(count, dtype=np.float64)
    npairs = (count + 1) // 2
    done = 0
    for p0 in range(0, npairs, _CHUNK):
        p1 = min(npairs, p0 + _CHUNK)
        u = uniforms(seed, start + 2 * p0, 2 * (p1 - p0))
        r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
        t = (2.0 * math.pi) * u[1::2]
        pair = np.empty(2 * (p1 - p0), dtype=np.float64)
        pair[0::2] = r * np.cos(t)
        pair[1::2] = r * np.sin(t)
        n = min(count - done, pair.size)
        out[done : done + n] = pair[:n]
        done += n
    return out


_HERE = os.path.dirname(os.path.abspath(__file__))
_CLIB_PATH = os.path.join(_HERE, "_gen.so")
_clib = None


def _native():
    """The C version of the same generator (workloads/_gen.c), built with gcc on first use."""
    global _clib
    if _clib is None:
        src = os.path.join(_HERE, "_gen.c")
        if not os.path.exists(_CLIB_PATH) or os.path.getmtime(_CLIB_PATH) < os.path.getmtime(src):
            tmp = _CLIB_PATH + f".{os.getpid()}.tmp"
            subprocess.run(["gcc", "-O2", "-shared", "-fPIC", "-o", tmp, src, "-lm", "-lpthread"], check=True)
            os.replace(tmp, _CLIB_PATH)
        lib = ctypes.CDLL(_CLIB_PATH)
        lib.sm64_normals_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.c_int]
        lib.sm64_normals_f32.restype = None
        lib.sm64_fill.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p]
        lib.sm64_fill.restype = None
        _clib = lib
    return _clib


def normals_f32(seed: int, start: int, count: int) -> np.ndarray:
    """`count` standard normals rounded to fp32, from stream output `start` (C, all cores)."""
    out = np.empty(count, dtype=np.float32)
    if count:
        _native().sm64_normals_f32(seed & 0xFFFFFFFFFFFFFFFF, start, count, out.ctypes.data, os.cpu_count() or 1)
    return out


def normal_outputs(count: int) -> int:
    """Stream outputs consumed by `normals(count)`."""
    return 2 * ((count + 1) // 2)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic forget-gated attention problem.

    gate kinds (z is always fp32, layout [B, N, H]):
      "normal"   z = mu + sigma * N(0,1)                       (iid per element)
      "head_uniform"  z = b_h + sigma * N(0,1), b_h ~ U[lo, hi] per head, shared over B
      "head_linspace" z = b_h + sigma * N(0,1), b_h evenly spaced in [lo, hi], endpoints included
      "alibi"    constant per-head gate f_h = exp(-m_h), m_h = 2^(-8(h+1)/H): z_h = -ln(expm1(m_h))
      "open"     z = +inf (f = 1)
    """

    name: str
    B: int
    N: int
    H: int
    d: int
    dtype: str  # "bf16" or "f32"
    seed: int
    gate: str = "normal"
    lo: float = 0.0
    hi: float = 0.0
    sigma: float = 1.0
    bias_from_j: bool = False
    backward: bool = False

    @property
    def tokens(self) -> int:
        return self.B * self.N * self.H

    def fwd_flops(self) -> float:
        """Nominal causal forward FLOPs, 2*B*H*N^2*d."""
        return 2.0 * self.B * self.H * self.N * self.N * self.d

    def bwd_flops(self) -> float:
        """Nominal causal backward FLOPs, 2.5x the forward."""
        return 2.5 * self.fwd_flops()


def _offsets(w: Workload):
    n = w.tokens * w.d
    step = normal_outputs(n)
    off = {"q": 0, "k": step, "v": 2 * step, "dO": 3 * step}
    off["bh"] = 4 * step
    off["gate"] = 4 * step + 2 * ((w.H + 1) // 2)
    return off


def gate_logits(w: Workload) -> np.ndarray:
    """z [B, N, H] as fp32 per the workload's gate recipe."""
    off = _offsets(w)
    shape = (w.B, w.N, w.H)
    if w.gate == "open":
        return np.full(shape, np.inf, dtype=np.float32)
    if w.gate == "alibi":
        h = np.arange(w.H, dtype=np.float64)
        m = 2.0 ** (-8.0 * (h + 1.0) / w.H)
        zh = (-np.log(np.expm1(m))).astype(np.float32)
        return np.broadcast_to(zh[None, None, :], shape).copy()
    noise = normals_f32(w.seed, off["gate"], w.tokens).astype(np.float64).reshape(shape)
    if w.gate == "normal":
        z = w.lo + w.sigma * noise
    elif w.gate == "head_uniform":
        bh = w.lo + (w.hi - w.lo) * uniforms(w.seed, off["bh"], w.H)
        z = bh[None, None, :] + w.sigma * noise
    elif w.gate == "head_linspace":
        bh = np.linspace(w.lo, w.hi, w.H) if w.H > 1 else np.array([w.lo])
        z = bh[None, None, :] + w.sigma * noise
    else:
        raise ValueError(f"unknown gate recipe {w.gate!r}")
    return z.astype(np.float32)


def draw(w: Workload, with_dO: Optional[bool] = None):
    """Inputs of workload `w` as numpy arrays.

    Returns dict with q, k, v (and dO): bf16 as uint16 bit patterns or fp32,
    layout [B, N, H, d]; z fp32 [B, N, H].
    """
    if with_dO is None:
        with_dO = w.backward
    off = _offsets(w)
    n = w.tokens * w.d
    shape = (w.B, w.N, w.H, w.d)
    out = {}
    names = ["q", "k", "v"] + (["dO"] if with_dO else [])
    for name in names:
        x = normals_f32(w.seed, off[name], n)
        out[name] = (f32_to_bf16_bits(x) if w.dtype == "bf16" else x).reshape(shape)
    out["z"] = gate_logits(w)
    return out


def gate_head_bias(w: Workload) -> np.ndarray:
    """The per-head gate bias b_h of the "head_uniform" / "head_linspace" recipes (fp64 [H])."""
    off = _offsets(w)
    if w.gate == "head_uniform":
        return w.lo + (w.hi - w.lo) * uniforms(w.seed, off["bh"], w.H)
    if w.gate == "head_linspace":
        return np.linspace(w.lo, w.hi, w.H) if w.H > 1 else np.array([w.lo])
    raise ValueError(f"gate recipe {w.gate!r} has no per-head bias")


PROJ_SEED_XOR = 0x6A09E667F3BCC908  # separate stream for the gate-projection inputs


def draw_gate_projection(w: Workload, hidden: int):
    """Synthetic inputs of the gate projection z = x W^T + b for workload `w`.

    x [B, N, hidden] ~ N(0, 1) and W [H, hidden] ~ N(0, sigma^2 / hidden), both
    rounded to bf16 (uint16 bit patterns); b [H] = the recipe's b_h (fp32). Then
    z_h is about b_h + N(0, sigma^2) per token, the recipe's own gate distribution.
    Drawn from their own SplitMix64 stream (seed ^ PROJ_SEED_XOR): x from output 0,
    W right after it.
    """
    seed = (w.seed ^ PROJ_SEED_XOR) & 0xFFFFFFFFFFFFFFFF
    nx = w.B * w.N * hidden
    x = normals_f32(seed, 0, nx)
    wt = normals_f32(seed, normal_outputs(nx), w.H * hidden) * np.float32(w.sigma / math.sqrt(hidden))
    return {
        "x": f32_to_bf16_bits(x).reshape(w.B, w.N, hidden),
        "w_f": f32_to_bf16_bits(wt).reshape(w.H, hidden),
        "b_f": gate_head_bias(w).astype(np.float32),
    }


def as_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 values of a drawn tensor (bf16 bit patterns are decoded)."""
    return bf16_bits_to_f64(x) if dtype == "bf16" else np.asarray(x, dtype=np.float64)


# The five workloads of this problem, as named input recipes.
TINY_F32 = Workload("tiny_f32_B1H2N256d64", 1, 256, 2, 64, "f32", 0, gate="normal", lo=2.0, sigma=1.0)
MID_BF16 = Workload("mid_bf16_B4H16N2048d64", 4, 2048, 16, 64, "bf16", 1, gate="head_uniform", lo=1.0, hi=5.0)
LONG_BF16 = Workload("long_bf16_B1H32N16384d128", 1, 16384, 32, 128, "bf16", 2, gate="head_linspace", lo=0.0,
                     hi=8.0, sigma=0.5)
ALIBI_BF16 = Workload("alibi_bf16_B2H16N4096d128", 2, 4096, 16, 128, "bf16", 3, gate="alibi")
OPEN_BF16 = Workload("open_bf16_B2H16N4096d128", 2, 4096, 16, 128, "bf16", 3, gate="open")
TRAIN_BF16 = Workload("train_bf16_B8H16N4096d128", 8, 4096, 16, 128, "bf16", 4, gate="head_uniform", lo=1.0,
                      hi=6.0, backward=True)

ALL = [TINY_F32, MID_BF16, LONG_BF16, ALIBI_BF16, OPEN_BF16, TRAIN_BF16]


def alibi_slopes(H: int) -> np.ndarray:
    """m_h = 2^(-8(h+1)/H): the per-head decay of the "alibi" gate recipe."""
    h = np.arange(H, dtype=np.float64)
    return 2.0 ** (-8.0 * (h + 1.0) / H)
