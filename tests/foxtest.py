"""Shared helpers for the tests: seeded inputs as torch tensors, oracle calls
on the exact (bf16-rounded) values, and the tolerances the comparisons use."""
from __future__ import annotations

import numpy as np

import workloads as wl

# Tolerances (fixed by the problem statement for this path):
#   bf16 inputs, fp32 accumulate: max |dO| <= 1e-2, max |dLSE| <= 1e-3,
#   gradients: ||g - g_ref||_F / ||g_ref||_F <= 2e-2 for dQ, dK, dV, dz.
#   fp32 inputs: max |dO| <= 1e-4.
TOL_O_BF16 = 1e-2
TOL_LSE_BF16 = 1e-3
TOL_GRAD_REL = 2e-2
TOL_O_F32 = 1e-4
TOL_LSE_F32 = 1e-4


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round to bf16 (nearest even) and back to fp64."""
    return wl.bf16_bits_to_f64(wl.f32_to_bf16_bits(np.asarray(x, dtype=np.float32)))


def o_excess_error(o_gpu: np.ndarray, o_ref: np.ndarray, dtype: str) -> float:
    """max |O_gpu - O_ref| beyond the rounding of O_ref itself to the output format.

    A bf16 output cannot be closer to the exact value than bf16(O_ref) is; for
    |O| in [4, 8) that rounding alone reaches 2^-6 = 0.0156 > 1e-2. So the
    stated O tolerance bounds the error left after subtracting, element by
    element, |bf16(O_ref) - O_ref| (zero for fp32 outputs)."""
    err = np.abs(o_gpu - o_ref)
    if dtype == "bf16":
        err = err - np.abs(bf16_round(o_ref) - o_ref)
    return float(err.max()) if err.size else 0.0


def to_torch(arrays, dtype: str, device="cuda"):
    """numpy arrays from workloads.draw -> torch tensors on `device`."""
    import torch

    out = {}
    for name, x in arrays.items():
        if name == "z":
            out[name] = torch.from_numpy(np.ascontiguousarray(x)).to(device)
        elif dtype == "bf16":
            out[name] = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)
        else:
            out[name] = torch.from_numpy(np.ascontiguousarray(x)).to(device)
    return out


def exact(arrays, dtype: str):
    """The exact fp64 values of drawn inputs (bf16 decoded), as the oracle consumes them."""
    return {n: (x.astype(np.float64) if n == "z" else wl.as_f64(x, dtype)) for n, x in arrays.items()}


def tensor_f64(t):
    import torch

    return t.detach().to("cpu", torch.float64).numpy()


def sample_rows(N: int, count: int, seed: int) -> np.ndarray:
    """Rows spanning tile edges (0, 1, 127, 128, 129, 255, 256, N-1, ...) plus seeded random rows."""
    edge = [0, 1, 2, 63, 64, 127, 128, 129, 255, 256, 257, N // 2, N - 129, N - 128, N - 2, N - 1]
    rng = np.random.default_rng(seed)
    rnd = rng.integers(0, N, size=max(0, count - len(edge)))
    return np.unique(np.clip(np.array(edge + list(rnd)), 0, N - 1))
