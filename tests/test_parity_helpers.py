"""The parity tests' own helpers, on the CPU: the bf16 neighbours of a value, and the O
rule (plain 1e-2 bound; the bf16-neighbour rule only where |O_ref| >= 4)."""
import numpy as np

import workloads as wl
from foxtest import bf16_neighbours, o_check


def _all_bf16_in(lo, hi):
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF].astype(np.uint16)  # finite patterns only
    vals = wl.bf16_bits_to_f64(bits)
    return np.unique(vals[(vals >= lo) & (vals <= hi)])


def test_bf16_neighbours_against_enumeration():
    grid = _all_bf16_in(-20.0, 20.0)
    r = np.random.default_rng(0)
    x = np.concatenate([r.uniform(-17, 17, 4000), grid[(np.abs(grid) > 1e-3)][::7],
                        [4.0, -4.0, 4.0 + 1e-12, 8.0 - 1e-12, 7.99, -5.0001]])
    lo, hi = bf16_neighbours(x)
    for xi, a, b in zip(x, lo, hi):
        below = grid[grid <= xi]
        above = grid[grid >= xi]
        assert a == below.max() and b == above.min(), (xi, a, b)


def test_o_rule():
    ref = np.array([0.5, -3.99, 4.1107, -6.3, 0.0])
    lo, hi = bf16_neighbours(ref[2:4])
    good = np.array([0.5 + 0.0099, -3.99 - 0.0099, hi[0], lo[1], 0.0])
    res = o_check(good, ref, "bf16")
    assert res["n_fail"] == 0 and res["n_big"] == 2
    # 1e-2 is the plain bar below 4
    bad = good.copy()
    bad[0] = 0.5 + 0.0101
    assert o_check(bad, ref, "bf16")["n_fail"] == 1
    # above 4: within 1e-2 of O_ref is not enough unless it is a neighbour; two ulps off fails
    bad = good.copy()
    bad[2] = hi[0] + 2.0**-5
    assert o_check(bad, ref, "bf16")["n_fail"] == 1
    # fp32 outputs take the plain 1e-4 bound everywhere
    assert o_check(ref + 5e-5, ref, "f32")["n_fail"] == 0
    assert o_check(ref + 2e-4, ref, "f32")["n_fail"] == 5
