"""The seeded input generator: determinism, stream layout and distributions."""
import math

import numpy as np

import workloads as wl


def test_splitmix64_first_outputs():
    # SplitMix64 with seed 0: the first outputs of the published generator.
    out = wl.splitmix64(0, 0, 3)
    assert [int(x) for x in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_stream_is_offset_invariant():
    a = wl.splitmix64(7, 0, 100)
    b = wl.splitmix64(7, 40, 60)
    np.testing.assert_array_equal(a[40:], b)


def test_normals_moments_and_chunking():
    x = wl.normals(3, 0, 200001)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    np.testing.assert_array_equal(x[:1001], wl.normals(3, 0, 1001))


def test_bf16_rounding_nearest_even():
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5, 3.0e38], dtype=np.float32)
    bits = wl.f32_to_bf16_bits(vals)
    back = wl.bf16_bits_to_f64(bits)
    # 1+2^-8 is a tie between 1 and 1+2^-7: even mantissa (1.0) wins; 1+3*2^-8 rounds up to 1+2^-6
    np.testing.assert_array_equal(back[:5], [1.0, 1.0, 1.0 + 2**-6, 1.0, -2.5])
    assert np.isfinite(back[5])


def test_draw_is_deterministic_and_dO_does_not_shift_others():
    w = wl.Workload("t", 2, 33, 3, 8, "bf16", 5, gate="head_uniform", lo=1.0, hi=5.0)
    a = wl.draw(w, with_dO=False)
    b = wl.draw(w, with_dO=True)
    for name in ("q", "k", "v", "z"):
        np.testing.assert_array_equal(a[name], b[name])
    assert b["dO"].shape == (2, 33, 3, 8) and b["dO"].dtype == np.uint16
    assert not np.array_equal(a["q"], a["k"])


def test_gate_recipes():
    w = wl.Workload("t", 2, 500, 4, 8, "bf16", 1, gate="head_uniform", lo=1.0, hi=5.0)
    z = wl.gate_logits(w)
    assert z.dtype == np.float32 and z.shape == (2, 500, 4)
    bh = z.mean(axis=(0, 1))
    assert np.all((bh > 0.8) & (bh < 5.2))
    np.testing.assert_allclose(z[0].mean(0) - z[1].mean(0), 0, atol=0.2)  # b_h shared over the batch
    lin = wl.gate_logits(wl.Workload("t", 1, 4000, 32, 8, "bf16", 2, gate="head_linspace", lo=0, hi=8, sigma=0.5))
    np.testing.assert_allclose(lin.mean(axis=(0, 1)), np.linspace(0, 8, 32), atol=0.05)
    al = wl.gate_logits(wl.ALIBI_BF16)
    m = wl.alibi_slopes(16)
    sig = 1.0 / (1.0 + np.exp(-al[0, 0].astype(np.float64)))
    np.testing.assert_allclose(-np.log(sig), m, rtol=1e-6)
    assert math.isinf(wl.gate_logits(wl.OPEN_BF16)[0, 0, 0])


def test_named_workload_shapes():
    assert (wl.LONG_BF16.B, wl.LONG_BF16.H, wl.LONG_BF16.N, wl.LONG_BF16.d) == (1, 32, 16384, 128)
    assert wl.LONG_BF16.fwd_flops() == 2 * 32 * 16384**2 * 128
    assert wl.TRAIN_BF16.backward and wl.TRAIN_BF16.bwd_flops() == 2.5 * wl.TRAIN_BF16.fwd_flops()


def test_native_generator_matches_numpy_definition():
    u = np.empty(64, dtype=np.uint64)
    wl._native().sm64_fill(11, 1000, 64, u.ctypes.data)
    np.testing.assert_array_equal(u, wl.splitmix64(11, 1000, 64))
    for start, count in ((0, 1), (6, 100001), (1 << 33, 4097)):
        np.testing.assert_array_equal(wl.normals_f32(9, start, count), wl.normals(9, start, count).astype(np.float32))


def test_gate_projection_inputs():
    """Shapes, bf16 patterns, determinism, and z = x W^T + b near the recipe's b_h + N(0, sigma^2)."""
    w = wl.Workload("proj", 2, 300, 4, 64, "bf16", 7, gate="head_linspace", lo=0.0, hi=3.0, sigma=0.5)
    a = wl.draw_gate_projection(w, 256)
    b = wl.draw_gate_projection(w, 256)
    assert a["x"].shape == (2, 300, 256) and a["x"].dtype == np.uint16
    assert a["w_f"].shape == (4, 256) and a["w_f"].dtype == np.uint16
    assert a["b_f"].dtype == np.float32
    for n in a:
        np.testing.assert_array_equal(a[n], b[n])
    np.testing.assert_allclose(a["b_f"], np.linspace(0.0, 3.0, 4), rtol=1e-6)
    z = wl.bf16_bits_to_f64(a["x"]) @ wl.bf16_bits_to_f64(a["w_f"]).T
    assert abs(z.mean()) < 0.05 and abs(z.std() - 0.5) < 0.05
