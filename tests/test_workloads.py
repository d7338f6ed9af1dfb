"""The seeded input recipe (host logic, no GPU)."""
import numpy as np

from gated_delta_rule_chunkwise_gb300 import workloads as wl


def test_bf16_rounding_is_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5 + 2 ** -9, 3.14159], np.float32)
    r = wl.round_bf16(x)
    np.testing.assert_array_equal(r[:5], np.array([1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5], np.float32))
    assert abs(r[5] - 3.140625) < 1e-7
    assert np.all((r.view(np.uint32) & 0xFFFF) == 0)


def test_recipe_shapes_norms_and_ranges():
    w = wl.make_chunk("kda_bf16_b8_t4096_h16_d128", B=2, T=70, H=3)
    assert w.q.shape == (2, 70, 3, 128) and w.gate.shape == (2, 70, 3, 128)
    assert np.all((w.q.view(np.uint32) & 0xFFFF) == 0)         # bf16-representable
    n = np.linalg.norm(w.q.astype(np.float64), axis=-1)
    assert np.all(np.abs(n - 1) < 1e-2)
    assert np.all((w.beta > 0) & (w.beta < 1))
    assert np.all(w.gate < 0) and w.S0 is None
    g = wl.make_chunk("gdn_bf16_long_b1_t8192_h16_d128", T=100, H=2)
    assert g.S0.shape == (1, 2, 128, 128) and abs(g.S0.std() - 0.02) < 0.002
    f = wl.make_chunk("deltanet_fp32_b1_t256_h1_d64")
    assert f.gate is None and f.q.dtype == np.float32
    np.testing.assert_allclose(np.linalg.norm(f.k, axis=-1), 1, atol=1e-6)


def test_recipe_is_deterministic_and_seeded():
    a = wl.make_chunk("gdn_bf16_b4_t2048_h16_d128", B=1, T=65, H=2)
    b = wl.make_chunk("gdn_bf16_b4_t2048_h16_d128", B=1, T=65, H=2)
    c = wl.make_chunk("gdn_bf16_b4_t2048_h16_d128", B=1, T=65, H=2, seed=1)
    np.testing.assert_array_equal(a.q, b.q)
    np.testing.assert_array_equal(a.gate, b.gate)
    assert not np.array_equal(a.q, c.q)


def test_decode_recipe():
    d = wl.make_decode("gdn_decode_b64_h16_dk64_dv128_steps1000", B=2, H=3, steps=5)
    assert d.q.shape == (5, 2, 3, 64) and d.v.shape == (5, 2, 3, 128)
    assert d.gate.shape == (5, 2, 3) and d.S0.shape == (2, 3, 64, 128)


def test_gdn2_recipe():
    w = wl.make_chunk("gdn2_bf16_b8_t4096_h16_d128", B=2, T=5, H=3, dk=64, dv=128)
    assert w.beta is None and w.erase.shape == (2, 5, 3, 64) and w.write.shape == (2, 5, 3, 128)
    assert np.all((w.erase > 0) & (w.erase < 1)) and np.all((w.write > 0) & (w.write < 1))
    assert w.gate.shape == (2, 5, 3, 64) and np.all(w.gate < 0)
    kda = wl.make_chunk("kda_bf16_b8_t4096_h16_d128", B=2, T=5, H=3, dk=64, dv=128)
    np.testing.assert_array_equal(w.q, kda.q)          # same draws up to the extra gates
    np.testing.assert_array_equal(w.gate, kda.gate)
    d = wl.make_decode("gdn2_decode_b64_h16_dk128_dv128_steps1000", B=2, H=3, steps=4)
    assert d.erase.shape == (4, 2, 3, 128) and d.write.shape == (4, 2, 3, 128) and d.beta is None
