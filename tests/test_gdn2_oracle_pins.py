"""Pins of the Gated DeltaNet-2 oracle (linear-attention notes, Sec. 2.6,
Eqs. 21-24) against what the pages and the algebra fix, independent of the
oracle's loop:
  * with b = beta 1 and w = beta 1 it is KDA (the notes state this reduction);
  * with the erase off (b = 0) and the write on (w = 1) the memory is purely
    additive: o_t = sum_{j<=t} v_j (k_j * e^{G_t - G_j}) . q_t, a direct sum;
  * with unit keys and b = w = 1 every token is written exactly: S_t k_t = v_t;
  * brute force through the notes' matrix expansion
    W_t = Wt (I - e k^T) + z k^T at d = 4, T = 8."""
import numpy as np

import oracle


def _inputs(B=2, T=9, H=2, dk=4, dv=3, seed=0):
    rng = np.random.default_rng(seed)
    f32 = np.float32
    q = rng.standard_normal((B, T, H, dk)).astype(f32)
    k = rng.standard_normal((B, T, H, dk)).astype(f32)
    k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(f32)
    v = rng.standard_normal((B, T, H, dv)).astype(f32)
    b = rng.random((B, T, H, dk)).astype(f32)
    w = rng.random((B, T, H, dv)).astype(f32)
    g = (-0.3 * rng.random((B, T, H, dk))).astype(f32)
    S0 = (0.1 * rng.standard_normal((B, H, dk, dv))).astype(f32)
    return q, k, v, b, w, g, S0


def test_reduces_to_kda_when_both_gates_are_beta():
    q, k, v, _, _, g, S0 = _inputs()
    beta = np.random.default_rng(1).random(q.shape[:3]).astype(np.float32)
    erase = np.repeat(beta[..., None], q.shape[-1], axis=-1)
    write = np.repeat(beta[..., None], v.shape[-1], axis=-1)
    o2, s2 = oracle.fwd_gdn2(q, k, v, erase, write, g, S0)
    ok, sk = oracle.fwd(q, k, v, beta, g, S0, mode=oracle.MODE_KDA)
    np.testing.assert_allclose(o2, ok, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s2, sk, rtol=1e-12, atol=1e-13)


def test_erase_off_write_on_is_decayed_additive_attention():
    q, k, v, _, _, g, _ = _inputs(seed=2)
    zeros = np.zeros_like(k)
    ones = np.ones_like(v)
    o, _ = oracle.fwd_gdn2(q, k, v, zeros, ones, g, None)
    G = np.cumsum(g.astype(np.float64), axis=1)   # inclusive log-decay prefix per key channel
    B, T, H, dk = q.shape
    ref = np.zeros_like(o)
    for t in range(T):
        for j in range(t + 1):
            # key j decayed by the steps j+1 .. t, read by the query of token t
            w_tj = np.einsum("bhc,bhc->bh", k[:, j] * np.exp(G[:, t] - G[:, j]), q[:, t])
            ref[:, t] += w_tj[..., None] * v[:, j]
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_unit_keys_with_full_erase_and_write_are_written_exactly():
    q, k, v, _, _, g, S0 = _inputs(seed=3)
    rng = np.random.default_rng(5)
    axis = np.eye(k.shape[-1], dtype=np.float32)[rng.integers(0, k.shape[-1], size=k.shape[:3])]   # |k| = 1 exactly
    o, _ = oracle.fwd_gdn2(axis, axis, v, np.ones_like(axis), np.ones_like(v), g, S0)   # read with q = k
    np.testing.assert_allclose(o, v.astype(np.float64), rtol=0, atol=1e-12)


def test_brute_force_matrix_expansion():
    q, k, v, b, w, g, S0 = _inputs(B=1, T=8, H=1, dk=4, dv=4, seed=4)
    o, sf = oracle.fwd_gdn2(q, k, v, b, w, g, S0)
    W = S0[0, 0].astype(np.float64).T   # math orientation d_v x d_k
    for t in range(8):
        kt, qt = k[0, t, 0].astype(np.float64), q[0, t, 0].astype(np.float64)
        e = b[0, t, 0].astype(np.float64) * kt
        z = w[0, t, 0].astype(np.float64) * v[0, t, 0].astype(np.float64)
        Wt = W @ np.diag(np.exp(g[0, t, 0].astype(np.float64)))
        W = Wt @ (np.eye(4) - np.outer(e, kt)) + np.outer(z, kt)
        np.testing.assert_allclose(o[0, t, 0], W @ qt, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sf[0, 0], W.T, rtol=1e-12, atol=1e-12)
