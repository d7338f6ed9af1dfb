"""Pins of the RLA / RDN oracle (Residual Linear Attention notes, Sec. 2.2-2.4)
against what the notes and the algebra fix, independent of its token loop:

  * RLA against its closed form: both states are decayed sums of their writes
    (the notes write R_t that way in Sec. 2.3), so S_{t-1}, r_t, R_t and o_t are
    formed here as explicit sums over earlier tokens, in numpy fp64;
  * RDN against the composition of the Gated DeltaNet oracle (pinned on its
    own): the base state is Gated DeltaNet on (v, beta), the residual state is
    Gated DeltaNet on (r, gamma), read after its update;
  * the notes' one-step expansion of the RLA output,
    o_t = alpha S_{t-1} q + alpha gamma R_{t-1} q + gamma^2 r (k . q);
  * the clip bound, with and without clipping."""
import numpy as np
import pytest

import oracle


def _inputs(B=2, T=7, H=2, dk=4, dv=3, seed=0, vscale=1.0):
    rng = np.random.default_rng(seed)
    f32 = np.float32
    q = rng.standard_normal((B, T, H, dk)).astype(f32)
    k = rng.standard_normal((B, T, H, dk)).astype(f32)
    k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(f32)
    v = (vscale * rng.standard_normal((B, T, H, dv))).astype(f32)
    beta = rng.random((B, T, H)).astype(f32)
    gamma = rng.random((B, T, H)).astype(f32)
    gate = (-0.5 * rng.random((B, T, H))).astype(f32)
    S0 = (0.3 * rng.standard_normal((B, H, dk, dv))).astype(f32)
    R0 = (0.3 * rng.standard_normal((B, H, dk, dv))).astype(f32)
    return q, k, v, beta, gamma, gate, S0, R0


def _rla_closed_form(q, k, v, beta, gamma, gate, S0, R0, c):
    """Explicit sums, math orientation (dv x dk), per (b, h)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    d = lambda a: np.asarray(a, np.float64)
    q, k, v, beta, gamma, gate = map(d, (q, k, v, beta, gamma, gate))
    o = np.zeros((B, T, H, dv))
    Sf, Rf = np.zeros((B, H, dk, dv)), np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            G = np.concatenate([[0.0], np.cumsum(gate[b, :, h])])   # G[t] = sum of log alpha over tokens < t
            S0m, R0m = d(S0[b, h]).T, d(R0[b, h]).T
            r = np.zeros((T, dv))
            for t in range(T + 1):
                # base state after tokens < t: S_{t-1} in the notes' 1-based count
                S = np.exp(G[t]) * S0m
                for i in range(t):
                    S = S + np.exp(G[t] - G[i + 1]) * beta[b, i, h] * np.outer(v[b, i, h], k[b, i, h])
                if t == T:
                    Sf[b, h] = S.T
                    break
                r[t] = np.clip(v[b, t, h] - S @ k[b, t, h], -c, c)
                R = np.exp(G[t + 1]) * R0m
                for i in range(t + 1):
                    R = R + np.exp(G[t + 1] - G[i + 1]) * gamma[b, i, h] * np.outer(r[i], k[b, i, h])
                o[b, t, h] = np.exp(gate[b, t, h]) * (S @ q[b, t, h]) + gamma[b, t, h] * (R @ q[b, t, h])
                if t == T - 1:
                    Rf[b, h] = R.T
    return o, Sf, Rf


@pytest.mark.parametrize("clip", [0.25, 1.0, np.inf])   # exact in fp32, the clip bound's input type
def test_rla_matches_its_closed_form(clip):
    x = _inputs(vscale=2.0)
    o, sf, rf = oracle.fwd_rla(*x[:6], clip=clip, S0=x[6], R0=x[7], delta=False)
    ro, rsf, rrf = _rla_closed_form(*x, c=clip)
    np.testing.assert_allclose(o, ro, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(sf, rsf, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(rf, rrf, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("clip", [0.3, np.inf])
def test_rdn_is_gated_deltanet_twice(clip):
    q, k, v, beta, gamma, gate, S0, R0 = _inputs(T=6, seed=1, vscale=1.5)
    B, T, H, dk = q.shape
    o, sf, rf = oracle.fwd_rla(q, k, v, beta, gamma, gate, clip=clip, S0=S0, R0=R0, delta=True)
    # base state: Gated DeltaNet on (v, beta); S_{t-1} from prefix runs
    prev = [S0.astype(np.float64)]
    for t in range(1, T + 1):
        _, s = oracle.fwd(q[:, :t], k[:, :t], v[:, :t], beta[:, :t], gate[:, :t], S0, mode=oracle.MODE_GDN)
        prev.append(s)
    np.testing.assert_allclose(sf, prev[T], rtol=1e-11, atol=1e-12)
    # residuals against the old base state (memory orientation: S^T, so S k = einsum over dk)
    r = np.stack([np.clip(v[:, t].astype(np.float64) - np.einsum("bhcd,bhc->bhd", prev[t], k[:, t]), -clip, clip)
                  for t in range(T)], axis=1)
    # residual state: Gated DeltaNet on (r, gamma), read after its update
    ro2, rs2 = oracle.fwd(q, k, r.astype(np.float32), gamma, gate, R0, mode=oracle.MODE_GDN)
    base = np.stack([np.exp(gate[:, t].astype(np.float64))[..., None] *
                     np.einsum("bhcd,bhc->bhd", prev[t], q[:, t]) for t in range(T)], axis=1)
    want = base + gamma.astype(np.float64)[..., None] * ro2
    # r passes through fp32 on its way into the Gated DeltaNet oracle
    np.testing.assert_allclose(o, want, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(rf, rs2, rtol=1e-5, atol=1e-6)


def test_rla_one_step_expansion():
    q, k, v, beta, gamma, gate, S0, R0 = _inputs(T=5, seed=2)
    o, _, _ = oracle.fwd_rla(q, k, v, beta, gamma, gate, clip=0.5, S0=S0, R0=R0)
    for t in range(1, 5):
        _, S, R = oracle.fwd_rla(q[:, :t], k[:, :t], v[:, :t], beta[:, :t], gamma[:, :t], gate[:, :t], clip=0.5,
                                 S0=S0, R0=R0)
        a = np.exp(gate[:, t].astype(np.float64))[..., None]
        g = gamma[:, t].astype(np.float64)[..., None]
        Sq = np.einsum("bhcd,bhc->bhd", S, q[:, t])
        Rq = np.einsum("bhcd,bhc->bhd", R, q[:, t])
        r = np.clip(v[:, t] - np.einsum("bhcd,bhc->bhd", S, k[:, t]), -0.5, 0.5)
        kq = np.einsum("bhc,bhc->bh", k[:, t].astype(np.float64), q[:, t])[..., None]
        np.testing.assert_allclose(o[:, t], a * Sq + a * g * Rq + g * g * r * kq, rtol=1e-11, atol=1e-12)


def test_clip_bounds_every_residual():
    """With gamma = 1, alpha = 1, R0 = 0, zero base state and a single token, the
    output is R_1 q = r (k . q), and |r| <= c."""
    q, k, v, beta, gamma, gate, _, _ = _inputs(T=1, seed=3, vscale=10.0)
    o, _, rf = oracle.fwd_rla(q, k, v, beta, np.ones_like(gamma), np.zeros_like(gate), clip=0.25)
    r = np.einsum("bhcd->bhd", rf * k[:, 0][..., None]) / np.sum(k[:, 0] ** 2, axis=-1)[..., None]
    assert np.max(np.abs(r)) <= 0.25 * (1 + 1e-8)   # r recovered from R_1 by a division
    np.testing.assert_allclose(np.abs(r), 0.25, rtol=1e-6)   # |v| >> c: every component clipped
