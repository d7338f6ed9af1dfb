"""Pins for the fp64 oracle: facts the pages and the mathematics fix.

None of these re-types the oracle's loop.  Each test checks the oracle against
something independent of it: a number the pages print, a closed form, an
invariant, a special case that reduces to a textbook formula, or a brute force
by explicit matrix products.  Citations name the page and the section /
equation the fact comes from.

Pages:
  [LA]  "Linear Attention Architectures: Mechanisms, Trade-offs, and
        Cross-Layer Routing" (reading notes)
  [RLA] "Residual Linear Attention" (reading notes)
  [SR]  "State reduction by key/query channel pruning" (reading notes)
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
DN, GDN, KDA = oracle.MODE_DELTANET, oracle.MODE_GDN, oracle.MODE_KDA


def _unit(x, axis=-1):
    return x / np.linalg.norm(x, axis=axis, keepdims=True)


def _rand_case(rng, B=2, T=9, H=3, dk=6, dv=5, mode=GDN, s0=True, strength=0.3):
    q = _unit(rng.standard_normal((B, T, H, dk)))
    k = _unit(rng.standard_normal((B, T, H, dk)))
    v = rng.standard_normal((B, T, H, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    if mode == GDN:
        gate = -strength * np.logaddexp(0, rng.standard_normal((B, T, H)))
    elif mode == KDA:
        gate = -strength * np.logaddexp(0, rng.standard_normal((B, T, H, dk)))
    else:
        gate = None
    S0 = 0.3 * rng.standard_normal((B, H, dk, dv)) if s0 else None
    # The oracle reads fp32 inputs; round here so the tests see the same values.
    f = lambda a: None if a is None else np.asarray(a, dtype=np.float32).astype(np.float64)
    return dict(q=f(q), k=f(k), v=f(v), beta=f(beta), gate=f(gate), S0=f(S0), mode=mode)


def _decay_factors(gate, mode, dk):
    """Per-token key-channel retention a_t (shape [..., dk]) for any mode."""
    if mode == DN or gate is None:
        return None
    if mode == GDN:
        return np.repeat(np.exp(gate)[..., None], dk, axis=-1)
    return np.exp(gate)


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, val = line.split()
                vals[key] = float(val)
    return vals


# ---------------------------------------------------------------------------
# [LA] Sec. 2.3: the printed worked example (golden fixture).
def test_worked_example_prediction_2_to_3_5():
    g = _read_golden("worked_example_deltanet.txt")
    dk, dv = 4, 1
    key = np.zeros(dk); key[1] = 1.0                      # unit key
    other = np.zeros(dk); other[3] = 1.0                  # orthogonal direction
    # Memory (math orientation W is dv x dk) predicting 2 for the key and 7 for `other`.
    W0 = np.zeros((dv, dk)); W0[0, 1] = g["prediction_before"]; W0[0, 3] = 7.0
    S0 = W0.T[None, None]                                 # memory orientation [B,H,dk,dv]
    for query, want in ((key, g["prediction_after"]), (other, 7.0)):
        o, _ = oracle.fwd(query[None, None, None], key[None, None, None],
                          np.full((1, 1, 1, dv), g["target_value"]), np.full((1, 1, 1), g["beta"]),
                          S0=S0, mode=DN)
        assert o[0, 0, 0, 0] == pytest.approx(want, abs=1e-12)


# [LA] Sec. 2.3: with a unit key the new prediction is (1 - beta) * old + beta * v,
# for every mode once the forget step has been applied (Sec. 2.4, 2.5).
@pytest.mark.parametrize("mode", [DN, GDN, KDA])
def test_exact_write_at_beta_one(mode):
    rng = np.random.default_rng(1)
    c = _rand_case(rng, mode=mode)
    c["beta"] = np.ones_like(c["beta"])
    # keys of exactly unit norm in fp32: four entries of +-1/2 at random places
    B, T, H, dk = c["k"].shape
    k = np.zeros((B, T, H, dk))
    for idx in np.ndindex(B, T, H):
        pos = rng.choice(dk, size=4, replace=False)
        k[idx][pos] = 0.5 * rng.choice([-1.0, 1.0], size=4)
    c["k"] = k
    c["q"] = k.copy()                                     # read back along the key just written
    o, _ = oracle.fwd(**c)
    np.testing.assert_allclose(o, c["v"], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# [RLA] Sec. 1.2: Gated DeltaNet prediction-correction decomposition
#   o_t = alpha_t S_{t-1} q_t + beta_t (v_t - alpha_t S_{t-1} k_t)(k_t^T q_t),
# with S_{t-1} taken from an independent run that stops one token earlier.
# The KDA version replaces alpha_t S_{t-1} by S_{t-1} Diag(a_t) ([LA] Eqs. 18-20).
@pytest.mark.parametrize("mode", [DN, GDN, KDA])
def test_prediction_correction_identity(mode):
    rng = np.random.default_rng(2)
    c = _rand_case(rng, T=7, mode=mode)
    o, _ = oracle.fwd(**c)
    dk = c["q"].shape[-1]
    a = _decay_factors(c["gate"], mode, dk)
    for t in range(c["q"].shape[1]):
        sl = lambda x: None if x is None else x[:, :t]
        _, Sprev = oracle.fwd(sl(c["q"]), sl(c["k"]), sl(c["v"]), sl(c["beta"]), sl(c["gate"]),
                              c["S0"], mode=mode)                   # [B,H,dk,dv] = S_{t-1}^T
        W = np.swapaxes(Sprev, -1, -2)                              # [B,H,dv,dk]
        if a is not None:
            W = W * a[:, t][:, :, None, :]                          # S_{t-1} Diag(a_t)
        qt, kt, vt, bt = c["q"][:, t], c["k"][:, t], c["v"][:, t], c["beta"][:, t]
        base = np.einsum("bhic,bhc->bhi", W, qt)
        pred = np.einsum("bhic,bhc->bhi", W, kt)
        kq = np.einsum("bhc,bhc->bh", kt, qt)
        want = base + bt[..., None] * (vt - pred) * kq[..., None]
        np.testing.assert_allclose(o[:, t], want, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Closed form with axis-aligned keys k_t = e_{c_t}: every state column evolves
# as its own scalar system (per-channel independence, [SR] Sec. 2.5), and the
# key column is rewritten as (1 - beta) * decayed + beta * v ([LA] Sec. 2.3),
# while untouched columns only decay by their own key-channel gate, because
# Diag(a) acts on the right ([LA] Sec. 2.5).
@pytest.mark.parametrize("mode", [DN, GDN, KDA])
def test_axis_keys_closed_form(mode):
    rng = np.random.default_rng(3)
    B, T, H, dk, dv = 1, 12, 2, 4, 3
    c = _rand_case(rng, B=B, T=T, H=H, dk=dk, dv=dv, mode=mode, strength=0.7)
    axes = rng.integers(0, dk, size=(B, T, H))             # repeats allowed
    k = np.zeros((B, T, H, dk)); np.put_along_axis(k, axes[..., None], 1.0, axis=-1)
    c["k"] = k
    o, S = oracle.fwd(**c)
    a = _decay_factors(c["gate"], mode, dk)
    W = np.swapaxes(c["S0"], -1, -2).copy()                 # [B,H,dv,dk]
    for t in range(T):
        for b in range(B):
            for h in range(H):
                for col in range(dk):
                    keep = 1.0 if a is None else a[b, t, h, col]
                    W[b, h, :, col] *= keep
                ct = axes[b, t, h]
                bt = c["beta"][b, t, h]
                W[b, h, :, ct] = (1 - bt) * W[b, h, :, ct] + bt * c["v"][b, t, h]
                want = W[b, h] @ c["q"][b, t, h]
                np.testing.assert_allclose(o[b, t, h], want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, np.swapaxes(W, -1, -2), rtol=0, atol=1e-12)


# Closed form with orthonormal keys and S0 = 0: the delta correction vanishes
# (S_{t-1} k_t = 0), so the rule reduces to decayed additive linear attention
# ([LA] Eqs. 4-5; [SR] Sec. 2.1):  o_t = sum_{j<=t} (prod_{i=j+1..t} alpha_i) beta_j v_j (k_j . q_t).
@pytest.mark.parametrize("mode", [DN, GDN])
def test_orthonormal_keys_reduce_to_gated_linear_attention(mode):
    rng = np.random.default_rng(4)
    B, T, H, d = 2, 6, 2, 8
    c = _rand_case(rng, B=B, T=T, H=H, dk=d, dv=5, mode=mode, s0=False)
    # Keys exactly orthonormal in fp32: rows of two 4x4 Hadamard blocks scaled
    # by 1/2, under a random signed permutation of the coordinates.
    H4 = 0.5 * np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]], float)
    basis = np.zeros((d, d)); basis[:4, :4] = H4; basis[4:, 4:] = H4
    for b in range(B):
        for h in range(H):
            P = np.eye(d)[rng.permutation(d)] * rng.choice([-1.0, 1.0], size=d)
            c["k"][b, :, h] = (basis @ P)[rng.permutation(d)[:T]]
    o, _ = oracle.fwd(**c)
    g = np.zeros((B, T, H)) if mode == DN else c["gate"]
    G = np.cumsum(g, axis=1)                                          # [B,T,H]
    for b in range(B):
        for h in range(H):
            Qb, Kb, Vb = c["q"][b, :, h], c["k"][b, :, h], c["v"][b, :, h]
            decay = np.exp(G[b, :, h][:, None] - G[b, :, h][None, :])  # prod_{i=j+1..t} alpha_i
            A = np.tril(Qb @ Kb.T * decay) * c["beta"][b, :, h][None, :]
            np.testing.assert_allclose(o[b, :, h], A @ Vb, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Linear-attention limit ([LA] Eqs. 4-5; [SR] Sec. 2.1).  (i) beta = 0 leaves the
# memory to its forget gate alone: o_t = (prod_{i<=t} alpha_i) S0 q_t.  (ii) As
# beta = eps -> 0 with S0 = 0, o_t / eps tends to causal (decayed) linear attention
# (tril(Q K^T) * Gamma) V, the textbook matrix form, with an O(eps * T) error.
@pytest.mark.parametrize("mode", [DN, GDN])
def test_linear_attention_limit(mode):
    rng = np.random.default_rng(5)
    c = _rand_case(rng, B=1, T=10, H=2, dk=6, dv=4, mode=mode)
    g = np.zeros(c["beta"].shape) if mode == DN else c["gate"]
    G = np.cumsum(g, axis=1)
    c0 = dict(c); c0["beta"] = np.zeros_like(c["beta"])
    o, S = oracle.fwd(**c0)
    want = np.exp(G)[..., None] * np.einsum("bhcv,bthc->bthv", c["S0"], c["q"])
    np.testing.assert_allclose(o, want, rtol=0, atol=1e-12)

    eps = 1e-7
    ce = dict(c); ce["beta"] = np.full_like(c["beta"], eps); ce["S0"] = None
    o, _ = oracle.fwd(**ce)
    for h in range(2):
        Qb, Kb, Vb = c["q"][0, :, h], c["k"][0, :, h], c["v"][0, :, h]
        decay = np.exp(G[0, :, h][:, None] - G[0, :, h][None, :])
        want = np.tril(Qb @ Kb.T * decay) @ Vb
        err = np.max(np.abs(o[0, :, h] / eps - want))
        assert err < 50 * eps * 10 * np.max(np.abs(want)), err


# ---------------------------------------------------------------------------
# [SR] Sec. 2.5, Prop. 3.1: orthogonal change of key basis (k' = T k, q' = T q,
# S' = S T^T) leaves every output unchanged; this holds for DeltaNet and for a
# scalar decay (Gated DeltaNet).  For KDA it holds for permutations of the key
# channels when the per-channel gates are permuted with them.
@pytest.mark.parametrize("mode", [DN, GDN, KDA])
def test_orthogonal_invariance(mode):
    rng = np.random.default_rng(6)
    c = _rand_case(rng, B=2, T=11, H=2, dk=6, dv=4, mode=mode)
    o, S = oracle.fwd(**c)
    if mode == KDA:
        perm = rng.permutation(6)
        Tm = np.eye(6)[perm]
    else:
        Tm, _ = np.linalg.qr(rng.standard_normal((6, 6)))
    c2 = dict(c)
    c2["q"] = np.einsum("ij,bthj->bthi", Tm, c["q"])
    c2["k"] = np.einsum("ij,bthj->bthi", Tm, c["k"])
    c2["S0"] = np.einsum("ij,bhjv->bhiv", Tm, c["S0"])      # memory orientation: H' = T H
    if mode == KDA:
        c2["gate"] = c["gate"][..., perm]
    o2, S2 = oracle.fwd(**c2)
    # A rotation is applied in fp64 and re-rounded to the oracle's fp32 inputs,
    # so a general rotation agrees to fp32 input resolution; a permutation is exact.
    tol = 0.0 if mode == KDA else 1e-5
    np.testing.assert_allclose(o2, o, rtol=0, atol=tol * np.abs(o).max() + 1e-13)
    np.testing.assert_allclose(S2, np.einsum("ij,bhjv->bhiv", Tm, S), rtol=0,
                               atol=tol * np.abs(S).max() + 1e-13)


# [SR] Sec. 2.5: each value channel is an independent linear time-varying
# system sharing the key-side transition, so running one value channel at a
# time (d_v = 1) reproduces every column of the full run, and permuting the
# value channels permutes outputs and state columns.
@pytest.mark.parametrize("mode", [DN, GDN, KDA])
def test_value_channel_independence(mode):
    rng = np.random.default_rng(7)
    c = _rand_case(rng, B=1, T=8, H=2, dk=5, dv=4, mode=mode)
    o, S = oracle.fwd(**c)
    for i in range(4):
        ci = dict(c); ci["v"] = c["v"][..., i:i + 1]; ci["S0"] = c["S0"][..., i:i + 1]
        oi, Si = oracle.fwd(**ci)
        np.testing.assert_allclose(oi[..., 0], o[..., i], rtol=0, atol=1e-13)
        np.testing.assert_allclose(Si[..., 0], S[..., i], rtol=0, atol=1e-13)
    perm = np.array([2, 0, 3, 1])
    cp = dict(c); cp["v"] = c["v"][..., perm]; cp["S0"] = c["S0"][..., perm]
    op, Sp = oracle.fwd(**cp)
    np.testing.assert_array_equal(op, o[..., perm])
    np.testing.assert_array_equal(Sp, S[..., perm])


# [SR] Eq. 3: with S0 = 0 the state's rank is at most the number of tokens seen
# and at most the rank of the values written.
@pytest.mark.parametrize("mode", [DN, GDN, KDA])
def test_rank_bound(mode):
    rng = np.random.default_rng(8)
    c = _rand_case(rng, B=1, T=8, H=1, dk=8, dv=8, mode=mode, s0=False)
    # small integers keep the span exact after the oracle's fp32 input rounding
    basis = rng.integers(-3, 4, size=(2, 8)).astype(float)
    c["v"][0, 4:, 0] = rng.integers(-3, 4, size=(4, 2)) @ basis  # late values in a 2-D span
    for t in range(1, 9):
        sl = lambda x: None if x is None else x[:, :t]
        _, S = oracle.fwd(sl(c["q"]), sl(c["k"]), sl(c["v"]), sl(c["beta"]), sl(c["gate"]),
                          None, mode=mode)
        sv = np.linalg.svd(S[0, 0], compute_uv=False)
        assert np.sum(sv > 1e-10 * sv[0]) <= t
    # values only from a 2-D span from the start: rank <= 2 at every length
    c["v"][0, :, 0] = rng.integers(-3, 4, size=(8, 2)) @ basis
    _, S = oracle.fwd(c["q"], c["k"], c["v"], c["beta"], c["gate"], None, mode=mode)
    sv = np.linalg.svd(S[0, 0], compute_uv=False)
    assert np.sum(sv > 1e-10 * sv[0]) <= 2


# [RLA] Sec. 2.4: for a unit key, (I - beta k k^T) has eigenvalue 1 - beta along k
# and 1 elsewhere; with v = 0 and alpha <= 1 the state can only shrink.
@pytest.mark.parametrize("mode", [DN, GDN, KDA])
def test_contraction_without_values(mode):
    rng = np.random.default_rng(9)
    c = _rand_case(rng, B=1, T=12, H=2, dk=6, dv=5, mode=mode)
    c["v"] = np.zeros_like(c["v"])
    prev = np.linalg.norm(c["S0"], axis=(-2, -1))
    for t in range(1, 13):
        sl = lambda x: None if x is None else x[:, :t]
        _, S = oracle.fwd(sl(c["q"]), sl(c["k"]), sl(c["v"]), sl(c["beta"]), sl(c["gate"]),
                          c["S0"], mode=mode)
        nrm = np.linalg.norm(S, axis=(-2, -1))
        assert np.all(nrm <= prev * (1 + 1e-12))
        prev = nrm
    # One DeltaNet step with v = 0 is W_1 = W_0 (I - beta k k^T): along k the
    # prediction scales by 1 - beta |k|^2 (= 1 - beta for a unit key), and an
    # orthogonal direction u keeps its old prediction.
    k = _unit(rng.standard_normal(6)).astype(np.float32).astype(np.float64)
    u = rng.standard_normal(6); u -= (u @ k) * k / (k @ k)
    S0 = rng.standard_normal((1, 1, 6, 5)).astype(np.float32).astype(np.float64)
    beta = float(np.float32(0.37))
    _, S1 = oracle.fwd(u[None, None, None], k[None, None, None], np.zeros((1, 1, 1, 5)),
                       np.full((1, 1, 1), beta), S0=S0, mode=DN)
    W0, W1 = S0[0, 0].T, S1[0, 0].T
    np.testing.assert_allclose(W1 @ k, (1 - beta * (k @ k)) * (W0 @ k), rtol=0, atol=1e-12)
    np.testing.assert_allclose(W1 @ u, W0 @ u - beta * (W0 @ k) * (k @ u), rtol=0, atol=1e-12)
    assert abs(k @ k - 1) < 1e-6


# ---------------------------------------------------------------------------
# State passing: the initial state is an input, so one run over T1 + T2 tokens
# equals a run over T1 tokens whose final state seeds a run over the next T2.
@pytest.mark.parametrize("mode", [DN, GDN, KDA])
def test_state_passing(mode):
    rng = np.random.default_rng(10)
    c = _rand_case(rng, B=2, T=13, H=2, dk=5, dv=3, mode=mode)
    o, S = oracle.fwd(**c)
    cut = 6
    a = lambda x, s: None if x is None else x[:, s]
    o1, S1 = oracle.fwd(a(c["q"], slice(0, cut)), a(c["k"], slice(0, cut)), a(c["v"], slice(0, cut)),
                        a(c["beta"], slice(0, cut)), a(c["gate"], slice(0, cut)), c["S0"], mode=mode)
    o2, S2 = oracle.fwd(a(c["q"], slice(cut, None)), a(c["k"], slice(cut, None)),
                        a(c["v"], slice(cut, None)), a(c["beta"], slice(cut, None)),
                        a(c["gate"], slice(cut, None)), S1, mode=mode)
    # S1 is re-read as fp32 by the second call: compare at fp32 resolution.
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), o, rtol=0, atol=1e-6)
    np.testing.assert_allclose(S2, S, rtol=0, atol=1e-6)


# Mode reductions: KDA with a gate equal on every key channel is Gated DeltaNet
# ([LA] Sec. 2.5); Gated DeltaNet with alpha = 1 (log-gate 0) is DeltaNet.
def test_mode_reductions():
    rng = np.random.default_rng(11)
    c = _rand_case(rng, mode=GDN)
    o_gdn, S_gdn = oracle.fwd(**c)
    ck = dict(c); ck["mode"] = KDA
    ck["gate"] = np.repeat(c["gate"][..., None], c["q"].shape[-1], axis=-1)
    o_kda, S_kda = oracle.fwd(**ck)
    np.testing.assert_array_equal(o_kda, o_gdn)
    np.testing.assert_array_equal(S_kda, S_gdn)
    cz = dict(c); cz["gate"] = np.zeros_like(c["gate"])
    o_g0, _ = oracle.fwd(**cz)
    cd = dict(c); cd["mode"] = DN; cd["gate"] = None
    o_dn, _ = oracle.fwd(**cd)
    np.testing.assert_array_equal(o_g0, o_dn)


# Brute force at d = 4, T = 8 by explicit matrix products of the expanded update
# ([LA] Eq. 14 with the forget step of Eqs. 15-20):
#   W_t = W_{t-1} D_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = W_t q_t.
@pytest.mark.parametrize("mode", [DN, GDN, KDA])
def test_brute_force_matrix_products(mode):
    rng = np.random.default_rng(12)
    c = _rand_case(rng, B=1, T=8, H=1, dk=4, dv=4, mode=mode)
    # unnormalised keys exercise the general (non-unit) form too
    c["k"] = np.asarray(1.3 * c["k"] + 0.2, np.float32).astype(np.float64)
    o, S = oracle.fwd(**c)
    a = _decay_factors(c["gate"], mode, 4)
    W = c["S0"][0, 0].T.copy()
    I = np.eye(4)
    for t in range(8):
        k, v, q, b = c["k"][0, t, 0], c["v"][0, t, 0], c["q"][0, t, 0], c["beta"][0, t, 0]
        D = I if a is None else np.diag(a[0, t, 0])
        W = W @ D @ (I - b * np.outer(k, k)) + b * np.outer(v, k)
        np.testing.assert_allclose(o[0, t, 0], W @ q, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S[0, 0], W.T, rtol=0, atol=1e-12)


# Edge cases of the interface: no tokens returns the initial state unchanged;
# a missing initial state means zeros.
def test_empty_and_zero_state():
    rng = np.random.default_rng(13)
    c = _rand_case(rng, T=0, mode=GDN)
    o, S = oracle.fwd(**c)
    assert o.shape[1] == 0
    np.testing.assert_array_equal(S, c["S0"].astype(np.float32))
    c = _rand_case(rng, T=5, mode=KDA)
    cz = dict(c); cz["S0"] = np.zeros_like(c["S0"])
    cn = dict(c); cn["S0"] = None
    np.testing.assert_array_equal(oracle.fwd(**cz)[0], oracle.fwd(**cn)[0])


# The decode helper is the same recurrence one token at a time.
def test_decode_matches_sequence_run():
    rng = np.random.default_rng(14)
    c = _rand_case(rng, B=3, T=5, H=2, mode=GDN)
    o, S = oracle.fwd(**c)
    sw = lambda x: np.swapaxes(x, 0, 1)
    od, Sd = oracle.decode(sw(c["q"]), sw(c["k"]), sw(c["v"]), sw(c["beta"]), sw(c["gate"]), c["S0"])
    np.testing.assert_array_equal(sw(od), o)
    np.testing.assert_array_equal(Sd, S)


def test_threads_do_not_change_results():
    rng = np.random.default_rng(15)
    c = _rand_case(rng, B=3, T=20, H=5, mode=KDA)
    o1, S1 = oracle.fwd(**c, nthreads=1)
    o4, S4 = oracle.fwd(**c, nthreads=4)
    np.testing.assert_array_equal(o1, o4)
    np.testing.assert_array_equal(S1, S4)
