"""The chunk algebra that the CUDA kernels implement, written out in fp64 and
checked against the token-by-token oracle on CPU.

The pages state the delta rule per token (linear-attention notes, Sec. 2.3
Eqs. 9-10 for DeltaNet, Sec. 2.4 Eqs. 15-17 for Gated DeltaNet, Sec. 2.5
Eqs. 18-20 for KDA, Sec. 2.6 Eqs. 21-24 for Gated DeltaNet-2) and do not print
the chunkwise form.  In H = S^T ([dk][dv]) every member of the family is

    H_t = D_t H_{t-1} - k_t (e_t^T D_t H_{t-1}) + k_t z_t^T,    o_t = H_t^T q_t,

with D_t the decay (1, alpha_t or Diag(a_t)), e_t the erase direction and z_t
the write (beta_t k_t and beta_t v_t for DeltaNet, Gated DeltaNet and KDA;
b_t * k_t and w_t * v_t for Gated DeltaNet-2).  Over a chunk with incoming state
H0, G the inclusive prefix of the log-decay and g_C its last row, the kernels use
    A  = strict_tril((E e^G)(K e^-G)^T),    T = (I + A)^-1,
    W  = T (E e^G),    U' = T Z,    P = tril((Q e^G)(K e^-G)^T),
    Q~ = Q e^G - P W,  K~ = K e^{g_C - G},
    O  = Q~ H0 + P U',    H_C = Diag(e^{g_C}) H0 + K~^T (U' - W H0),
and the state step is the affine map H_C = M H0 + N with M = Diag(e^{g_C}) - K~^T W
and N = K~^T U'.  Composing these maps over sequence segments gives every
segment's incoming state by a scan (the sequence split of a long sequence; this
composition is derived here, not on the pages).

Each identity is checked against the oracle to fp64 rounding, at chunk sizes that
leave a ragged tail, with a non-zero initial state, for every mode."""
import numpy as np
import pytest

import oracle


def _inputs(mode, B=2, T=37, H=2, dk=8, dv=6, seed=0):
    rng = np.random.default_rng(seed)
    f32 = np.float32
    q = rng.standard_normal((B, T, H, dk)).astype(f32)
    k = rng.standard_normal((B, T, H, dk))
    k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(f32)
    q = (q / np.linalg.norm(q, axis=-1, keepdims=True)).astype(f32)
    v = rng.standard_normal((B, T, H, dv)).astype(f32)
    beta = (1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))).astype(f32)
    if mode == oracle.MODE_GDN:
        gate = (-0.2 * rng.random((B, T, H))).astype(f32)
    elif mode in (oracle.MODE_KDA, "gdn2"):
        gate = (-0.2 * rng.random((B, T, H, dk))).astype(f32)
    else:
        gate = None
    S0 = (0.3 * rng.standard_normal((B, H, dk, dv))).astype(f32)
    erase = rng.random((B, T, H, dk)).astype(f32)
    write = rng.random((B, T, H, dv)).astype(f32)
    return q, k, v, beta, gate, S0, erase, write


def _per_token(mode, q, k, v, beta, gate, erase, write, b, h):
    """fp64 per-token operands of one (b, h): Q, K, erase E, write Z, log-decay [T, dk]."""
    f = lambda x: x[b, :, h].astype(np.float64)
    Q, K, V = f(q), f(k), f(v)
    T, dk = K.shape
    if mode == "gdn2":
        E, Z = K * f(erase), V * f(write)
    else:
        bt = beta[b, :, h].astype(np.float64)[:, None]
        E, Z = bt * K, bt * V
    if gate is None:
        lg = np.zeros((T, dk))
    elif gate.ndim == 3:
        lg = np.repeat(gate[b, :, h].astype(np.float64)[:, None], dk, axis=1)
    else:
        lg = gate[b, :, h].astype(np.float64)
    return Q, K, E, Z, lg


def _chunk(Q, K, E, Z, lg, H0):
    """One chunk: (O, H_C, M, N) by the chunk algebra above."""
    L = K.shape[0]
    G = np.cumsum(lg, axis=0)                  # inclusive prefix, per row and key channel
    gC = G[-1]
    A = np.tril((E * np.exp(G)) @ (K * np.exp(-G)).T, -1)
    Tm = np.linalg.inv(np.eye(L) + A)          # unit lower-triangular
    W = Tm @ (E * np.exp(G))
    Up = Tm @ Z
    P = np.tril((Q * np.exp(G)) @ (K * np.exp(-G)).T)
    Qt = Q * np.exp(G) - P @ W
    Kt = K * np.exp(gC - G)
    O = Qt @ H0 + P @ Up
    U = Up - W @ H0
    HC = np.exp(gC)[:, None] * H0 + Kt.T @ U
    M = np.diag(np.exp(gC)) - Kt.T @ W
    N = Kt.T @ Up
    return O, HC, M, N


def _run_chunks(mode, ins, C):
    q, k, v, beta, gate, S0, erase, write = ins
    B, T, Hh, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, T, Hh, dv))
    sf = np.zeros((B, Hh, dk, dv))
    maps = {}
    for b in range(B):
        for h in range(Hh):
            Q, K, E, Z, lg = _per_token(mode, q, k, v, beta, gate, erase, write, b, h)
            Hs = S0[b, h].astype(np.float64)
            maps[b, h] = []
            for t0 in range(0, T, C):
                sl = slice(t0, min(T, t0 + C))
                O, HC, M, N = _chunk(Q[sl], K[sl], E[sl], Z[sl], lg[sl], Hs)
                np.testing.assert_allclose(M @ Hs + N, HC, rtol=1e-12, atol=1e-12)   # affine form
                maps[b, h].append((M, N))
                out[b, sl, h] = O
                Hs = HC
            sf[b, h] = Hs
    return out, sf, maps


def _oracle(mode, ins):
    q, k, v, beta, gate, S0, erase, write = ins
    if mode == "gdn2":
        return oracle.fwd_gdn2(q, k, v, erase, write, gate, S0)
    return oracle.fwd(q, k, v, beta, gate, S0, mode=mode)


MODES = [oracle.MODE_DELTANET, oracle.MODE_GDN, oracle.MODE_KDA, "gdn2"]


def _close(a, ref, tol=1e-10):
    err = np.max(np.abs(a - ref)) / np.sqrt(np.mean(ref ** 2))
    assert err <= tol, f"max |err| / rms = {err:.3g}"


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_chunk_form_equals_recurrence(mode, C):
    """O = Q~ H0 + P U' and H_C = Diag(e^{g_C}) H0 + K~^T (U' - W H0), chunk after chunk,
    give the recurrence's outputs and final state (T = 37: every C leaves a tail)."""
    ins = _inputs(mode, seed=C)
    o, s, _ = _run_chunks(mode, ins, C)
    ro, rs = _oracle(mode, ins)
    _close(o, ro)
    _close(s, rs)


@pytest.mark.parametrize("mode", MODES)
def test_chunk_form_at_kernel_chunk_size(mode):
    """The kernels' chunk of 64 over two full chunks and a 22-row tail, dk = 16."""
    ins = _inputs(mode, B=1, T=150, H=2, dk=16, dv=8, seed=7)
    o, s, _ = _run_chunks(mode, ins, 64)
    ro, rs = _oracle(mode, ins)
    _close(o, ro)
    _close(s, rs)


@pytest.mark.parametrize("mode", MODES)
def test_transform_matrix_is_unit_lower_triangular(mode):
    """T = (I + A)^-1 with A strictly lower: T is unit lower-triangular, so the UT/WY
    solve is a forward substitution (no pivoting) in every mode."""
    q, k, v, beta, gate, S0, erase, write = _inputs(mode, T=16, seed=3)
    Q, K, E, Z, lg = _per_token(mode, q, k, v, beta, gate, erase, write, 0, 0)
    G = np.cumsum(lg, axis=0)
    A = np.tril((E * np.exp(G)) @ (K * np.exp(-G)).T, -1)
    Tm = np.linalg.inv(np.eye(16) + A)
    np.testing.assert_allclose(np.triu(Tm, 1), 0.0, atol=1e-13)
    np.testing.assert_allclose(np.diag(Tm), 1.0, atol=1e-13)
    # forward substitution row by row gives the same matrix
    Tf = np.eye(16)
    for i in range(16):
        Tf[i, :i] = -A[i, :i] @ Tf[:i, :i]
    np.testing.assert_allclose(Tf, Tm, atol=1e-11)


@pytest.mark.parametrize("mode", MODES)
def test_segment_maps_compose_by_scan(mode):
    """Splitting the sequence into segments: each segment's affine map (M, N) is the
    composition of its chunks' maps; an exclusive scan of the segment maps applied to
    S0 gives every segment's incoming state, and running each segment alone from that
    state gives the whole sequence's outputs and final state."""
    T, C, seg_chunks = 96, 8, 3                # 12 chunks in 4 segments of 24 tokens
    ins = _inputs(mode, B=1, T=T, H=1, dk=8, dv=5, seed=11)
    o_ref, s_ref = _oracle(mode, ins)
    _, _, maps = _run_chunks(mode, ins, C)
    chunk_maps = maps[0, 0]
    Hin = ins[5][0, 0].astype(np.float64)
    seg_T = C * seg_chunks
    for i, s0 in enumerate(range(0, len(chunk_maps), seg_chunks)):
        M, N = np.eye(8), np.zeros((8, 5))
        for Mc, Nc in chunk_maps[s0:s0 + seg_chunks]:
            M, N = Mc @ M, Mc @ N + Nc         # apply (M, N), then (Mc, Nc)
        sl = slice(i * seg_T, (i + 1) * seg_T)
        seg = tuple(x[:, sl] if x is not None and x.ndim >= 3 and x.shape[1] == T else x for x in ins)
        seg = seg[:5] + (Hin[None, None],) + seg[6:]
        po, ps, _ = _run_chunks(mode, seg, C)
        _close(po, o_ref[:, sl])
        Hin = M @ Hin + N
        _close(ps[0, 0], Hin)
    _close(Hin, s_ref[0, 0])
