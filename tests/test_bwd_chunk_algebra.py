"""The chunkwise backward that the CUDA kernels implement, written out in fp64
and checked against the token-by-token backward oracle on CPU (DeltaNet and
Gated DeltaNet, scalar decay).

The pages give the recurrence per token and no chunk form of its derivative
(the method sources describe a first-order backward that keeps the state
history, checked in fp64).  In H = S^T ([dk][dv]), over a chunk with incoming
state H0, g the inclusive prefix of the log-decay, Gamma_rj = e^{g_r - g_j},
ge = e^{g}, gc = e^{g_last - g} and gamma = e^{g_last}, the forward is

    A = strict_tril(Diag(beta) (K K^T * Gamma)),   T = (I + A)^-1,
    W = T Diag(beta ge) K,   U' = T Diag(beta) V,   U = U' - W H0,
    P = tril(Q K^T * Gamma),   O = Diag(ge) Q H0 + P U,
    H_C = gamma H0 + K^T Diag(gc) U,

and, given dO and dH_C, its reverse is (every line a dense product)

    dU  = Diag(gc) K dH_C + P^T dO              dW = -dU H0^T
    dH0 = gamma dH_C + Q^T Diag(ge) dO - W^T dU (the chain from chunk to chunk)
    dP  = tril(dO U^T)                          dT = dU Vb^T + dW Kb^T
    dA  = strict_tril(-T^T dT T^T)              (Vb = Diag(beta) V, Kb = Diag(beta ge) K)
    E   = Diag(beta) dA * Gamma,  F = dP * Gamma
    dQ  = Diag(ge) dO H0^T + F K
    dK  = E K + E^T K + F^T Q + Diag(gc) U dH_C^T + Diag(beta ge) T^T dW
    dV  = Diag(beta) T^T dU
    dbeta = rowsum(dA * (K K^T * Gamma)) + rowsum(V * T^T dU) + ge rowsum(K * T^T dW)
    dg  = the row sums of the decay terms (see _chunk_bwd), then the log-decay input's
          gradient is the reverse cumulative sum of dg within the chunk.

The checks run at chunk sizes that leave a ragged tail (padded rows are zero and
carry no decay), with a non-zero initial state and final-state gradient."""
import numpy as np
import pytest

import oracle


def _inputs(mode, B=2, T=37, H=2, dk=8, dv=6, seed=0):
    rng = np.random.default_rng(seed)
    f32 = np.float32
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    q = (q / np.linalg.norm(q, axis=-1, keepdims=True)).astype(f32)
    k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(f32)
    v = rng.standard_normal((B, T, H, dv)).astype(f32)
    beta = (1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))).astype(f32)
    gate = (-0.3 * rng.random((B, T, H))).astype(f32) if mode == oracle.MODE_GDN else None
    S0 = (0.3 * rng.standard_normal((B, H, dk, dv))).astype(f32)
    dout = rng.standard_normal((B, T, H, dv)).astype(f32)
    dsf = rng.standard_normal((B, H, dk, dv)).astype(f32)
    return q, k, v, beta, gate, S0, dout, dsf


def _chunk_fwd(Q, K, V, bet, g, H0):
    """Forward quantities of one chunk (fp64), zero-padded rows allowed."""
    L = K.shape[0]
    Gam = np.exp(g[:, None] - g[None, :])
    ge, gl = np.exp(g), g[-1]
    gc, gam = np.exp(gl - g), np.exp(gl)
    SA = (K @ K.T) * Gam
    A = np.tril(bet[:, None] * SA, -1)
    T = np.linalg.inv(np.eye(L) + A)
    Kb = (bet * ge)[:, None] * K
    Vb = bet[:, None] * V
    W, U1 = T @ Kb, T @ Vb
    U = U1 - W @ H0
    SP = (Q @ K.T) * Gam
    P = np.tril(SP)
    O = ge[:, None] * (Q @ H0) + P @ U
    HC = gam * H0 + K.T @ (gc[:, None] * U)
    return dict(Gam=Gam, ge=ge, gc=gc, gam=gam, SA=SA, A=A, T=T, Kb=Kb, Vb=Vb, W=W, U=U, SP=SP, P=P, O=O, HC=HC)


def _chunk_bwd(Q, K, V, bet, g, H0, dO, dHC, plant=None):
    """Reverse of _chunk_fwd: (dQ, dK, dV, dbeta, dg (per-row log prefix), dH0).
    `plant` names a mistake to make on purpose (for the test that the checks catch it)."""
    f = _chunk_fwd(Q, K, V, bet, g, H0)
    Gam, ge, gc, gam, T, W, U, P = f["Gam"], f["ge"], f["gc"], f["gam"], f["T"], f["W"], f["U"], f["P"]
    L = K.shape[0]
    KdH = K @ dHC                                    # L x dv
    dU = gc[:, None] * KdH + (0 if plant == "dU_without_P" else P.T @ dO)
    dW = -dU @ H0.T
    dH0 = (1.0 if plant == "dH_without_decay" else gam) * dHC + Q.T @ (ge[:, None] * dO) - W.T @ dU
    dP = np.tril(dO @ U.T) if plant != "dP_strict" else np.tril(dO @ U.T, -1)
    dT = dU @ f["Vb"].T + dW @ f["Kb"].T
    dA = np.tril((1 if plant == "dA_sign" else -1) * T.T @ dT @ T.T, -1)
    E = bet[:, None] * dA * Gam
    F = dP * (1.0 if plant == "F_without_decay" else Gam)
    TdU, TdW = T.T @ dU, T.T @ dW
    dQhat = dO @ H0.T                                # gradient of Q^ = Diag(ge) Q
    dQ = ge[:, None] * dQhat + F @ K
    dKt = U @ dHC.T                                  # gradient of K~ = Diag(gc) K
    dK = E @ K + E.T @ K + F.T @ Q + gc[:, None] * dKt + (bet * ge)[:, None] * TdW
    dV = bet[:, None] * TdU
    KK, QK = K @ K.T, Q @ K.T
    dbeta = (dA * KK * Gam).sum(1) + (V * TdU).sum(1) + ge * (K * TdW).sum(1)
    # decay: dGamma (from A and P), ge, gc and gamma
    dGam = bet[:, None] * dA * KK + dP * QK
    R = dGam * Gam
    dg = R.sum(1) - R.sum(0)
    dg += ge * ((Q * dQhat).sum(1) + bet * (K * TdW).sum(1))
    dgc = (K * dKt).sum(1) * gc
    dg -= dgc
    dg[L - 1] += dgc.sum() + gam * (H0 * dHC).sum()
    return dQ, dK, dV, dbeta, dg, dH0


def chunk_backward(mode, q, k, v, beta, gate, S0, dout, dsf, C, plant=None):
    """Whole-sequence backward by chunks: forward states H_c, the reverse chain of dH,
    then every chunk's gradients from (H_c, dH_{c+1})."""
    B, Tn, Hn, dk = q.shape
    dv = v.shape[-1]
    out = {n: np.zeros(s) for n, s in (("dq", (B, Tn, Hn, dk)), ("dk", (B, Tn, Hn, dk)), ("dv", (B, Tn, Hn, dv)),
                                       ("dbeta", (B, Tn, Hn)), ("dgate", (B, Tn, Hn)), ("dS0", (B, Hn, dk, dv)))}
    nch = (Tn + C - 1) // C
    for b in range(B):
        for h in range(Hn):
            def chunk(c):
                t0, t1 = c * C, min(Tn, (c + 1) * C)
                pad = lambda x: np.concatenate([x, np.zeros((C - (t1 - t0),) + x.shape[1:])]) if t1 - t0 < C else x
                f = lambda a: pad(a[b, t0:t1, h].astype(np.float64))
                a = f(gate) if gate is not None else np.zeros(C)
                return f(q), f(k), f(v), f(beta), np.cumsum(a), f(dout), t0, t1
            Hs = [S0[b, h].astype(np.float64)]
            for c in range(nch):
                Q, K, V, bet, g, _, _, _ = chunk(c)
                Hs.append(_chunk_fwd(Q, K, V, bet, g, Hs[-1])["HC"])
            dH = dsf[b, h].astype(np.float64)
            for c in reversed(range(nch)):
                Q, K, V, bet, g, dO, t0, t1 = chunk(c)
                dQ, dK, dV, dbt, dg, dH = _chunk_bwd(Q, K, V, bet, g, Hs[c], dO, dH, plant)
                n = t1 - t0
                out["dq"][b, t0:t1, h], out["dk"][b, t0:t1, h], out["dv"][b, t0:t1, h] = dQ[:n], dK[:n], dV[:n]
                out["dbeta"][b, t0:t1, h] = dbt[:n]
                out["dgate"][b, t0:t1, h] = (np.cumsum(dg) if plant == "dgate_forward_cumsum"
                                             else np.cumsum(dg[::-1])[::-1])[:n]
            out["dS0"][b, h] = dH
    if gate is None:
        out["dgate"] = None
    return out


@pytest.mark.parametrize("mode", [oracle.MODE_DELTANET, oracle.MODE_GDN])
@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_chunk_backward_equals_the_token_backward(mode, C):
    q, k, v, beta, gate, S0, dout, dsf = _inputs(mode)
    ref = oracle.bwd(q, k, v, beta, gate, S0, dout, dsf, mode=mode)
    got = chunk_backward(mode, q, k, v, beta, gate, S0, dout, dsf, C)
    for name in ("dq", "dk", "dv", "dbeta", "dgate", "dS0"):
        if ref[name] is None:
            continue
        err = np.abs(got[name] - ref[name]).max() / max(np.sqrt(np.mean(ref[name] ** 2)), 1e-30)
        assert err < 1e-10, f"{name}: {err:.3g} (mode {mode}, C {C})"


@pytest.mark.parametrize("plant", ["dU_without_P", "dH_without_decay", "dP_strict", "dA_sign", "F_without_decay",
                                   "dgate_forward_cumsum"])
def test_planted_mistakes_are_caught(plant):
    """Plausible slips in the derivation (a dropped P^T dO term, the chain without its
    decay, a strict mask on dP, the sign of dA, F without the decay ratios, the gate
    gradient summed forward instead of backward) make it disagree with the oracle."""
    mode = oracle.MODE_GDN
    q, k, v, beta, gate, S0, dout, dsf = _inputs(mode, T=20)
    ref = oracle.bwd(q, k, v, beta, gate, S0, dout, dsf, mode=mode)
    got = chunk_backward(mode, q, k, v, beta, gate, S0, dout, dsf, 4, plant)
    worst = max(np.abs(got[n] - ref[n]).max() / np.sqrt(np.mean(ref[n] ** 2))
                for n in ("dq", "dk", "dv", "dbeta", "dgate", "dS0"))
    assert worst > 1e-3, plant
