"""Pins of the backward oracle (oracle.bwd) against what the mathematics fixes,
independent of its adjoint code:

  * central finite differences of the forward oracle, in fp64, for every element
    of every input and the initial state (the benchmark's method sources check
    their KDA backward the same way: an FP64 gradient check over all inputs and
    the initial state), for DeltaNet, Gated DeltaNet and KDA, with a loss that
    also weights the final state;
  * the recurrence is linear in (v, S0) jointly and, for a fixed state sequence,
    in q, so L = <dv, v> + <dS0, S0> and <dO, O> = <dq, q> hold exactly
    (Euler's identity for homogeneous maps of degree one).

Inputs sit on a dyadic grid (multiples of 2^-8) and the difference step is 2^-12,
so x +- h is exact in fp32 (the oracle's input type) and the only error of the
difference quotient is its O(h^2) truncation."""
import numpy as np
import pytest

import oracle

H_STEP = 2.0 ** -12


def _grid(a):
    return (np.round(np.asarray(a, np.float64) * 256.0) / 256.0).astype(np.float32)


def _inputs(mode, B=1, T=5, H=1, dk=3, dv=2, seed=0):
    rng = np.random.default_rng(seed)
    q = _grid(0.8 * rng.standard_normal((B, T, H, dk)))
    k = _grid(0.6 * rng.standard_normal((B, T, H, dk)))
    v = _grid(rng.standard_normal((B, T, H, dv)))
    beta = _grid(0.2 + 0.6 * rng.random((B, T, H)))
    gate = None
    if mode == oracle.MODE_GDN:
        gate = _grid(-0.4 * rng.random((B, T, H)))
    elif mode == oracle.MODE_KDA:
        gate = _grid(-0.4 * rng.random((B, T, H, dk)))
    S0 = _grid(0.5 * rng.standard_normal((B, H, dk, dv)))
    dout = _grid(rng.standard_normal((B, T, H, dv)))
    dsf = _grid(rng.standard_normal((B, H, dk, dv)))
    return dict(q=q, k=k, v=v, beta=beta, gate=gate, S0=S0), dout, dsf


def _loss(x, dout, dsf, mode):
    o, sf = oracle.fwd(x["q"], x["k"], x["v"], x["beta"], x["gate"], x["S0"], mode=mode)
    return float(np.sum(o * dout.astype(np.float64)) + np.sum(sf * dsf.astype(np.float64)))


@pytest.mark.parametrize("mode", [oracle.MODE_DELTANET, oracle.MODE_GDN, oracle.MODE_KDA])
def test_gradients_match_central_differences(mode):
    x, dout, dsf = _inputs(mode)
    g = oracle.bwd(x["q"], x["k"], x["v"], x["beta"], x["gate"], x["S0"], dout, dsf, mode=mode)
    names = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "gate": "dgate", "S0": "dS0"}
    for name, gname in names.items():
        if x[name] is None:
            assert g[gname] is None
            continue
        fd = np.zeros(x[name].shape)
        for idx in np.ndindex(x[name].shape):
            vals = []
            for sgn in (1.0, -1.0):
                y = {kk: (None if vv is None else vv.copy()) for kk, vv in x.items()}
                y[name][idx] = np.float32(float(x[name][idx]) + sgn * H_STEP)
                assert float(y[name][idx]) == float(x[name][idx]) + sgn * H_STEP   # exact in fp32
                vals.append(_loss(y, dout, dsf, mode))
            fd[idx] = (vals[0] - vals[1]) / (2.0 * H_STEP)
        np.testing.assert_allclose(g[gname], fd, rtol=1e-5, atol=1e-6, err_msg=f"{gname} (mode {mode})")


@pytest.mark.parametrize("mode", [oracle.MODE_DELTANET, oracle.MODE_GDN, oracle.MODE_KDA])
def test_linearity_identities(mode):
    x, dout, dsf = _inputs(mode, B=2, T=70, H=2, dk=8, dv=4, seed=3)
    o, sf = oracle.fwd(x["q"], x["k"], x["v"], x["beta"], x["gate"], x["S0"], mode=mode)
    g = oracle.bwd(x["q"], x["k"], x["v"], x["beta"], x["gate"], x["S0"], dout, dsf, mode=mode)
    L = np.sum(o * dout) + np.sum(sf * dsf)
    np.testing.assert_allclose(np.sum(g["dv"] * x["v"]) + np.sum(g["dS0"] * x["S0"]), L, rtol=1e-11)
    g0 = oracle.bwd(x["q"], x["k"], x["v"], x["beta"], x["gate"], x["S0"], dout, None, mode=mode)
    np.testing.assert_allclose(np.sum(g0["dq"] * x["q"]), np.sum(o * dout), rtol=1e-11)


def test_no_initial_state_and_empty_sequence():
    """S0 = None is the zero state (its gradient is still returned); T = 0 returns
    dS0 = dS_final."""
    x, dout, dsf = _inputs(oracle.MODE_GDN, T=4)
    g = oracle.bwd(x["q"], x["k"], x["v"], x["beta"], x["gate"], None, dout, dsf, mode=oracle.MODE_GDN)
    z = dict(x, S0=np.zeros_like(x["S0"]))
    gz = oracle.bwd(z["q"], z["k"], z["v"], z["beta"], z["gate"], z["S0"], dout, dsf, mode=oracle.MODE_GDN)
    for kk in g:
        np.testing.assert_array_equal(g[kk], gz[kk])
    e = lambda a: a[:, :0]
    g = oracle.bwd(e(x["q"]), e(x["k"]), e(x["v"]), e(x["beta"]), e(x["gate"]), x["S0"], e(dout), dsf,
                   mode=oracle.MODE_GDN)
    np.testing.assert_array_equal(g["dS0"], dsf.astype(np.float64))
