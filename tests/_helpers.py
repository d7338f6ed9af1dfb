"""Shared test helpers: the parity metric and oracle calls on workloads."""
import numpy as np

import oracle

# Tolerances on max|gpu - oracle| / RMS(oracle): fp32 inputs 1e-4, bf16 inputs
# with an fp32 state 2e-2 (the precision targets stated for this method).
TOL = {"f32": 1e-4, "bf16": 2e-2}


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(got - ref))) / max(rms, 1e-30)


def oracle_chunk(w, b_idx=None, h_idx=None):
    """fp64 oracle on a workload, optionally on a subset of batches / heads."""
    sel = lambda a, hdim=2: a if a is None else a
    q, k, v, beta, gate, S0 = w.q, w.k, w.v, w.beta, w.gate, w.S0
    if b_idx is not None:
        q, k, v, beta = q[b_idx], k[b_idx], v[b_idx], beta[b_idx]
        gate = None if gate is None else gate[b_idx]
        S0 = None if S0 is None else S0[b_idx]
    if h_idx is not None:
        q, k, v, beta = q[:, :, h_idx], k[:, :, h_idx], v[:, :, h_idx], beta[:, :, h_idx]
        gate = None if gate is None else gate[:, :, h_idx]
        S0 = None if S0 is None else S0[:, h_idx]
    return oracle.fwd(q, k, v, beta, gate, S0, mode=w.mode)
