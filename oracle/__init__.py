"""fp64 CPU oracle for the delta-rule linear-attention family.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg import this package; the product path (the CUDA library and
its Python binding) never does, and this package imports nothing from it.

The arithmetic lives in ``ldn_oracle.c`` (plain C, fp64, token by token); this
module only builds it with gcc, loads it with ctypes and marshals numpy arrays.
Every function's passage is cited in the C source.

Parity status: pinned.  The pins are in tests/test_oracle_pins.py: the worked
example of the linear-attention notes (Sec. 2.3), the exact write at beta = 1,
the Gated DeltaNet prediction-correction identity of the Residual Linear
Attention notes (Sec. 1.2), closed forms for orthonormal / axis keys, the
linear-attention limit, orthogonal invariance and per-value-channel
independence from the state-reduction notes (Sec. 2.5, Prop. 3.1), the rank
bound (Eq. 3), the contraction of (I - beta k k^T), state passing, and a brute
force by explicit matrix products at d = 4, T = 8.  Gated DeltaNet-2 (Sec. 2.6) is
pinned in tests/test_gdn2_oracle_pins.py: its reduction to KDA, the erase-off /
write-on additive limit, the exact write with unit keys, and a brute force through
the notes' matrix expansion.  The backward (``bwd``, the reverse-mode derivative
of the same recurrence) is pinned in tests/test_bwd_oracle_pins.py by central
finite differences of the forward oracle on every input and the initial state,
and by the exact linearity identities of the recurrence in (v, S0) and in q.
RLA / RDN (``fwd_rla``, Residual Linear Attention notes Sec. 2.2, 2.4) are pinned
in tests/test_rla_oracle_pins.py: RLA against its closed form (decayed sums of
the writes, written in numpy), RDN against the composition of the Gated DeltaNet
oracle for both states, the notes' one-step expansion of the output, and the
clip bound.  ``ldn_oracle_selftest.c`` (built by ``build`` into an executable
beside the library) repeats the worked example, the exact write, the brute
force, the mode reductions and state passing natively, without numpy; the CPU
suite runs it (tests/test_oracle_selftest_c.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ldn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libldn_oracle.so")
_lock = threading.Lock()
_lib = None

MODE_DELTANET, MODE_GDN, MODE_KDA, MODE_GDN2 = 0, 1, 2, 3


_SELFTEST_SRC = os.path.join(_HERE, "ldn_oracle_selftest.c")
SELFTEST_PATH = os.path.join(_HERE, "ldn_oracle_selftest")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-pthread", "-D_POSIX_C_SOURCE=200809L"]


def build(force: bool = False) -> str:
    """Compile ldn_oracle.c into libldn_oracle.so beside it (gcc, no fast-math,
    no FMA contraction, so the fp64 rounding is the same on every host), and the
    native self-test beside it (``build_selftest``)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    build_selftest(force)
    return _LIB_PATH


def build_selftest(force: bool = False, oracle_src: str | None = None, out: str | None = None) -> str:
    """Compile the native self-test (ldn_oracle_selftest.c, linked with the oracle
    source under the library's flags) into an executable; ``oracle_src`` and
    ``out`` let a test build it against a modified copy of the oracle."""
    src = oracle_src or _SRC
    out = out or SELFTEST_PATH
    stale = not os.path.exists(out) or any(os.path.getmtime(out) < os.path.getmtime(f) for f in (src, _SELFTEST_SRC))
    if force or oracle_src or stale:
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, _SELFTEST_SRC, src, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, out)
    return out


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # LDN_ORACLE_LIB points the tests' mutation check at a deliberately
            # broken copy of this oracle; nothing else sets it.
            path = os.environ.get("LDN_ORACLE_LIB") or build()
            lib = ctypes.CDLL(path)
            f = lib.ldn_oracle_fwd
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_int)]
            g2 = lib.ldn_oracle_fwd_gdn2
            g2.restype = ctypes.c_int
            g2.argtypes = [ctypes.c_void_p] * 9 + [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_int)]
            rl = lib.ldn_oracle_rla
            rl.restype = ctypes.c_int
            rl.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_float] + [ctypes.c_void_p] * 5 + [ctypes.c_int] * 7
            bw = lib.ldn_oracle_bwd
            bw.restype = ctypes.c_int
            bw.argtypes = [ctypes.c_void_p] * 14 + [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_int)]
            lib.ldn_oracle_default_threads.restype = ctypes.c_int
            lib.ldn_oracle_default_threads.argtypes = []
            _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().ldn_oracle_default_threads())


def _f32(x, name):
    if x is None:
        return None
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if not np.all(np.isfinite(a)):
        raise ValueError(f"oracle input {name} has non-finite values")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data


def fwd(q, k, v, beta, gate=None, S0=None, mode=MODE_DELTANET, nthreads=0,
        want_state=True, return_threads=False):
    """Token-by-token recurrence in fp64.

    q, k: [B, T, H, dk]; v: [B, T, H, dv]; beta: [B, T, H];
    gate (natural-log decay): [B, T, H] for Gated DeltaNet, [B, T, H, dk] for
    KDA, ignored for DeltaNet; S0: [B, H, dk, dv] (memory orientation, i.e. the
    transpose of the d_v x d_k math state) or None for zeros.
    Returns (o [B, T, H, dv] float64, S_final [B, H, dk, dv] float64 or None).
    """
    q, k, v, beta = _f32(q, "q"), _f32(k, "k"), _f32(v, "v"), _f32(beta, "beta")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, T, H) or beta.shape != (B, T, H):
        raise ValueError("oracle: inconsistent shapes")
    if mode == MODE_DELTANET:
        gate = None
    else:
        gate = _f32(gate, "gate")
        want = (B, T, H) if mode == MODE_GDN else (B, T, H, dk)
        if gate is None or gate.shape != want:
            raise ValueError(f"oracle: gate must have shape {want}")
    S0 = _f32(S0, "S0")
    if S0 is not None and S0.shape != (B, H, dk, dv):
        raise ValueError("oracle: S0 must be [B, H, dk, dv]")
    out = np.empty((B, T, H, dv), dtype=np.float64)
    sf = np.empty((B, H, dk, dv), dtype=np.float64) if want_state else None
    used = ctypes.c_int(0)
    rc = _load().ldn_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(gate), _ptr(S0),
                                _ptr(out), _ptr(sf), B, T, H, dk, dv, int(mode), int(nthreads),
                                ctypes.byref(used))
    if rc != 0:
        raise RuntimeError(f"ldn_oracle_fwd failed with {rc}")
    if return_threads:
        return out, sf, int(used.value)
    return out, sf


def bwd(q, k, v, beta, gate, S0, dout, dS_final=None, mode=MODE_DELTANET, nthreads=0):
    """Reverse-mode gradients of L = sum <dout, o> + <dS_final, S_T> through the
    token recurrence of ``fwd`` (fp64, state history kept; see ldn_oracle.c).

    Shapes as ``fwd``; dout [B, T, H, dv]; dS_final [B, H, dk, dv] or None.
    Returns a dict of float64 arrays: dq, dk [B,T,H,dk], dv [B,T,H,dv],
    dbeta [B,T,H], dgate (shape of gate; None for DeltaNet), dS0 [B,H,dk,dv]."""
    q, k, v, beta = _f32(q, "q"), _f32(k, "k"), _f32(v, "v"), _f32(beta, "beta")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, T, H) or beta.shape != (B, T, H):
        raise ValueError("oracle: inconsistent shapes")
    if mode == MODE_DELTANET:
        gate = None
    else:
        gate = _f32(gate, "gate")
        want = (B, T, H) if mode == MODE_GDN else (B, T, H, dk)
        if gate is None or gate.shape != want:
            raise ValueError(f"oracle: gate must have shape {want}")
    S0 = _f32(S0, "S0")
    dout, dS_final = _f32(dout, "dout"), _f32(dS_final, "dS_final")
    if dout.shape != v.shape:
        raise ValueError("oracle: dout must be shaped like v")
    if S0 is not None and S0.shape != (B, H, dk, dv) or dS_final is not None and dS_final.shape != (B, H, dk, dv):
        raise ValueError("oracle: states must be [B, H, dk, dv]")
    g = dict(dq=np.empty((B, T, H, dk)), dk=np.empty((B, T, H, dk)), dv=np.empty((B, T, H, dv)),
             dbeta=np.empty((B, T, H)), dgate=None if gate is None else np.empty(gate.shape),
             dS0=np.empty((B, H, dk, dv)))
    rc = _load().ldn_oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(gate), _ptr(S0), _ptr(dout),
                                _ptr(dS_final), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dbeta"]),
                                _ptr(g["dgate"]), _ptr(g["dS0"]), B, T, H, dk, dv, int(mode), int(nthreads), None)
    if rc != 0:
        raise RuntimeError(f"ldn_oracle_bwd failed with {rc}")
    return g


def fwd_rla(q, k, v, beta, gamma, gate, clip=1.0, S0=None, R0=None, delta=False, nthreads=0):
    """Residual Linear Attention (delta=False) or Residual DeltaNet (delta=True) in
    fp64 (Residual Linear Attention notes, Sec. 2.2 and 2.4; see ldn_oracle.c).

    q, k [B,T,H,dk]; v [B,T,H,dv]; beta, gamma, gate (log alpha) [B,T,H];
    clip c > 0 (np.inf: none); S0, R0 [B,H,dk,dv] or None.
    Returns (o [B,T,H,dv], S_final, R_final), all float64."""
    q, k, v = _f32(q, "q"), _f32(k, "k"), _f32(v, "v")
    beta, gamma, gate = _f32(beta, "beta"), _f32(gamma, "gamma"), _f32(gate, "gate")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, T, H) or any(a.shape != (B, T, H) for a in (beta, gamma, gate)):
        raise ValueError("oracle: inconsistent shapes")
    S0, R0 = _f32(S0, "S0"), _f32(R0, "R0")
    out = np.empty((B, T, H, dv))
    sf, rf = np.empty((B, H, dk, dv)), np.empty((B, H, dk, dv))
    c = float(clip)
    if not c > 0:
        raise ValueError("oracle: clip must be > 0")
    rc = _load().ldn_oracle_rla(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(gamma), _ptr(gate),
                                ctypes.c_float(np.float32(c) if np.isfinite(c) else np.float32(np.inf)),
                                _ptr(S0), _ptr(R0), _ptr(out), _ptr(sf), _ptr(rf), B, T, H, dk, dv,
                                int(bool(delta)), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"ldn_oracle_rla failed with {rc}")
    return out, sf, rf


def fwd_gdn2(q, k, v, erase, write, gate, S0=None, nthreads=0, want_state=True):
    """Gated DeltaNet-2 token recurrence in fp64 (linear-attention notes, Sec. 2.6,
    Eqs. 21-24): per-key-channel decay, erase direction e = erase * k, write
    target z = write * v, outer product with k.

    q, k, erase, gate (log-decay): [B, T, H, dk]; v, write: [B, T, H, dv];
    S0: [B, H, dk, dv] or None.  Returns (o, S_final or None) as in ``fwd``."""
    q, k, v = _f32(q, "q"), _f32(k, "k"), _f32(v, "v")
    erase, write, gate = _f32(erase, "erase"), _f32(write, "write"), _f32(gate, "gate")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or erase.shape != q.shape or gate.shape != q.shape or v.shape[:3] != (B, T, H) \
            or write.shape != v.shape:
        raise ValueError("oracle: inconsistent shapes")
    S0 = _f32(S0, "S0")
    if S0 is not None and S0.shape != (B, H, dk, dv):
        raise ValueError("oracle: S0 must be [B, H, dk, dv]")
    out = np.empty((B, T, H, dv), dtype=np.float64)
    sf = np.empty((B, H, dk, dv), dtype=np.float64) if want_state else None
    used = ctypes.c_int(0)
    rc = _load().ldn_oracle_fwd_gdn2(_ptr(q), _ptr(k), _ptr(v), _ptr(erase), _ptr(write), _ptr(gate), _ptr(S0),
                                     _ptr(out), _ptr(sf), B, T, H, dk, dv, int(nthreads), ctypes.byref(used))
    if rc != 0:
        raise RuntimeError(f"ldn_oracle_fwd_gdn2 failed with {rc}")
    return out, sf


def decode_gdn2(q, k, v, erase, write, gate, S0, nthreads=0):
    """Consecutive Gated DeltaNet-2 decode steps: inputs [steps, B, H, d]."""
    tr = lambda a: None if a is None else np.ascontiguousarray(np.swapaxes(np.asarray(a), 0, 1))
    o, sf = fwd_gdn2(tr(q), tr(k), tr(v), tr(erase), tr(write), tr(gate), S0, nthreads=nthreads)
    return np.ascontiguousarray(np.swapaxes(o, 0, 1)), sf


def decode(q, k, v, beta, gate, S0, mode=MODE_GDN, nthreads=0):
    """Consecutive single-token steps: inputs [steps, B, H, d], state [B, H, dk, dv].

    A decode step is the same recurrence applied to one token; ``steps``
    consecutive steps equal one pass over a sequence of that length, so this
    transposes the step axis next to the batch axis and calls ``fwd``.
    Returns (o [steps, B, H, dv], S_final [B, H, dk, dv])."""
    tr = lambda a: None if a is None else np.ascontiguousarray(np.swapaxes(np.asarray(a), 0, 1))
    o, sf = fwd(tr(q), tr(k), tr(v), tr(beta), tr(gate), S0, mode=mode, nthreads=nthreads)
    return np.ascontiguousarray(np.swapaxes(o, 0, 1)), sf
