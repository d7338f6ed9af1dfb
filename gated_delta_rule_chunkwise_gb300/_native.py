"""Thin ctypes binding of libldn (include/ldn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of lib/libldn.so.  There is no CPU fallback: if the library has not
been built, or no GPU is present, the calls raise.

Two layers:
  * ``ldn_chunk_fwd``, ``ldn_chunk_fwd_variant``, ``ldn_chunk_fwd_ws``,
    ``ldn_chunk_fwd_workspace_size``, ``ldn_chunk_fwd_noalloc``, ``ldn_decode_step``,
    ``ldn_chunk_fwd_gdn2``, ``ldn_decode_step_gdn2``, ``ldn_backward``,
    ``ldn_backward_workspace_size``, ``ldn_rla_fwd``, ``ldn_rla_fwd_ws``,
    ``ldn_rla_fwd_workspace_size``, ``ldn_prologue``,
    ``ldn_rmsnorm_gated``,
    ``ldn_get_device_status``, ``ldn_status_string``, ``ldn_version``: the C
    entry points under the same names, taking raw integer pointers;
  * ``chunk_fwd``, ``decode_step``, ``chunk_fwd_gdn2``, ``decode_step_gdn2``, ``backward`` and
    ``rla_fwd``:
    the same calls on torch CUDA tensors,
    with shape / dtype checks and allocation of outputs and of the split
    variant's workspace (torch is used for device memory and the current
    stream only).
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libldn.so")

LDN_DELTANET, LDN_GDN, LDN_KDA, LDN_GDN2 = 0, 1, 2, 3
LDN_F32, LDN_BF16 = 0, 1
LDN_OK, LDN_ERR_INVALID_ARG, LDN_ERR_UNSUPPORTED, LDN_ERR_CUDA, LDN_ERR_TIMEOUT = 0, 1, 2, 3, 4
LDN_VARIANT_AUTO, LDN_VARIANT_SIMT, LDN_VARIANT_TENSOR, LDN_VARIANT_SPLIT, LDN_VARIANT_PAIR = 0, 1, 2, 3, 4
LDN_VARIANT_PRESOLVED = 5

MODES = {"deltanet": LDN_DELTANET, "gdn": LDN_GDN, "kda": LDN_KDA}

_lock = threading.Lock()
_lib = None


class LdnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: status {status} ({ldn_status_string(status)})" if what else
                         f"status {status} ({ldn_status_string(status)})")


_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGNATURES = {
    "ldn_chunk_fwd": ([_P] * 8 + [_I] * 8 + [_P], _I),
    "ldn_chunk_fwd_variant": ([_P] * 8 + [_I] * 9 + [_P], _I),
    "ldn_chunk_fwd_select": ([_I] * 5, _I),
    "ldn_chunk_fwd_ws": ([_P] * 8 + [_I] * 9 + [_P, ctypes.c_size_t, _P], _I),
    "ldn_chunk_fwd_workspace_size": ([_I] * 8, ctypes.c_size_t),
    "ldn_chunk_fwd_select_ws": ([_I] * 8 + [ctypes.c_size_t], _I),
    "ldn_chunk_fwd_split_segments": ([_I] * 8 + [ctypes.c_size_t], _I),
    "ldn_chunk_fwd_noalloc": ([_P] * 8 + [_I] * 9 + [_P], _I),
    "ldn_decode_step": ([_P] * 7 + [_I] * 6 + [_P], _I),
    "ldn_chunk_fwd_gdn2": ([_P] * 9 + [_I] * 8 + [_P], _I),
    "ldn_backward": ([_P] * 14 + [_I] * 7 + [_P, ctypes.c_size_t, _P], _I),
    "ldn_rla_fwd": ([_P] * 6 + [ctypes.c_float] + [_P] * 5 + [_I] * 7 + [_P], _I),
    "ldn_backward_workspace_size": ([_I] * 7, ctypes.c_size_t),
    "ldn_rla_fwd_ws": ([_P] * 6 + [ctypes.c_float] + [_P] * 5 + [_I] * 7 + [_P, ctypes.c_size_t, _P], _I),
    "ldn_rla_fwd_workspace_size": ([_I] * 7, ctypes.c_size_t),
    "ldn_decode_steps": ([_P] * 7 + [_I] * 7 + [_P], _I),
    "ldn_decode_step_gdn2": ([_P] * 8 + [_I] * 5 + [_P], _I),
    "ldn_prologue": ([_P] * 6 + [_I] + [_P] * 9 + [_I] * 7 + [ctypes.c_float, _P], _I),
    "ldn_rmsnorm_gated": ([_P] * 4 + [_I] * 5 + [ctypes.c_float, _P], _I),
    "ldn_get_device_status": ([_P], _I),
    "ldn_status_string": ([_I], ctypes.c_char_p),
    "ldn_version": ([], _I),
}
EXPORTS = tuple(_SIGNATURES)


def load(path: str | None = None):
    """Load libldn.so (raises if it is missing: build it first)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libldn.so not found at {p}; run __graft_entry__.build() "
                                   "(or gated_delta_rule_chunkwise_gb300.build.build()) first")
            lib = ctypes.CDLL(p)
            for name, (args, res) in _SIGNATURES.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


# --- C entry points under their own names ---------------------------------
def ldn_chunk_fwd(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode, dtype, stream):
    return load().ldn_chunk_fwd(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk,
                                mode, dtype, stream)


def ldn_chunk_fwd_variant(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode,
                          dtype, variant, stream):
    return load().ldn_chunk_fwd_variant(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv,
                                        chunk, mode, dtype, variant, stream)


def ldn_chunk_fwd_select(dk, dv, chunk, mode, dtype):
    return load().ldn_chunk_fwd_select(dk, dv, chunk, mode, dtype)


def ldn_chunk_fwd_ws(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode, dtype, variant,
                     workspace, workspace_bytes, stream):
    return load().ldn_chunk_fwd_ws(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode, dtype,
                                   variant, workspace, workspace_bytes, stream)


def ldn_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, mode, dtype):
    return load().ldn_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, mode, dtype)


def ldn_chunk_fwd_select_ws(B, T, H, dk, dv, chunk, mode, dtype, workspace_bytes):
    return load().ldn_chunk_fwd_select_ws(B, T, H, dk, dv, chunk, mode, dtype, workspace_bytes)


def ldn_chunk_fwd_split_segments(B, T, H, dk, dv, chunk, mode, dtype, workspace_bytes):
    return load().ldn_chunk_fwd_split_segments(B, T, H, dk, dv, chunk, mode, dtype, workspace_bytes)


def ldn_chunk_fwd_noalloc(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode, dtype,
                          variant, stream):
    return load().ldn_chunk_fwd_noalloc(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk,
                                        mode, dtype, variant, stream)


def ldn_decode_step(q, k, v, beta, gate, S, out, B, H, dk, dv, mode, dtype, stream):
    return load().ldn_decode_step(q, k, v, beta, gate, S, out, B, H, dk, dv, mode, dtype, stream)


def ldn_chunk_fwd_gdn2(q, k, v, erase, write, gate, S0, out, S_final, B, T, H, dk, dv, chunk, dtype, variant,
                       stream):
    return load().ldn_chunk_fwd_gdn2(q, k, v, erase, write, gate, S0, out, S_final, B, T, H, dk, dv, chunk,
                                     dtype, variant, stream)


def ldn_decode_step_gdn2(q, k, v, erase, write, gate, S, out, B, H, dk, dv, dtype, stream):
    return load().ldn_decode_step_gdn2(q, k, v, erase, write, gate, S, out, B, H, dk, dv, dtype, stream)


def ldn_backward(q, k, v, beta, gate, S0, dout, dS_final, dq, dk, dv, dbeta, dgate, dS0, B, T, H, dk_dim, dv_dim,
                 mode, dtype, workspace, workspace_bytes, stream):
    return load().ldn_backward(q, k, v, beta, gate, S0, dout, dS_final, dq, dk, dv, dbeta, dgate, dS0, B, T, H,
                               dk_dim, dv_dim, mode, dtype, workspace, workspace_bytes, stream)


def ldn_backward_workspace_size(B, T, H, dk, dv, mode, dtype):
    return load().ldn_backward_workspace_size(B, T, H, dk, dv, mode, dtype)


def ldn_rla_fwd(q, k, v, beta, gamma, gate, clip, S0, R0, out, S_final, R_final, B, T, H, dk, dv, delta, dtype,
                stream):
    return load().ldn_rla_fwd(q, k, v, beta, gamma, gate, clip, S0, R0, out, S_final, R_final, B, T, H, dk, dv,
                              delta, dtype, stream)


def ldn_decode_steps(q, k, v, beta, gate, S, out, n_steps, B, H, dk, dv, mode, dtype, stream):
    return load().ldn_decode_steps(q, k, v, beta, gate, S, out, n_steps, B, H, dk, dv, mode, dtype, stream)


def ldn_rla_fwd_ws(q, k, v, beta, gamma, gate, clip, S0, R0, out, S_final, R_final, B, T, H, dk, dv, delta, dtype,
                   workspace, workspace_bytes, stream):
    return load().ldn_rla_fwd_ws(q, k, v, beta, gamma, gate, clip, S0, R0, out, S_final, R_final, B, T, H, dk, dv,
                                 delta, dtype, workspace, workspace_bytes, stream)


def ldn_rla_fwd_workspace_size(B, T, H, dk, dv, delta, dtype):
    return load().ldn_rla_fwd_workspace_size(B, T, H, dk, dv, delta, dtype)


def ldn_prologue(q_in, k_in, v_in, conv_q, conv_k, conv_v, width, beta_logit, gate_z, gate_a, gate_b,
                 q, k, v, beta, gate, B, T, H, dk, dv, mode, dtype, eps, stream):
    return load().ldn_prologue(q_in, k_in, v_in, conv_q, conv_k, conv_v, width, beta_logit, gate_z, gate_a, gate_b,
                               q, k, v, beta, gate, B, T, H, dk, dv, mode, dtype, eps, stream)


def ldn_rmsnorm_gated(o, g, weight, y, B, T, H, dv, dtype, eps, stream):
    return load().ldn_rmsnorm_gated(o, g, weight, y, B, T, H, dv, dtype, eps, stream)


def ldn_get_device_status(stream):
    return load().ldn_get_device_status(stream)


def ldn_status_string(status: int) -> str:
    try:
        return load().ldn_status_string(int(status)).decode()
    except RuntimeError:
        return "libldn not loaded"


def ldn_version() -> int:
    return load().ldn_version()


# --- torch-tensor convenience layer ---------------------------------------
def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return LDN_F32
    if t.dtype == torch.bfloat16:
        return LDN_BF16
    raise TypeError(f"q/k/v must be float32 or bfloat16, got {t.dtype}")


def _check(t, name, shape=None, dtype=None):
    import torch
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")


def chunk_fwd(q, k, v, beta, gate=None, S0=None, *, mode, chunk=64, out=None, S_final=None,
              want_state=True, variant=LDN_VARIANT_AUTO, workspace=None, stream=None):
    """Chunkwise forward on torch CUDA tensors (see ldn_chunk_fwd in include/ldn.h).

    q, k [B,T,H,dk], v [B,T,H,dv] (float32 or bfloat16, same dtype);
    beta [B,T,H] float32; gate [B,T,H] (gdn) or [B,T,H,dk] (kda) float32;
    S0 [B,H,dk,dv] float32 or None.  Returns (out, S_final or None).
    `workspace`: a uint8 CUDA tensor for the split variant, or None; with
    variant=LDN_VARIANT_SPLIT and no workspace one of the required size
    (ldn_chunk_fwd_workspace_size) is allocated."""
    import torch
    mode = MODES.get(mode, mode)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    _check(q, "q"); _check(k, "k", q.shape, q.dtype); _check(v, "v", (B, T, H, dv), q.dtype)
    _check(beta, "beta", (B, T, H), torch.float32)
    if mode == LDN_DELTANET:
        gate = None
    else:
        _check(gate, "gate", (B, T, H) if mode == LDN_GDN else (B, T, H, dk), torch.float32)
    _check(S0, "S0", (B, H, dk, dv), torch.float32)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    _check(out, "out", (B, T, H, dv), q.dtype)
    if S_final is None and want_state:
        S_final = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    _check(S_final, "S_final", (B, H, dk, dv), torch.float32)
    if variant in (LDN_VARIANT_SPLIT, LDN_VARIANT_PRESOLVED) and workspace is None:
        need = ldn_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, mode, _dtype_code(q))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if workspace is not None:
        _check(workspace, "workspace", dtype=torch.uint8)
        st = ldn_chunk_fwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(gate), _ptr(S0), _ptr(out),
                              _ptr(S_final), B, T, H, dk, dv, chunk, mode, _dtype_code(q), variant,
                              _ptr(workspace), workspace.numel(), _stream_handle(stream))
    else:
        st = ldn_chunk_fwd_variant(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(gate), _ptr(S0),
                                   _ptr(out), _ptr(S_final), B, T, H, dk, dv, chunk, mode,
                                   _dtype_code(q), variant, _stream_handle(stream))
    if st != LDN_OK:
        raise LdnError(st, "ldn_chunk_fwd")
    return out, S_final


def decode_step(q, k, v, beta, gate, S, *, mode, out=None, stream=None):
    """One recurrent step on torch CUDA tensors; S [B,H,dk,dv] float32 is updated
    in place.  q, k [B,H,dk], v [B,H,dv]; beta [B,H]; gate [B,H] / [B,H,dk]."""
    import torch
    mode = MODES.get(mode, mode)
    B, H, dk = q.shape
    dv = v.shape[-1]
    _check(q, "q"); _check(k, "k", q.shape, q.dtype); _check(v, "v", (B, H, dv), q.dtype)
    _check(beta, "beta", (B, H), torch.float32)
    if mode == LDN_DELTANET:
        gate = None
    else:
        _check(gate, "gate", (B, H) if mode == LDN_GDN else (B, H, dk), torch.float32)
    _check(S, "S", (B, H, dk, dv), torch.float32)
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    _check(out, "out", (B, H, dv), q.dtype)
    st = ldn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(gate), _ptr(S), _ptr(out),
                         B, H, dk, dv, mode, _dtype_code(q), _stream_handle(stream))
    if st != LDN_OK:
        raise LdnError(st, "ldn_decode_step")
    return out


def decode_steps(q, k, v, beta, gate, S, *, mode, out=None, stream=None):
    """n consecutive recurrent steps in one launch (ldn_decode_steps) on torch CUDA
    tensors; S [B,H,dk,dv] float32 is updated in place.  q, k [n,B,H,dk], v [n,B,H,dv];
    beta [n,B,H]; gate [n,B,H] / [n,B,H,dk].  Returns out [n,B,H,dv]."""
    import torch
    mode = MODES.get(mode, mode)
    n, B, H, dk = q.shape
    dv = v.shape[-1]
    _check(q, "q"); _check(k, "k", q.shape, q.dtype); _check(v, "v", (n, B, H, dv), q.dtype)
    _check(beta, "beta", (n, B, H), torch.float32)
    if mode == LDN_DELTANET:
        gate = None
    else:
        _check(gate, "gate", (n, B, H) if mode == LDN_GDN else (n, B, H, dk), torch.float32)
    _check(S, "S", (B, H, dk, dv), torch.float32)
    if out is None:
        out = torch.empty((n, B, H, dv), dtype=q.dtype, device=q.device)
    _check(out, "out", (n, B, H, dv), q.dtype)
    st = ldn_decode_steps(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(gate), _ptr(S), _ptr(out), n,
                          B, H, dk, dv, mode, _dtype_code(q), _stream_handle(stream))
    if st != LDN_OK:
        raise LdnError(st, "ldn_decode_steps")
    return out


def chunk_fwd_gdn2(q, k, v, erase, write, gate, S0=None, *, chunk=64, out=None, S_final=None, want_state=True,
                   variant=LDN_VARIANT_AUTO, stream=None):
    """Gated DeltaNet-2 chunkwise forward on torch CUDA tensors (ldn_chunk_fwd_gdn2).

    q, k [B,T,H,dk], v [B,T,H,dv] (float32 or bfloat16); erase, gate [B,T,H,dk]
    and write [B,T,H,dv] float32; S0 [B,H,dk,dv] float32 or None.
    Returns (out, S_final or None)."""
    import torch
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    _check(q, "q"); _check(k, "k", q.shape, q.dtype); _check(v, "v", (B, T, H, dv), q.dtype)
    _check(erase, "erase", (B, T, H, dk), torch.float32); _check(write, "write", (B, T, H, dv), torch.float32)
    _check(gate, "gate", (B, T, H, dk), torch.float32)
    _check(S0, "S0", (B, H, dk, dv), torch.float32)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    _check(out, "out", (B, T, H, dv), q.dtype)
    if S_final is None and want_state:
        S_final = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    _check(S_final, "S_final", (B, H, dk, dv), torch.float32)
    st = ldn_chunk_fwd_gdn2(_ptr(q), _ptr(k), _ptr(v), _ptr(erase), _ptr(write), _ptr(gate), _ptr(S0), _ptr(out),
                            _ptr(S_final), B, T, H, dk, dv, chunk, _dtype_code(q), variant, _stream_handle(stream))
    if st != LDN_OK:
        raise LdnError(st, "ldn_chunk_fwd_gdn2")
    return out, S_final


def decode_step_gdn2(q, k, v, erase, write, gate, S, *, out=None, stream=None):
    """One Gated DeltaNet-2 step on torch CUDA tensors; S [B,H,dk,dv] float32 is
    updated in place.  q, k, erase, gate [B,H,dk]; v, write [B,H,dv]."""
    import torch
    B, H, dk = q.shape
    dv = v.shape[-1]
    _check(q, "q"); _check(k, "k", q.shape, q.dtype); _check(v, "v", (B, H, dv), q.dtype)
    _check(erase, "erase", (B, H, dk), torch.float32); _check(write, "write", (B, H, dv), torch.float32)
    _check(gate, "gate", (B, H, dk), torch.float32)
    _check(S, "S", (B, H, dk, dv), torch.float32)
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    _check(out, "out", (B, H, dv), q.dtype)
    st = ldn_decode_step_gdn2(_ptr(q), _ptr(k), _ptr(v), _ptr(erase), _ptr(write), _ptr(gate), _ptr(S), _ptr(out),
                              B, H, dk, dv, _dtype_code(q), _stream_handle(stream))
    if st != LDN_OK:
        raise LdnError(st, "ldn_decode_step_gdn2")
    return out


def backward(q, k, v, beta, gate, S0, dout, dS_final=None, *, mode, workspace=None, stream=None):
    """Gradients of sum <dout, o> + <dS_final, S_T> on torch CUDA tensors (ldn_backward).

    Shapes and dtypes as ``chunk_fwd``; dout like v.  Returns a dict of float32
    tensors dq, dk, dv, dbeta, dgate (None for DeltaNet), dS0.  `workspace`: a
    uint8 CUDA tensor of at least ldn_backward_workspace_size bytes, or None to
    allocate one."""
    import torch
    mode = MODES.get(mode, mode)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    _check(q, "q"); _check(k, "k", q.shape, q.dtype); _check(v, "v", (B, T, H, dv), q.dtype)
    _check(dout, "dout", (B, T, H, dv), q.dtype)
    _check(beta, "beta", (B, T, H), torch.float32)
    if mode == LDN_DELTANET:
        gate = None
    else:
        _check(gate, "gate", (B, T, H) if mode == LDN_GDN else (B, T, H, dk), torch.float32)
    _check(S0, "S0", (B, H, dk, dv), torch.float32)
    _check(dS_final, "dS_final", (B, H, dk, dv), torch.float32)
    f32 = dict(dtype=torch.float32, device=q.device)
    g = dict(dq=torch.empty((B, T, H, dk), **f32), dk=torch.empty((B, T, H, dk), **f32),
             dv=torch.empty((B, T, H, dv), **f32), dbeta=torch.empty((B, T, H), **f32),
             dgate=None if gate is None else torch.empty(tuple(gate.shape), **f32),
             dS0=torch.empty((B, H, dk, dv), **f32))
    need = ldn_backward_workspace_size(B, T, H, dk, dv, mode, _dtype_code(q))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", dtype=torch.uint8)
    st = ldn_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(gate), _ptr(S0), _ptr(dout), _ptr(dS_final),
                      _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dbeta"]), _ptr(g["dgate"]), _ptr(g["dS0"]),
                      B, T, H, dk, dv, mode, _dtype_code(q), _ptr(workspace), workspace.numel(),
                      _stream_handle(stream))
    if st != LDN_OK:
        raise LdnError(st, "ldn_backward")
    return g


def rla_fwd(q, k, v, beta, gamma, gate, S0=None, R0=None, *, clip=1.0, delta=False, workspace=True, stream=None):
    """RLA (delta=False) or RDN (delta=True) forward on torch CUDA tensors
    (ldn_rla_fwd_ws).  q, k [B,T,H,dk], v [B,T,H,dv] (float32 or bfloat16); beta,
    gamma, gate [B,T,H] float32; S0, R0 [B,H,dk,dv] float32 or None.  With
    workspace=True the workspace ldn_rla_fwd_workspace_size asks for is allocated
    (Residual DeltaNet then takes the chunk form); False passes none.
    Returns (out, S_final, R_final)."""
    import torch
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    _check(q, "q"); _check(k, "k", q.shape, q.dtype); _check(v, "v", (B, T, H, dv), q.dtype)
    for name, t in (("beta", beta), ("gamma", gamma), ("gate", gate)):
        _check(t, name, (B, T, H), torch.float32)
    _check(S0, "S0", (B, H, dk, dv), torch.float32); _check(R0, "R0", (B, H, dk, dv), torch.float32)
    out = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    sf = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    rf = torch.empty_like(sf)
    need = ldn_rla_fwd_workspace_size(B, T, H, dk, dv, int(bool(delta)), _dtype_code(q)) if workspace else 0
    ws = torch.empty(need, dtype=torch.uint8, device=q.device) if need else None
    st = ldn_rla_fwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(gamma), _ptr(gate), float(clip), _ptr(S0),
                        _ptr(R0), _ptr(out), _ptr(sf), _ptr(rf), B, T, H, dk, dv, int(bool(delta)), _dtype_code(q),
                        _ptr(ws), need, _stream_handle(stream))
    if st != LDN_OK:
        raise LdnError(st, "ldn_rla_fwd")
    return out, sf, rf


def device_status(stream=None) -> int:
    """Synchronise the stream and read/clear the device status word."""
    return ldn_get_device_status(_stream_handle(stream))
