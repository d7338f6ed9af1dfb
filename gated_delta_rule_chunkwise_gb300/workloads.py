"""Seeded synthetic inputs for the delta-rule kernels and the oracle.

This module holds input generation only (none of the method's arithmetic):
both the CUDA path and the fp64 oracle consume the same arrays from here.

Recipe (every named workload):
  * numpy ``Generator(PCG64(seed))``, seed 0 unless given; draws in this order:
    q, k, v, beta-logits, gate noise, per-head gate bias b_h (KDA), S0;
  * q, k ~ N(0, 1) then L2-normalised over d_k per (b, t, h) in fp32 (the
    method sources normalise q and k per head); v ~ N(0, 1);
  * beta = sigmoid(N(0, 1)) per (b, t, h);
  * Gated DeltaNet log-decay g = -softplus(N(0, 1)) * 0.1 per (b, t, h);
    KDA log-decay g = -softplus(N(0, 1) + b_h) * 0.1 per (b, t, h, c) with one
    b_h ~ N(0, 0.5^2) per head (0.5 read as the standard deviation);
  * S0 ~ N(0, 0.02^2) where the workload has a nonzero initial state, else none;
  * Gated DeltaNet-2 draws everything KDA draws (its beta is then dropped), the
    same per-channel log-decay, and after S0 an erase gate b = sigmoid(N(0, 1))
    per (b, t, h, c) and a write gate w = sigmoid(N(0, 1)) per (b, t, h, i):
    gates in (0, 1) like beta, the plainest reading of the notes' channel-wise
    gates (they fix no range);
  * for bf16 workloads q, k, v are rounded to bf16 (round to nearest even)
    AFTER normalisation; beta, gates and states stay fp32.
Arrays are returned as float32 numpy arrays holding exactly the values the
kernels see (bf16 values are exact in fp32).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

MODE_DELTANET, MODE_GDN, MODE_KDA, MODE_GDN2 = 0, 1, 2, 3
MODE_NAMES = {MODE_DELTANET: "deltanet", MODE_GDN: "gdn", MODE_KDA: "kda", MODE_GDN2: "gdn2"}

# name -> recipe.  Sizes are the benchmark workloads; tests shrink them with overrides.
CHUNK_WORKLOADS = {
    "deltanet_fp32_b1_t256_h1_d64": dict(mode=MODE_DELTANET, dtype="f32", B=1, T=256, H=1, dk=64, dv=64, s0=False),
    "gdn_bf16_b4_t2048_h16_d128": dict(mode=MODE_GDN, dtype="bf16", B=4, T=2048, H=16, dk=128, dv=128, s0=False),
    "kda_bf16_b8_t4096_h16_d128": dict(mode=MODE_KDA, dtype="bf16", B=8, T=4096, H=16, dk=128, dv=128, s0=False),
    "gdn_bf16_long_b1_t8192_h16_d128": dict(mode=MODE_GDN, dtype="bf16", B=1, T=8192, H=16, dk=128, dv=128, s0=True),
    "gdn_bf16_long_b1_t32768_h16_d128": dict(mode=MODE_GDN, dtype="bf16", B=1, T=32768, H=16, dk=128, dv=128, s0=True),
    "gdn_bf16_long_b1_t65536_h16_d128": dict(mode=MODE_GDN, dtype="bf16", B=1, T=65536, H=16, dk=128, dv=128, s0=True),
    "gdn2_bf16_b8_t4096_h16_d128": dict(mode=MODE_GDN2, dtype="bf16", B=8, T=4096, H=16, dk=128, dv=128, s0=False),
}
DECODE_WORKLOADS = {
    "gdn_decode_b64_h16_dk128_dv128_steps1000": dict(mode=MODE_GDN, dtype="f32", B=64, H=16, dk=128, dv=128, steps=1000),
    "gdn_decode_b64_h16_dk64_dv128_steps1000": dict(mode=MODE_GDN, dtype="f32", B=64, H=16, dk=64, dv=128, steps=1000),
    "gdn2_decode_b64_h16_dk128_dv128_steps1000": dict(mode=MODE_GDN2, dtype="f32", B=64, H=16, dk=128, dv=128,
                                                      steps=1000),
}


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even), returned as fp32 values (finite inputs:
    their bit patterns are at most 0xFF7FFFFF, so adding at most 0x8000 stays
    inside 32 bits)."""
    u = np.array(x, dtype=np.float32, copy=True, order="C").view(np.uint32)
    lsb = u >> np.uint32(16)
    lsb &= np.uint32(1)
    lsb += np.uint32(0x7FFF)
    u += lsb
    u &= np.uint32(0xFFFF0000)
    return u.view(np.float32)


def _l2norm(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))
    return (x / n).astype(np.float32)


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(np.float32(0), x).astype(np.float32)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


@dataclasses.dataclass
class Workload:
    name: str
    mode: int
    dtype: str              # "f32" or "bf16": element type of q, k, v, out
    B: int
    T: int                  # tokens per sequence (decode: number of steps)
    H: int
    dk: int
    dv: int
    q: np.ndarray           # chunk: [B,T,H,dk]   decode: [steps,B,H,dk]
    k: np.ndarray
    v: np.ndarray
    beta: Optional[np.ndarray]   # None for Gated DeltaNet-2
    gate: Optional[np.ndarray]
    S0: Optional[np.ndarray]  # [B,H,dk,dv]
    chunk: int = 64
    decode: bool = False
    erase: Optional[np.ndarray] = None   # Gated DeltaNet-2: erase gate, shaped like k
    write: Optional[np.ndarray] = None   # Gated DeltaNet-2: write gate, shaped like v

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def torch_inputs(self, device="cuda"):
        """The inputs as torch tensors on `device` in the kernel dtypes."""
        import torch
        el = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        cv = lambda a, dt: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dt)
        return dict(q=cv(self.q, el), k=cv(self.k, el), v=cv(self.v, el), beta=cv(self.beta, torch.float32),
                    gate=cv(self.gate, torch.float32), S0=cv(self.S0, torch.float32),
                    erase=cv(self.erase, torch.float32), write=cv(self.write, torch.float32))


def _draw(rng, lead, mode, dtype, H, dk, dv, s0, B):
    """Draws in the documented order; `lead` is the leading shape ([B,T] or [steps,B])."""
    f32 = np.float32
    q = _l2norm(rng.standard_normal((*lead, H, dk), dtype=f32))
    k = _l2norm(rng.standard_normal((*lead, H, dk), dtype=f32))
    v = rng.standard_normal((*lead, H, dv), dtype=f32)
    beta = _sigmoid(rng.standard_normal((*lead, H), dtype=f32))
    gate = erase = write = None
    if mode == MODE_GDN:
        gate = (-_softplus(rng.standard_normal((*lead, H), dtype=f32)) * f32(0.1)).astype(f32)
    elif mode in (MODE_KDA, MODE_GDN2):
        noise = rng.standard_normal((*lead, H, dk), dtype=f32)
        b_h = (rng.standard_normal(H, dtype=f32) * f32(0.5)).astype(f32)
        gate = (-_softplus(noise + b_h[:, None]) * f32(0.1)).astype(f32)
    S0 = (rng.standard_normal((B, H, dk, dv), dtype=f32) * f32(0.02)).astype(f32) if s0 else None
    if mode == MODE_GDN2:
        erase = _sigmoid(rng.standard_normal((*lead, H, dk), dtype=f32))
        write = _sigmoid(rng.standard_normal((*lead, H, dv), dtype=f32))
        beta = None
    if dtype == "bf16":
        q, k, v = round_bf16(q), round_bf16(k), round_bf16(v)
    return q, k, v, beta, gate, S0, erase, write


def make_chunk(name: str = "gdn_bf16_b4_t2048_h16_d128", seed: int = 0, **over) -> Workload:
    """A chunkwise-forward workload; keyword overrides (B, T, H, dk, dv, mode,
    dtype, s0) shrink or vary it while keeping the recipe."""
    r = dict(CHUNK_WORKLOADS[name]); r.update(over)
    rng = np.random.default_rng(seed)
    q, k, v, beta, gate, S0, erase, write = _draw(rng, (r["B"], r["T"]), r["mode"], r["dtype"], r["H"], r["dk"],
                                                  r["dv"], r["s0"], r["B"])
    return Workload(name=name, mode=r["mode"], dtype=r["dtype"], B=r["B"], T=r["T"], H=r["H"],
                    dk=r["dk"], dv=r["dv"], q=q, k=k, v=v, beta=beta, gate=gate, S0=S0, erase=erase, write=write)


def make_decode(name: str = "gdn_decode_b64_h16_dk128_dv128_steps1000", seed: int = 0, **over) -> Workload:
    """A decode workload: `steps` consecutive tokens per sequence, drawn as
    [steps, B, H, .] in one go, from a random S0 ~ N(0, 0.02^2)."""
    r = dict(DECODE_WORKLOADS[name]); r.update(over)
    rng = np.random.default_rng(seed)
    q, k, v, beta, gate, S0, erase, write = _draw(rng, (r["steps"], r["B"]), r["mode"], r["dtype"], r["H"],
                                                  r["dk"], r["dv"], True, r["B"])
    return Workload(name=name, mode=r["mode"], dtype=r["dtype"], B=r["B"], T=r["steps"], H=r["H"],
                    dk=r["dk"], dv=r["dv"], q=q, k=k, v=v, beta=beta, gate=gate, S0=S0, decode=True,
                    erase=erase, write=write)


# ---- Residual Linear Attention / Residual DeltaNet inputs --------------------------
# Recipe: the Gated DeltaNet draws in the same order (q, k, v, beta logits, gate
# noise, S0), then gamma = sigmoid(N(0, 1)) per (b, t, h) and R0 ~ N(0, 0.02^2)
# when the workload has initial states.  The notes' main experiments clip at
# c = 1; alpha, beta, gamma follow their parameterisations (Mamba2-style decay,
# sigmoid strengths).  The pages give RLA no workload of its own: the Gated
# DeltaNet bench shape stands in.
RLA_WORKLOADS = {
    "rla_bf16_b4_t2048_h16_d128": dict(delta=False, dtype="bf16", B=4, T=2048, H=16, dk=128, dv=128, s0=False),
    "rdn_bf16_b4_t2048_h16_d128": dict(delta=True, dtype="bf16", B=4, T=2048, H=16, dk=128, dv=128, s0=False),
}


def make_rla(name: str = "rdn_bf16_b4_t2048_h16_d128", seed: int = 0, **over) -> dict:
    """Inputs of ldn_rla_fwd as float32 numpy arrays (bf16 values exact in fp32)."""
    r = dict(RLA_WORKLOADS[name]); r.update(over)
    rng = np.random.default_rng(seed)
    q, k, v, beta, gate, S0, _, _ = _draw(rng, (r["B"], r["T"]), MODE_GDN, r["dtype"], r["H"], r["dk"], r["dv"],
                                          r["s0"], r["B"])
    f32 = np.float32
    gamma = _sigmoid(rng.standard_normal((r["B"], r["T"], r["H"]), dtype=f32))
    R0 = (rng.standard_normal((r["B"], r["H"], r["dk"], r["dv"]), dtype=f32) * f32(0.02)).astype(f32) \
        if r["s0"] else None
    return dict(name=name, delta=r["delta"], dtype=r["dtype"], B=r["B"], T=r["T"], H=r["H"], dk=r["dk"], dv=r["dv"],
                q=q, k=k, v=v, beta=beta, gamma=gamma, gate=gate, S0=S0, R0=R0, clip=float(r.get("clip", 1.0)))


def make_upstream(w: Workload, seed: int = 1, final_state: bool = True):
    """Upstream gradients for the backward of a chunk workload: dout ~ N(0, 1)
    shaped like v (rounded to bf16 for bf16 workloads, as the kernels read it in
    the workload's dtype) and dS_final ~ N(0, 1) [B, H, dk, dv] fp32 (or None),
    drawn in that order from Generator(PCG64(seed))."""
    rng = np.random.default_rng(seed)
    f32 = np.float32
    dout = rng.standard_normal(w.v.shape, dtype=f32)
    if w.dtype == "bf16":
        dout = round_bf16(dout)
    dsf = rng.standard_normal((w.B, w.H, w.dk, w.dv), dtype=f32) if final_state else None
    return dout, dsf


# ---- prologue / epilogue inputs ------------------------------------------------
# Recipe: numpy Generator(PCG64(seed)), draws in this order: q_in, k_in, v_in
# ~ N(0, 1) (projection outputs); conv weights ~ N(0, 1/W) per (channel, tap)
# for q, k, v; beta logits ~ N(0, 1); gate noise z ~ N(0, 1) per (b, t, h)
# (Gated DeltaNet) or (b, t, h, c) (KDA); a_h = exp(N(0, 0.5^2)) > 0 per head;
# bias b ~ N(0, 0.5^2) per head (GDN) or per head and key channel (KDA); then the
# epilogue's output o ~ N(0, 1), output gate g ~ N(0, 1) and gain ~ 1 + N(0, 0.1^2)
# per value channel.  For bf16 the q/k/v inputs, o and g are rounded to bf16.

PROLOGUE_WORKLOADS = {
    "gdn_prologue_bf16_b4_t2048_h16_d128_w4": dict(mode=MODE_GDN, dtype="bf16", B=4, T=2048, H=16, dk=128, dv=128, width=4),
    "kda_prologue_bf16_b8_t4096_h16_d128_w4": dict(mode=MODE_KDA, dtype="bf16", B=8, T=4096, H=16, dk=128, dv=128, width=4),
}


def make_prologue(name: str = "gdn_prologue_bf16_b4_t2048_h16_d128_w4", seed: int = 0, **over) -> dict:
    """Inputs of ldn_prologue and ldn_rmsnorm_gated as float32 numpy arrays (bf16
    values exact in fp32), plus the sizes."""
    r = dict(PROLOGUE_WORKLOADS[name]); r.update(over)
    B, T, H, dk, dv, W, mode = r["B"], r["T"], r["H"], r["dk"], r["dv"], r["width"], r["mode"]
    rng = np.random.default_rng(seed)
    f32 = np.float32
    qi = rng.standard_normal((B, T, H, dk), dtype=f32)
    ki = rng.standard_normal((B, T, H, dk), dtype=f32)
    vi = rng.standard_normal((B, T, H, dv), dtype=f32)
    sc = f32(1.0 / np.sqrt(W))
    cq = (rng.standard_normal((H * dk, W), dtype=f32) * sc).astype(f32)
    ck = (rng.standard_normal((H * dk, W), dtype=f32) * sc).astype(f32)
    cv = (rng.standard_normal((H * dv, W), dtype=f32) * sc).astype(f32)
    bl = rng.standard_normal((B, T, H), dtype=f32)
    gz = ga = gb = None
    if mode == MODE_GDN:
        gz = rng.standard_normal((B, T, H), dtype=f32)
        ga = np.exp(rng.standard_normal(H, dtype=f32) * f32(0.5)).astype(f32)
        gb = (rng.standard_normal(H, dtype=f32) * f32(0.5)).astype(f32)
    elif mode == MODE_KDA:
        gz = rng.standard_normal((B, T, H, dk), dtype=f32)
        ga = np.exp(rng.standard_normal(H, dtype=f32) * f32(0.5)).astype(f32)
        gb = (rng.standard_normal((H, dk), dtype=f32) * f32(0.5)).astype(f32)
    o = rng.standard_normal((B, T, H, dv), dtype=f32)
    g = rng.standard_normal((B, T, H, dv), dtype=f32)
    gain = (1.0 + rng.standard_normal(dv, dtype=f32) * f32(0.1)).astype(f32)
    if r["dtype"] == "bf16":
        qi, ki, vi, o, g = round_bf16(qi), round_bf16(ki), round_bf16(vi), round_bf16(o), round_bf16(g)
    return dict(r, name=name, q_in=qi, k_in=ki, v_in=vi, conv_q=cq, conv_k=ck, conv_v=cv, beta_logit=bl,
                gate_z=gz, gate_a=ga, gate_b=gb, o=o, g=g, gain=gain)
