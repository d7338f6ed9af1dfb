"""fp64 CPU oracle of the steps on either side of the chunkwise path: the input
prologue (short causal convolution with SiLU, L2 normalisation of q and k,
sigmoid write strength, Mamba2-style decay gate) and the gated RMSNorm output
epilogue.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg import this module; the product path never does, and this
module imports nothing from it.

Plain numpy in fp64, one definition per function, each citing the passage it
follows.  Inputs are read as stored (bf16 values already widened by the
caller, or fp32) and widened to fp64.

Where the pages leave a detail open, the plainest reading is taken:
  * the short convolution is depthwise and causal, of width W, with the
    weight layout of the causal_conv1d routine the pages name (a row of W taps
    per channel; tap W-1 multiplies the current token, tap W-1-i the token i
    steps back; tokens before the start of the sequence are zero);
  * L2 normalisation divides by sqrt(sum of squares + eps), eps inside the root;
  * the decay gate is log alpha = -a * softplus(z + b) with a > 0 given per head
    and b per head (Gated DeltaNet) or per head and key channel (KDA);
  * the output RMSNorm is per head over the value channels with one gain
    vector of length dv shared by the heads, eps inside the root, and the SiLU
    output gate multiplies the normalised value.

Parity status: pinned (tests/test_prologue_oracle_pins.py: impulse response,
causality and linearity of the convolution; closed-form values of SiLU,
sigmoid and softplus; unit norm and scale invariance of the L2 normalisation;
the RMSNorm of a constant row; reduction of the gate to the plain decay).
"""
from __future__ import annotations

import numpy as np

MODE_DELTANET, MODE_GDN, MODE_KDA = 0, 1, 2


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def sigmoid(x):
    """Logistic function (write strength beta = sigmoid(W_beta x): Residual Linear
    Attention notes, Sec. 3.2-3.4; the DeltaNet entry of the model-zoo page)."""
    x = _f64(x)
    return 0.5 * (1.0 + np.tanh(0.5 * x))


def silu(x):
    """x * sigmoid(x) (the SiLU after the short convolution: model-zoo page,
    DeltaNet entry; q/k path of the Residual Linear Attention notes, Fig. 1)."""
    x = _f64(x)
    return x * sigmoid(x)


def softplus(x):
    """log(1 + e^x), written to stay finite for large |x|."""
    x = _f64(x)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def short_conv(x, w):
    """Depthwise causal convolution along the sequence (model-zoo page: DeltaNet,
    "causal convolution plus SiLU"; KDA, "short convolution"; the backend notes
    name causal_conv1d with the SiLU activation).

    x [B, T, H, d]; w [H * d, W] (tap W - 1 on the current token).  Returns
    y[b, t, h, c] = sum_{i=0}^{W-1} w[h*d + c, W-1-i] * x[b, t-i, h, c], with x = 0
    before t = 0."""
    x = _f64(x)
    B, T, H, d = x.shape
    w = _f64(w).reshape(H, d, -1)
    W = w.shape[-1]
    y = np.zeros_like(x)
    for i in range(W):
        if i >= T:
            break
        y[:, i:] += x[:, :T - i] * w[None, None, :, :, W - 1 - i]
    return y


def l2_normalize(x, eps):
    """x / sqrt(sum_c x_c^2 + eps) over the last axis (model-zoo page: "Q/K are
    L2-normalised"; Residual Linear Attention notes, Fig. 1)."""
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def decay_gate(z, a, b):
    """log alpha = -a * softplus(z + b) (the Mamba2-style decay gate of the
    Residual Linear Attention notes, Sec. 3.2-3.4: alpha_t = exp[-a softplus(W_a x_t + b)]).

    Gated DeltaNet: z [B, T, H], a [H], b [H].  KDA: z [B, T, H, dk], a [H],
    b [H, dk] (a learnable per-channel decay bias: model-zoo page, KDA entry)."""
    z = _f64(z)
    a = _f64(a)
    b = _f64(b)
    if z.ndim == 3:
        return -a[None, None, :] * softplus(z + b[None, None, :])
    return -a[None, None, :, None] * softplus(z + b[None, None, :, :])


def prologue(q_in, k_in, v_in, conv_q, conv_k, conv_v, beta_logit, gate_z=None, gate_a=None, gate_b=None,
             mode=MODE_GDN, eps=1e-6):
    """The whole prologue in its order: q, k, v through the short convolution and
    SiLU; q and k L2-normalised per head; beta = sigmoid(logit); the decay gate
    (none for DeltaNet).  Returns (q, k, v, beta, gate)."""
    q = l2_normalize(silu(short_conv(q_in, conv_q)), eps)
    k = l2_normalize(silu(short_conv(k_in, conv_k)), eps)
    v = silu(short_conv(v_in, conv_v))
    beta = sigmoid(beta_logit)
    gate = None if mode == MODE_DELTANET else decay_gate(gate_z, gate_a, gate_b)
    return q, k, v, beta, gate


def rmsnorm_gated(o, g, weight, eps):
    """Output epilogue: per head, o * (mean_c o_c^2 + eps)^(-1/2) * weight * silu(g)
    (model-zoo page, Gated DeltaNet entry: "the output goes through RMSNorm, a
    gain and a SiLU gate"; the backend notes name rms_norm_gated).

    o, g [B, T, H, dv]; weight [dv]."""
    o = _f64(o)
    rs = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o * rs * _f64(weight) * silu(g)
