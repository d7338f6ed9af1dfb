"""torch.autograd binding of the forward (ldn_chunk_fwd) and the backward
(ldn_backward): ``delta_rule(q, k, v, beta, gate, S0, mode=...)`` returns
(out, S_final) with gradients for q, k, v, beta, gate and S0.  Argument
marshalling only: both directions run in the CUDA kernels of libldn.so.

The gradients of q, k and v are returned in their dtype (the kernel computes
them in fp32); beta, gate and S0 are fp32 throughout.  The output's gradient
reaches backward() in the output's dtype (autograd casts every incoming
gradient to the dtype of the tensor it belongs to), which is the inputs' dtype:
ldn_backward takes it in that dtype, and the conversion below only makes the
layout contiguous.
"""
from __future__ import annotations

import torch

from . import _native


class _DeltaRule(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, beta, gate, S0, mode):
        mode = _native.MODES.get(mode, mode)
        out, sf = _native.chunk_fwd(q, k, v, beta, gate, S0, mode=mode)
        ctx.mode = mode
        ctx.save_for_backward(q, k, v, beta, gate, S0)
        return out, sf

    @staticmethod
    def backward(ctx, dout, dsf):
        q, k, v, beta, gate, S0 = ctx.saved_tensors
        g = _native.backward(q, k, v, beta, gate, S0, dout.to(q.dtype).contiguous(),
                             None if dsf is None else dsf.float().contiguous(), mode=ctx.mode)
        return (g["dq"].to(q.dtype), g["dk"].to(k.dtype), g["dv"].to(v.dtype), g["dbeta"], g["dgate"],
                None if S0 is None else g["dS0"], None)


def delta_rule(q, k, v, beta, gate=None, S0=None, *, mode):
    """Chunkwise forward with autograd support (see ldn_chunk_fwd / ldn_backward
    in include/ldn.h).  Shapes as ``chunk_fwd``; returns (out, S_final)."""
    return _DeltaRule.apply(q, k, v, beta, gate, S0, mode)
