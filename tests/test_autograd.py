"""GPU: gradients through the torch.autograd binding (forward by ldn_chunk_fwd,
backward by ldn_backward) against the fp64 backward oracle, for a loss that
weights both the output and the final state."""
import numpy as np
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl
from tests._helpers import BF16_HALF_ULP, rel_err
import oracle

pytestmark = pytest.mark.gpu

BASE = {0: "deltanet_fp32_b1_t256_h1_d64", 1: "gdn_bf16_b4_t2048_h16_d128", 2: "kda_bf16_b8_t4096_h16_d128"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_autograd_gradients_match_the_oracle(mode, dtype):
    import torch
    from gated_delta_rule_chunkwise_gb300.autograd import delta_rule
    w = wl.make_chunk(BASE[mode], B=2, T=90, H=2, dk=128, dv=64, mode=mode, dtype=dtype, s0=True)
    dout, dsf = wl.make_upstream(w)
    t = w.torch_inputs("cuda")
    leaves = {kk: (vv.clone().requires_grad_(True) if vv is not None else None) for kk, vv in t.items()
              if kk in ("q", "k", "v", "beta", "gate", "S0")}
    out, sf = delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["beta"], leaves["gate"], leaves["S0"], mode=mode)
    loss = (out.float() * torch.from_numpy(dout).cuda()).sum() + (sf * torch.from_numpy(dsf).cuda()).sum()
    loss.backward()
    ref = oracle.bwd(w.q, w.k, w.v, w.beta, w.gate, w.S0, dout, dsf, mode=mode)
    names = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "gate": "dgate", "S0": "dS0"}
    # q, k, v gradients come back in the input dtype: bf16 storage rounds them by up to
    # half a bf16 ulp, measured beyond that rounding as for the bf16 outputs
    for name, gname in names.items():
        if leaves[name] is None:
            assert ref[gname] is None
            continue
        stored = BF16_HALF_ULP if dtype == "bf16" and name in ("q", "k", "v") else 0.0
        e = rel_err(leaves[name].grad.float().cpu().numpy(), ref[gname], stored)
        assert e <= 1e-3, f"{gname}: {e:.3g}"
