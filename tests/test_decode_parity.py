"""GPU parity of ldn_decode_step (consecutive steps, state in place) against
the fp64 oracle run over the same tokens."""
import numpy as np
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl
from tests._helpers import TOL, out_err, rel_err
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def run_steps(w, steps=None):
    import torch
    t = w.torch_inputs("cuda")
    S = t["S0"].clone()
    n = steps or w.T
    outs = []
    for i in range(n):
        g = None if t["gate"] is None else t["gate"][i]
        outs.append(ldn.decode_step(t["q"][i], t["k"][i], t["v"][i], t["beta"][i], g, S, mode=w.mode))
    assert ldn.device_status() == ldn.LDN_OK
    return torch.stack(outs).float().cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (64, 64), (128, 64)])
def test_decode_parity(mode, dtype, dk, dv):
    w = wl.make_decode("gdn_decode_b64_h16_dk128_dv128_steps1000", B=3, H=5, dk=dk, dv=dv, steps=24,
                       mode=mode, dtype=dtype)
    o, S = run_steps(w)
    ro, rs = oracle.decode(w.q, w.k, w.v, w.beta, w.gate, w.S0, mode=mode)
    assert out_err(o, ro, dtype) <= TOL[dtype]
    assert rel_err(S, rs) <= TOL[dtype]


@pytest.mark.parametrize("name", sorted(n for n, r in wl.DECODE_WORKLOADS.items() if r["mode"] != wl.MODE_GDN2))
def test_decode_full_1000_steps_sampled(name):
    """Full batch 64 x 16 heads, 1000 consecutive tokens; sampled heads vs the oracle."""
    w = wl.make_decode(name)
    o, S = run_steps(w)
    for b, h in [(0, 0), (17, 9), (63, 15)]:
        ro, rs = oracle.decode(w.q[:, b:b + 1, h:h + 1], w.k[:, b:b + 1, h:h + 1], w.v[:, b:b + 1, h:h + 1],
                               w.beta[:, b:b + 1, h:h + 1], w.gate[:, b:b + 1, h:h + 1],
                               w.S0[b:b + 1, h:h + 1], mode=w.mode)
        assert rel_err(o[:, b:b + 1, h:h + 1], ro) <= TOL["f32"]
        assert rel_err(S[b:b + 1, h:h + 1], rs) <= TOL["f32"]
    assert np.all(np.isfinite(o))
