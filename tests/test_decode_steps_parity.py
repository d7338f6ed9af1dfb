"""GPU parity of ldn_decode_steps (n consecutive steps in one launch) against
the fp64 oracle over the same tokens, and against the same steps taken one
ldn_decode_step call at a time: both run each step's arithmetic in the same
order, so they agree bit for bit."""
import numpy as np
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl
from tests._helpers import TOL, out_err, parity, rel_err
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def run_multi(w):
    t = w.torch_inputs("cuda")
    S = t["S0"].clone()
    o = ldn.decode_steps(t["q"], t["k"], t["v"], t["beta"], t["gate"], S, mode=w.mode)
    assert ldn.device_status() == ldn.LDN_OK
    return o.float().cpu().numpy(), S.cpu().numpy()


def run_single(w):
    import torch
    t = w.torch_inputs("cuda")
    S = t["S0"].clone()
    outs = [ldn.decode_step(t["q"][i], t["k"][i], t["v"][i], t["beta"][i], None if t["gate"] is None else t["gate"][i],
                            S, mode=w.mode) for i in range(w.T)]
    assert ldn.device_status() == ldn.LDN_OK
    return torch.stack(outs).float().cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (64, 64), (128, 64)])
def test_decode_steps_parity_and_bits(mode, dtype, dk, dv):
    w = wl.make_decode("gdn_decode_b64_h16_dk128_dv128_steps1000", B=3, H=5, dk=dk, dv=dv, steps=24,
                       mode=mode, dtype=dtype)
    o, S = run_multi(w)
    ro, rs = oracle.decode(w.q, w.k, w.v, w.beta, w.gate, w.S0, mode=mode)
    assert out_err(o, ro, dtype) <= TOL[dtype]
    assert rel_err(S, rs) <= TOL[dtype]
    o1, S1 = run_single(w)
    assert np.array_equal(o, o1) and np.array_equal(S, S1)


@pytest.mark.parametrize("name", ["gdn_decode_b64_h16_dk128_dv128_steps1000", "gdn_decode_b64_h16_dk64_dv128_steps1000"])
def test_decode_steps_full_1000_steps_whole_tensors(name):
    """Batch 64 x 16 heads, 1000 tokens in one launch: every output and the final
    state against the oracle."""
    w = wl.make_decode(name)
    o, S = run_multi(w)
    ro, rs = oracle.decode(w.q, w.k, w.v, w.beta, w.gate, w.S0, mode=w.mode)
    po, ps = parity(o, ro, "f32"), parity(S, rs, "f32")
    print(f"\n{name}: outputs plain {po['plain']:.3g} over {po['n']} elements; state plain {ps['plain']:.3g}")
    assert po["plain"] <= TOL["f32"] and ps["plain"] <= TOL["f32"]


def test_decode_steps_zero_steps_leaves_the_state():
    import torch
    w = wl.make_decode("gdn_decode_b64_h16_dk128_dv128_steps1000", B=2, H=3, steps=1)
    t = w.torch_inputs("cuda")
    S = t["S0"].clone()
    st = ldn.ldn_decode_steps(0, 0, 0, 0, 0, S.data_ptr(), 0, 0, w.B, w.H, w.dk, w.dv, w.mode, ldn.LDN_F32,
                              torch.cuda.current_stream().cuda_stream)
    assert st == ldn.LDN_OK
    torch.cuda.synchronize()
    assert torch.equal(S, t["S0"])
