"""GPU parity of ldn_decode_step (consecutive steps, state in place) against
the fp64 oracle run over the same tokens."""
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
def test_decode_full_1000_steps_whole_tensors(name):
    """Full batch 64 x 16 heads, 1000 consecutive tokens: every output of every
    step and every element of the final state against the oracle."""
    w = wl.make_decode(name)
    o, S = run_steps(w)
    ro, rs = oracle.decode(w.q, w.k, w.v, w.beta, w.gate, w.S0, mode=w.mode)
    po, ps = parity(o, ro, "f32"), parity(S, rs, "f32")
    print(f"\n{name}: outputs plain {po['plain']:.3g} over {po['n']} elements; state plain {ps['plain']:.3g}")
    assert np.all(np.isfinite(o))
    assert po["plain"] <= TOL["f32"] and ps["plain"] <= TOL["f32"]


def test_decode_steps_in_a_cuda_graph_match_eager():
    """ldn_decode_step is capture-safe: 24 steps captured in a CUDA graph and
    replayed give the same bits as the same steps run eagerly."""
    import torch
    w = wl.make_decode("gdn_decode_b64_h16_dk128_dv128_steps1000", B=3, H=5, steps=24, dtype="f32")
    t = w.torch_inputs("cuda")
    o_eager, S_eager = run_steps(w)
    S = t["S0"].clone()
    outs = [torch.empty((w.B, w.H, w.dv), dtype=torch.float32, device="cuda") for _ in range(w.T)]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # first call outside capture (library set-up)
        ldn.decode_step(t["q"][0], t["k"][0], t["v"][0], t["beta"][0], t["gate"][0], S.clone(), mode=w.mode)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        for i in range(w.T):
            ldn.decode_step(t["q"][i], t["k"][i], t["v"][i], t["beta"][i], t["gate"][i], S, mode=w.mode, out=outs[i])
    S.copy_(t["S0"])
    g.replay()
    torch.cuda.synchronize()
    assert ldn.device_status() == ldn.LDN_OK
    np.testing.assert_array_equal(torch.stack(outs).cpu().numpy(), o_eager)
    np.testing.assert_array_equal(S.cpu().numpy(), S_eager)
