"""GPU parity of ldn_backward (gradients of sum <dout, o> + <dS_final, S_T>)
against the fp64 backward oracle, element by element.

Tolerances from the arithmetic.  Recurrent form (fp32 inputs, KDA, and dims
other than 128 x 128): the kernel runs the recurrence and its adjoint in fp32
(a relative rounding of ~6e-8 per operation, accumulated over the sequence and
over the sums of up to dv columns), so every gradient must agree to 1e-4 of its
RMS; the decay-gate gradient, a sum over a full state of products whose terms
cancel, to 1e-3.  Chunkwise form (bf16 DeltaNet / Gated DeltaNet, dk = dv =
128): its products take fp16 operands (2^-11 relative) with fp32 accumulation,
the precision class of the bf16 forward, so the bf16 target 2e-2 applies
(measured: below 1e-2)."""
import numpy as np
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl
from tests._helpers import rel_err
import oracle

pytestmark = pytest.mark.gpu

BASE = {0: "deltanet_fp32_b1_t256_h1_d64", 1: "gdn_bf16_b4_t2048_h16_d128", 2: "kda_bf16_b8_t4096_h16_d128"}
TOL = {"dq": 1e-4, "dk": 1e-4, "dv": 1e-4, "dbeta": 1e-4, "dgate": 1e-3, "dS0": 1e-4}
TOL_CHUNKWISE = 2e-2


def chunkwise(w) -> bool:
    """The shapes ldn_backward runs in chunk form."""
    return w.dtype == "bf16" and w.dk == 128 and w.dv == 128 and w.mode in (0, 1)


def tol(w, gname) -> float:
    return TOL_CHUNKWISE if chunkwise(w) else TOL[gname]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def run_bwd(w, dout, dsf, S0=True):
    import torch
    t = w.torch_inputs("cuda")
    el = t["q"].dtype
    d = torch.from_numpy(dout).to("cuda", el)
    f = None if dsf is None else torch.from_numpy(dsf).cuda()
    g = ldn.backward(t["q"], t["k"], t["v"], t["beta"], t["gate"], t["S0"] if S0 else None, d, f, mode=w.mode)
    torch.cuda.synchronize()
    return {kk: (None if vv is None else vv.cpu().numpy()) for kk, vv in g.items()}


def check(w, dout, dsf, S0=True, sel=None):
    got = run_bwd(w, dout, dsf, S0)
    ref = oracle.bwd(w.q, w.k, w.v, w.beta, w.gate, w.S0 if S0 else None, dout, dsf, mode=w.mode)
    for name, r in ref.items():
        if r is None:
            assert got[name] is None
            continue
        e = rel_err(got[name], r)
        assert e <= tol(w, name), f"{name}: {e:.3g} (mode {w.mode}, {w.dtype}, T={w.T})"


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_backward_modes_dtypes_dims(mode, dtype, dk, dv):
    w = wl.make_chunk(BASE[mode], B=2, T=37, H=2, dk=dk, dv=dv, mode=mode, dtype=dtype, s0=True)
    dout, dsf = wl.make_upstream(w)
    check(w, dout, dsf)


@pytest.mark.parametrize("T", [1, 7, 8, 9, 64, 100])
@pytest.mark.parametrize("mode", [1, 2])
def test_backward_lengths(T, mode):
    w = wl.make_chunk(BASE[mode], B=1, T=T, H=2, s0=True)
    dout, dsf = wl.make_upstream(w, final_state=(T % 2 == 0))
    check(w, dout, dsf)


def test_backward_without_initial_state():
    w = wl.make_chunk(BASE[1], B=2, T=50, H=2, s0=False)
    dout, _ = wl.make_upstream(w, final_state=False)
    check(w, dout, None, S0=False)


def test_backward_zero_length_copies_final_state_gradient():
    import torch
    w = wl.make_chunk(BASE[1], B=2, T=3, H=2, s0=True)
    _, dsf = wl.make_upstream(w)
    f = torch.from_numpy(dsf).cuda()
    dS0 = torch.full_like(f, 7.0)
    st = ldn.ldn_backward(0, 0, 0, 0, 0, 0, 0, f.data_ptr(), 0, 0, 0, 0, 0, dS0.data_ptr(), 2, 0, 2, 128, 128, 1,
                          ldn.LDN_BF16, 0, 0, torch.cuda.current_stream().cuda_stream)
    assert st == ldn.LDN_OK
    torch.cuda.synchronize()
    assert torch.equal(dS0, f)


@pytest.mark.parametrize("name,pairs", [("gdn_bf16_b4_t2048_h16_d128", [(0, 0), (3, 15)]),
                                        ("kda_bf16_b8_t4096_h16_d128", [(5, 7)])])
def test_backward_full_workload_sampled(name, pairs):
    """The forward workloads at full size in one call; sampled (b, h) pairs
    against the oracle (each (b, h) is independent)."""
    w = wl.make_chunk(name)
    dout, dsf = wl.make_upstream(w)
    got = run_bwd(w, dout, dsf)
    for b, h in pairs:
        sl = lambda a: None if a is None else a[b:b + 1, :, h:h + 1]
        ref = oracle.bwd(sl(w.q), sl(w.k), sl(w.v), sl(w.beta), sl(w.gate), None, sl(dout), dsf[b:b + 1, h:h + 1],
                         mode=w.mode, nthreads=1)
        for gname, r in ref.items():
            if r is None:
                continue
            gv = got[gname][b:b + 1, h:h + 1] if gname == "dS0" else got[gname][b:b + 1, :, h:h + 1]
            e = rel_err(gv, r)
            assert e <= tol(w, gname), f"{name} ({b},{h}) {gname}: {e:.3g}"
