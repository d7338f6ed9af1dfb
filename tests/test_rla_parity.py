"""GPU parity of ldn_rla_fwd / ldn_rla_fwd_ws (Residual Linear Attention and
Residual DeltaNet) against the fp64 RLA / RDN oracle, element by element, in
both forms: the chunk form (bf16, dk = dv = 128; Residual DeltaNet with a
workspace) and the recurrent form (every other case, and Residual DeltaNet
without a workspace).

Tolerances: fp32 inputs 1e-4; bf16 inputs 2e-2, with the bf16-stored output
measured beyond its half-ulp rounding as for the other modes (both forms carry
the states in fp32; the chunk form's products take fp16 operands)."""
import numpy as np
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl
from tests._helpers import TOL, fmt_parity, out_err, parity, rel_err
import oracle

pytestmark = pytest.mark.gpu

BASE = {False: "rla_bf16_b4_t2048_h16_d128", True: "rdn_bf16_b4_t2048_h16_d128"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def run(p, workspace=True):
    import torch
    el = torch.bfloat16 if p["dtype"] == "bf16" else torch.float32
    d = lambda a, dt=torch.float32: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dt)
    out, sf, rf = ldn.rla_fwd(d(p["q"], el), d(p["k"], el), d(p["v"], el), d(p["beta"]), d(p["gamma"]), d(p["gate"]),
                              d(p["S0"]), d(p["R0"]), clip=p["clip"], delta=p["delta"], workspace=workspace)
    assert ldn.device_status() == ldn.LDN_OK
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), sf.cpu().numpy(), rf.cpu().numpy()


def check(p, workspace=True):
    o, sf, rf = run(p, workspace)
    ro, rsf, rrf = oracle.fwd_rla(p["q"], p["k"], p["v"], p["beta"], p["gamma"], p["gate"], clip=p["clip"],
                                  S0=p["S0"], R0=p["R0"], delta=p["delta"])
    tol = TOL[p["dtype"]]
    eo, es, er = out_err(o, ro, p["dtype"]), rel_err(sf, rsf), rel_err(rf, rrf)
    assert eo <= tol and es <= tol and er <= tol, f"out {eo:.3g} S {es:.3g} R {er:.3g} (tol {tol})"


@pytest.mark.parametrize("delta", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_rla_rdn_dtypes_dims(delta, dtype, dk, dv):
    check(wl.make_rla(BASE[delta], B=2, T=150, H=2, dk=dk, dv=dv, dtype=dtype, s0=True))


@pytest.mark.parametrize("delta", [False, True])
@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130])
def test_rla_rdn_lengths(delta, T):
    check(wl.make_rla(BASE[delta], B=1, T=T, H=2, s0=(T % 2 == 1)))


@pytest.mark.parametrize("delta", [False, True])
@pytest.mark.parametrize("clip", [0.05, float("inf")])
def test_rla_rdn_clip_extremes(delta, clip):
    """A tight clip (most residuals saturate) and no clip at all."""
    for dtype in ("f32", "bf16"):
        check(wl.make_rla(BASE[delta], B=2, T=100, H=2, dtype=dtype, s0=True, clip=clip))


def test_rla_zero_length_copies_states():
    import torch
    p = wl.make_rla(BASE[True], B=2, T=3, H=2, s0=True)
    S0, R0 = torch.from_numpy(p["S0"]).cuda(), torch.from_numpy(p["R0"]).cuda()
    sf, rf = torch.full_like(S0, 7.0), torch.full_like(R0, 7.0)
    st = ldn.ldn_rla_fwd(0, 0, 0, 0, 0, 0, 1.0, S0.data_ptr(), R0.data_ptr(), 0, sf.data_ptr(), rf.data_ptr(),
                         2, 0, 2, 128, 128, 1, ldn.LDN_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == ldn.LDN_OK
    torch.cuda.synchronize()
    assert torch.equal(sf, S0) and torch.equal(rf, R0)


@pytest.mark.parametrize("delta", [False, True])
def test_rla_rdn_full_workload_whole_tensors(delta):
    """B=4, T=2048, H=16, d=128 bf16 in one call: every output element and both
    final states against the oracle."""
    p = wl.make_rla(BASE[delta])
    o, sf, rf = run(p)
    ro, rsf, rrf = oracle.fwd_rla(p["q"], p["k"], p["v"], p["beta"], p["gamma"], p["gate"], clip=p["clip"],
                                  delta=delta)
    po = parity(o, ro, "bf16")
    ps, pr = parity(sf, rsf, "f32", tol=TOL["bf16"]), parity(rf, rrf, "f32", tol=TOL["bf16"])
    print(f"\n{BASE[delta]}: output: {fmt_parity(po)}; states plain {ps['plain']:.3g} / {pr['plain']:.3g}")
    assert po["excess"] <= TOL["bf16"]
    assert ps["plain"] <= TOL["bf16"] and pr["plain"] <= TOL["bf16"]


@pytest.mark.parametrize("delta", [False, True])
def test_rla_rdn_both_forms(delta):
    """The same bf16 128 x 128 inputs through the chunk form and (Residual DeltaNet
    without a workspace) the recurrent form; fp32 inputs take the recurrent form."""
    p = wl.make_rla(BASE[delta], B=2, T=300, H=2, s0=True)
    check(p, workspace=True)
    if delta:
        check(p, workspace=False)
    check(wl.make_rla(BASE[delta], B=2, T=300, H=2, dtype="f32", s0=True))


@pytest.mark.parametrize("delta", [False, True])
def test_rla_rdn_strong_decay(delta):
    """Log-decays of -6 per token: the decay factors across a chunk underflow fp32
    (e^-378); every factor is formed from a difference of log prefixes, so none
    overflows, and the states of a chunk's start are forgotten by its end."""
    p = wl.make_rla(BASE[delta], B=1, T=200, H=2, s0=True)
    p["gate"] = np.full_like(p["gate"], -6.0)
    check(p)
