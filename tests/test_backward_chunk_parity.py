"""GPU parity of the chunkwise backward (bf16 DeltaNet / Gated DeltaNet with
dk = dv = 128: the solve and the pre-solved forward with chunk states, the
reverse chain of the state gradient, the per-chunk gradients) against the fp64
backward oracle, on whole tensors.

Cases span several chunks and a ragged tail (T = 1, 63, 64, 65, 200, 321,
1000), with and without an initial state and a final-state gradient, several
sequences and heads; and a long sequence (T = 32768, the long-context
workload's length) on sampled heads.  Tolerance: the bf16 target 2e-2 of the
RMS for every gradient (products on fp16 operands with fp32 accumulation; the
measured errors are below 1e-2)."""
import numpy as np
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl
from tests._helpers import fmt_parity, parity
import oracle

pytestmark = pytest.mark.gpu

TOL = 2e-2
BASE = {0: "gdn_bf16_b4_t2048_h16_d128", 1: "gdn_bf16_b4_t2048_h16_d128"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def run_bwd(w, dout, dsf, S0):
    import torch
    t = w.torch_inputs("cuda")
    d = torch.from_numpy(dout).to("cuda", t["q"].dtype)
    f = None if dsf is None else torch.from_numpy(dsf).cuda()
    g = ldn.backward(t["q"], t["k"], t["v"], t["beta"], t["gate"], t["S0"] if S0 else None, d, f, mode=w.mode)
    torch.cuda.synchronize()
    assert ldn.device_status() == 0
    return {kk: (None if vv is None else vv.cpu().numpy()) for kk, vv in g.items()}


def compare(got, ref, what):
    for name, r in ref.items():
        if r is None:
            assert got[name] is None, name
            continue
        p = parity(got[name], r, "f32", tol=TOL)
        assert p["plain"] <= TOL, f"{what} {name}: {fmt_parity(p)}"


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 321, 1000])
def test_chunkwise_backward_lengths(mode, T):
    B, H = (2, 3) if T <= 321 else (1, 2)
    w = wl.make_chunk(BASE[mode], B=B, T=T, H=H, mode=mode, s0=True)
    dout, dsf = wl.make_upstream(w)
    got = run_bwd(w, dout, dsf, S0=True)
    ref = oracle.bwd(w.q, w.k, w.v, w.beta, w.gate, w.S0, dout, dsf, mode=mode)
    compare(got, ref, f"mode {mode} T {T}")


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("s0,final", [(False, False), (True, False), (False, True)])
def test_chunkwise_backward_optional_states(mode, s0, final):
    w = wl.make_chunk(BASE[mode], B=2, T=150, H=2, mode=mode, s0=s0)
    dout, dsf = wl.make_upstream(w, final_state=final)
    got = run_bwd(w, dout, dsf, S0=s0)
    ref = oracle.bwd(w.q, w.k, w.v, w.beta, w.gate, w.S0 if s0 else None, dout, dsf, mode=mode)
    compare(got, ref, f"mode {mode} S0 {s0} dS_final {final}")


def test_chunkwise_backward_long_sequence_sampled():
    """B = 1, T = 32768, H = 16 in one call; heads 0 and 15 against the oracle
    (each head is independent)."""
    w = wl.make_chunk("gdn_bf16_b4_t2048_h16_d128", B=1, T=32768, H=16, mode=1, s0=False)
    dout, dsf = wl.make_upstream(w)
    got = run_bwd(w, dout, dsf, S0=False)
    for h in (0, 15):
        sl = lambda a: None if a is None else a[:, :, h:h + 1]
        ref = oracle.bwd(sl(w.q), sl(w.k), sl(w.v), sl(w.beta), sl(w.gate), None, sl(dout), dsf[:, h:h + 1],
                         mode=1, nthreads=1)
        sub = {n: (None if g is None else (g[:, h:h + 1] if n == "dS0" else g[:, :, h:h + 1])) for n, g in got.items()}
        compare(sub, ref, f"T 32768 head {h}")


def test_chunkwise_backward_is_deterministic():
    """Two calls on the same inputs give the same bits (no atomics across CTAs)."""
    w = wl.make_chunk("gdn_bf16_b4_t2048_h16_d128", B=2, T=500, H=4, s0=True)
    dout, dsf = wl.make_upstream(w)
    a = run_bwd(w, dout, dsf, S0=True)
    b = run_bwd(w, dout, dsf, S0=True)
    for n in a:
        if a[n] is not None:
            assert np.array_equal(a[n], b[n]), n


@pytest.mark.parametrize("mode", [0, 1])
def test_chunkwise_backward_strong_decay_and_many_heads(mode):
    """Log-decays of -6 per token (a chunk's decay products underflow fp32: every
    factor is a difference of log prefixes, at most 1) and 32 heads in one call."""
    w = wl.make_chunk(BASE[mode], B=2, T=130, H=32, mode=mode, s0=True)
    if w.gate is not None:
        w.gate[...] = -6.0
    dout, dsf = wl.make_upstream(w)
    got = run_bwd(w, dout, dsf, S0=True)
    ref = oracle.bwd(w.q, w.k, w.v, w.beta, w.gate, w.S0, dout, dsf, mode=mode)
    for name, g in got.items():
        if g is not None:
            assert np.all(np.isfinite(g)), name
    compare(got, ref, f"mode {mode} strong decay")
