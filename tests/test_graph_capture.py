"""The entry points with several launches per call are capture-safe: each call is
captured into a CUDA graph and replayed, and the replay gives the eager call's
results bit for bit (every kernel of these paths is deterministic: no atomics).

Covered: the pre-solved forward (solve + fed chain, the second launched with
programmatic dependent launch), the chunkwise backward (five launches), Residual
DeltaNet in chunk form (two solves + the chunk kernel) and the multi-step decode.
The first call of each runs outside the capture (kernel attributes are set then)."""
import numpy as np
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def capture_and_compare(call, outputs, reset=None):
    """call(stream_handle) enqueues the work; outputs() returns the result tensors.
    The eager results are kept, the call is captured on a side stream and replayed,
    and the replay's results must equal them."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        if reset:
            reset()
        call(side.cuda_stream)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert ldn.device_status() == ldn.LDN_OK
    eager = [t.clone() for t in outputs()]
    for t in outputs():
        t.fill_(float("nan")) if t.is_floating_point() else t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
        call(side.cuda_stream)
    if reset:
        reset()
    g.replay()
    torch.cuda.synchronize()
    assert ldn.device_status() == ldn.LDN_OK
    for a, b in zip(eager, outputs()):
        assert torch.equal(a, b)


def test_presolved_forward_captures():
    import torch
    w = wl.make_chunk("gdn_bf16_b4_t2048_h16_d128", B=2, T=300, H=4, s0=True)
    t = w.torch_inputs("cuda")
    out = torch.empty_like(t["v"])
    sf = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    need = ldn.ldn_chunk_fwd_workspace_size(w.B, w.T, w.H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def call(sh):
        st = ldn.ldn_chunk_fwd_ws(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), t["beta"].data_ptr(),
                                  t["gate"].data_ptr(), t["S0"].data_ptr(), out.data_ptr(), sf.data_ptr(), w.B, w.T,
                                  w.H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16, ldn.LDN_VARIANT_PRESOLVED, ws.data_ptr(),
                                  need, sh)
        assert st == ldn.LDN_OK

    capture_and_compare(call, lambda: (out, sf))


def test_chunkwise_backward_captures():
    import torch
    w = wl.make_chunk("gdn_bf16_b4_t2048_h16_d128", B=2, T=200, H=3, s0=True)
    t = w.torch_inputs("cuda")
    dout, dsf = wl.make_upstream(w)
    d = torch.from_numpy(dout).to("cuda", torch.bfloat16)
    f = torch.from_numpy(dsf).cuda()
    f32 = dict(dtype=torch.float32, device="cuda")
    g = {n: torch.empty(s, **f32) for n, s in (("dq", (w.B, w.T, w.H, w.dk)), ("dk", (w.B, w.T, w.H, w.dk)),
                                               ("dv", (w.B, w.T, w.H, w.dv)), ("dbeta", (w.B, w.T, w.H)),
                                               ("dgate", (w.B, w.T, w.H)), ("dS0", (w.B, w.H, w.dk, w.dv)))}
    need = ldn.ldn_backward_workspace_size(w.B, w.T, w.H, w.dk, w.dv, w.mode, ldn.LDN_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def call(sh):
        st = ldn.ldn_backward(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), t["beta"].data_ptr(),
                              t["gate"].data_ptr(), t["S0"].data_ptr(), d.data_ptr(), f.data_ptr(),
                              g["dq"].data_ptr(), g["dk"].data_ptr(), g["dv"].data_ptr(), g["dbeta"].data_ptr(),
                              g["dgate"].data_ptr(), g["dS0"].data_ptr(), w.B, w.T, w.H, w.dk, w.dv, w.mode,
                              ldn.LDN_BF16, ws.data_ptr(), need, sh)
        assert st == ldn.LDN_OK

    capture_and_compare(call, lambda: tuple(g.values()))


def test_rdn_chunk_form_captures():
    import torch
    p = wl.make_rla("rdn_bf16_b4_t2048_h16_d128", B=2, T=200, H=2, s0=True)
    dv = lambda a, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dt)
    q, k, v = dv(p["q"], torch.bfloat16), dv(p["k"], torch.bfloat16), dv(p["v"], torch.bfloat16)
    beta, gamma, gate, S0, R0 = dv(p["beta"]), dv(p["gamma"]), dv(p["gate"]), dv(p["S0"]), dv(p["R0"])
    out = torch.empty_like(v)
    sf = torch.empty((p["B"], p["H"], p["dk"], p["dv"]), dtype=torch.float32, device="cuda")
    rf = torch.empty_like(sf)
    need = ldn.ldn_rla_fwd_workspace_size(p["B"], p["T"], p["H"], p["dk"], p["dv"], 1, ldn.LDN_BF16)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def call(sh):
        st = ldn.ldn_rla_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), beta.data_ptr(), gamma.data_ptr(),
                                gate.data_ptr(), p["clip"], S0.data_ptr(), R0.data_ptr(), out.data_ptr(),
                                sf.data_ptr(), rf.data_ptr(), p["B"], p["T"], p["H"], p["dk"], p["dv"], 1,
                                ldn.LDN_BF16, ws.data_ptr(), need, sh)
        assert st == ldn.LDN_OK

    capture_and_compare(call, lambda: (out, sf, rf))


def test_multi_step_decode_captures():
    import torch
    w = wl.make_decode("gdn_decode_b64_h16_dk128_dv128_steps1000", B=3, H=5, steps=16, dtype="f32")
    t = w.torch_inputs("cuda")
    S = t["S0"].clone()
    o = torch.empty((w.T, w.B, w.H, w.dv), dtype=torch.float32, device="cuda")

    def call(sh):
        st = ldn.ldn_decode_steps(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), t["beta"].data_ptr(),
                                  t["gate"].data_ptr(), S.data_ptr(), o.data_ptr(), w.T, w.B, w.H, w.dk, w.dv,
                                  w.mode, ldn.LDN_F32, sh)
        assert st == ldn.LDN_OK

    capture_and_compare(call, lambda: (o, S), reset=lambda: S.copy_(t["S0"]))
