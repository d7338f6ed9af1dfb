"""GPU parity of the pre-solved variant (LDN_VARIANT_PRESOLVED) against the fp64
oracle: every chunk's UT/WY solve X = [P T ; T] first, into the workspace (one
launch over all chunks), then the fused kernel reading X (the second launch).

Cases cover every mode, ragged tails, one-token and one-chunk sequences, an
initial state, chunks whose decay span needs the entry-wise paths, Gated
DeltaNet-2 through its own entry point, the no-allocation entry cut into
pieces, and state passing between calls."""
import numpy as np
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl
from tests._helpers import TOL, oracle_chunk, out_err, rel_err
import oracle

pytestmark = pytest.mark.gpu

PRE = ldn.LDN_VARIANT_PRESOLVED
BASE = {0: "deltanet_fp32_b1_t256_h1_d64", 1: "gdn_bf16_b4_t2048_h16_d128", 2: "kda_bf16_b8_t4096_h16_d128"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def run(w, S0=True, variant=PRE):
    import torch
    t = w.torch_inputs("cuda")
    out, sf = ldn.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["gate"], t["S0"] if S0 else None, mode=w.mode,
                            variant=variant)
    torch.cuda.synchronize()
    assert ldn.device_status() == ldn.LDN_OK
    return out.float().cpu().numpy(), sf.cpu().numpy()


def check(w, S0=True):
    o, s = run(w, S0)
    ro, rs = oracle_chunk(w) if S0 else oracle.fwd(w.q, w.k, w.v, w.beta, w.gate, None, mode=w.mode)
    eo, es = out_err(o, ro, "bf16"), rel_err(s, rs)
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], f"{w.name} mode {w.mode}: out {eo:.3g} state {es:.3g}"


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("B,T,H,dv,s0", [(2, 200, 3, 128, True), (1, 64, 2, 64, False), (1, 1, 1, 128, True),
                                         (1, 700, 1, 128, True), (2, 333, 2, 64, True), (3, 1000, 2, 128, False)])
def test_presolved_parity(mode, B, T, H, dv, s0):
    w = wl.make_chunk(BASE[mode], B=B, T=T, H=H, dk=128, dv=dv, mode=mode, dtype="bf16", s0=s0)
    check(w, S0=s0)


def test_presolved_gdn_strong_gates_entrywise_chunks():
    """Gated DeltaNet chunks whose log-decay span exceeds the factored decay ratios."""
    w = wl.make_chunk(BASE[1], B=1, T=320, H=2, s0=True)
    w.gate = (w.gate * 40.0).astype(np.float32)
    check(w)


def test_presolved_kda_strong_gates_entrywise_chunks():
    """KDA chunks with a channel whose decay span exceeds the fp16 factors: the solve and
    the fused kernel both take the entry-wise forms for them."""
    w = wl.make_chunk(BASE[2], B=1, T=320, H=2, s0=True)
    g = w.gate.copy()
    g[:, 64:192, :, 5] = -1.2
    g[:, 256:300, 1, 100] = -0.9
    w.gate = g.astype(np.float32)
    check(w)


def test_presolved_gdn2_through_its_entry_point():
    import torch
    w = wl.make_chunk("gdn2_bf16_b8_t4096_h16_d128", B=2, T=333, H=3, s0=True)
    t = w.torch_inputs("cuda")
    out, sf = ldn.chunk_fwd_gdn2(t["q"], t["k"], t["v"], t["erase"], t["write"], t["gate"], t["S0"], variant=PRE)
    torch.cuda.synchronize()
    assert ldn.device_status() == ldn.LDN_OK
    ro, rs = oracle.fwd_gdn2(w.q, w.k, w.v, w.erase, w.write, w.gate, w.S0)
    assert out_err(out.float().cpu().numpy(), ro, "bf16") <= TOL["bf16"]
    assert rel_err(sf.cpu().numpy(), rs) <= TOL["bf16"]


def test_presolved_no_alloc_entry_in_token_runs():
    """Through the library's array, one sequence whose X exceeds the array (T = 8400 at
    H = 128: 132 chunks x 128 heads x 16 KiB = 264 MiB > 256 MiB): chunk-aligned token runs
    with the state carried between them."""
    import torch
    w = wl.make_chunk(BASE[1], B=1, T=8400, H=128, s0=True)
    t = w.torch_inputs("cuda")
    out = torch.empty((w.B, w.T, w.H, w.dv), dtype=t["q"].dtype, device="cuda")
    sf = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    st = ldn.ldn_chunk_fwd_noalloc(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), t["beta"].data_ptr(),
                                   t["gate"].data_ptr(), t["S0"].data_ptr(), out.data_ptr(), sf.data_ptr(), w.B, w.T,
                                   w.H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16, PRE,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == ldn.LDN_OK
    torch.cuda.synchronize()
    assert ldn.device_status() == ldn.LDN_OK
    o, s = out.float().cpu().numpy(), sf.cpu().numpy()
    for h in (0, 77):   # sampled heads (the token runs cut every head at the same chunks)
        sl = lambda a: a[:, :, h:h + 1]
        ro, rs = oracle.fwd(sl(w.q), sl(w.k), sl(w.v), sl(w.beta), sl(w.gate), w.S0[:, h:h + 1], mode=w.mode)
        assert out_err(o[:, :, h:h + 1], ro, "bf16") <= TOL["bf16"]
        assert rel_err(s[:, h:h + 1], rs) <= TOL["bf16"]


def test_presolved_state_passing():
    """run(T1) -> S_final -> run(T2) equals run(T1 + T2) up to rounding (the state passes in fp32)."""
    w = wl.make_chunk(BASE[1], B=2, T=448, H=2, s0=True)
    o, s = run(w)
    a = wl.Workload(name=w.name, mode=w.mode, dtype=w.dtype, B=w.B, T=192, H=w.H, dk=w.dk, dv=w.dv,
                    q=w.q[:, :192], k=w.k[:, :192], v=w.v[:, :192], beta=w.beta[:, :192], gate=w.gate[:, :192],
                    S0=w.S0)
    oa, sa = run(a)
    b2 = wl.Workload(name=w.name, mode=w.mode, dtype=w.dtype, B=w.B, T=256, H=w.H, dk=w.dk, dv=w.dv,
                     q=w.q[:, 192:], k=w.k[:, 192:], v=w.v[:, 192:], beta=w.beta[:, 192:], gate=w.gate[:, 192:],
                     S0=sa)
    ob, sb = run(b2)
    assert np.array_equal(o[:, :192], oa)
    assert rel_err(np.concatenate([oa, ob], axis=1), o) < 1e-2 and rel_err(sb, s) < 1e-2


def test_auto_picks_presolved_for_many_sequences():
    """The cost model picks the pre-solved variant for the Gated DeltaNet bench shape (64
    sequences of 2048 tokens) and keeps the split variant for one long sequence."""
    big = 1 << 40
    assert ldn.ldn_chunk_fwd_select_ws(4, 2048, 16, 128, 128, 64, 1, 1, big) == PRE
    assert ldn.ldn_chunk_fwd_select_ws(1, 65536, 16, 128, 128, 64, 1, 1, big) == ldn.LDN_VARIANT_SPLIT
