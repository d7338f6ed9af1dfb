"""GPU tests of ldn_chunk_fwd_noalloc: the split variant run through the
library's static device scratch, cut into pieces that fit it (groups of
sequences, or chunk-aligned token runs of one sequence with the state carried
between runs).  The file name sorts it last, so the scratch's one-time load
comes after every other test."""
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl
from tests._helpers import TOL, oracle_chunk, out_err, rel_err

pytestmark = pytest.mark.gpu

SCRATCH = 256 << 20          # bytes of the library's static scratch per device
UNIT = lambda dv: 32768 + (dv // 64) * 16384 + 16384 + 512   # workspace bytes per (b, h, chunk)
GDN_BASE = "gdn_bf16_b4_t2048_h16_d128"
BASE = {0: "deltanet_fp32_b1_t256_h1_d64", 1: GDN_BASE, 2: "kda_bf16_b8_t4096_h16_d128"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def _outputs(t, w, want_state):
    import torch
    out = torch.empty((w.B, w.T, w.H, w.dv), dtype=t["q"].dtype, device="cuda")
    sf = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda") if want_state else None
    return out, sf


def _p(x):
    return None if x is None else x.data_ptr()


def run_noalloc(w, variant=ldn.LDN_VARIANT_SPLIT, S0=True, want_state=True, stream=None, t=None, sync=True):
    import torch
    t = t or w.torch_inputs("cuda")
    out, sf = _outputs(t, w, want_state)
    s = stream or torch.cuda.current_stream()
    dt = ldn.LDN_BF16 if w.dtype == "bf16" else ldn.LDN_F32
    st = ldn.ldn_chunk_fwd_noalloc(_p(t["q"]), _p(t["k"]), _p(t["v"]), _p(t["beta"]), _p(t["gate"]),
                                   _p(t["S0"]) if S0 else None, _p(out), _p(sf), w.B, w.T, w.H, w.dk, w.dv,
                                   64, w.mode, dt, variant, s.cuda_stream)
    assert st == ldn.LDN_OK, ldn.ldn_status_string(st)
    if sync:
        torch.cuda.synchronize()
        assert ldn.device_status() == ldn.LDN_OK
    return out, sf


def run_ref(w, variant, S0=True, want_state=True):
    """The same call through the workspace entry (torch-allocated workspace)."""
    import torch
    t = w.torch_inputs("cuda")
    out, sf = ldn.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["gate"], t["S0"] if S0 else None,
                            mode=w.mode, variant=variant, want_state=want_state)
    torch.cuda.synchronize()
    assert ldn.device_status() == ldn.LDN_OK
    return out, sf


def _np(x):
    return None if x is None else x.float().cpu().numpy()


def _same(a, b):
    """Bit-identical results (same kernels, same per-chunk arithmetic)."""
    import torch
    assert (a is None) == (b is None)
    if a is not None:
        assert torch.equal(a, b), f"max |diff| {float((a.float() - b.float()).abs().max())}"


# ---- one piece: identical to the split variant with a caller workspace ----
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("B,T,H,dv,s0", [(2, 500, 4, 128, True), (1, 64, 3, 64, False), (3, 1, 2, 128, True)])
def test_single_piece_equals_workspace_split(mode, B, T, H, dv, s0):
    w = wl.make_chunk(BASE[mode], dtype="bf16", B=B, T=T, H=H, dk=128, dv=dv, s0=s0)
    o, s = run_noalloc(w)
    ro, rs = run_ref(w, ldn.LDN_VARIANT_SPLIT)
    _same(o, ro)
    _same(s, rs)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_parity_against_oracle(mode):
    w = wl.make_chunk(BASE[mode], dtype="bf16", B=2, T=333, H=3, dk=128, dv=128, s0=True)
    o, s = run_noalloc(w)
    ro, rs = oracle_chunk(w)
    eo, es = out_err(_np(o), ro, "bf16"), rel_err(_np(s), rs)
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], (eo, es)


# ---- several pieces ----
def test_sequence_groups_kda_full_workload():
    """KDA B=8, T=4096, H=16: 675 MB of workspace, run as groups of 3 sequences."""
    w = wl.make_chunk("kda_bf16_b8_t4096_h16_d128")
    assert w.B * w.H * (w.T // 64) * UNIT(w.dv) > SCRATCH
    o, s = run_noalloc(w)
    ro, rs = run_ref(w, ldn.LDN_VARIANT_SPLIT)
    _same(o, ro)
    _same(s, rs)
    b, h = 7, 12   # a sequence of the last group against the oracle
    sub = wl.Workload(name=w.name, mode=w.mode, dtype=w.dtype, B=1, T=w.T, H=1, dk=w.dk, dv=w.dv,
                      q=w.q[b:b + 1, :, h:h + 1], k=w.k[b:b + 1, :, h:h + 1], v=w.v[b:b + 1, :, h:h + 1],
                      beta=w.beta[b:b + 1, :, h:h + 1], gate=w.gate[b:b + 1, :, h:h + 1],
                      S0=None if w.S0 is None else w.S0[b:b + 1, h:h + 1])
    ro1, rs1 = oracle_chunk(sub)
    assert out_err(_np(o)[b:b + 1, :, h:h + 1], ro1, "bf16") <= TOL["bf16"]
    assert rel_err(_np(s)[b:b + 1, h:h + 1], rs1) <= TOL["bf16"]


@pytest.mark.parametrize("want_state", [True, False])
def test_token_runs_of_long_sequences(want_state):
    """Two sequences of 16421 tokens x 16 heads: one sequence alone needs 339 MB of
    workspace, so each runs as 203-chunk token runs with the state carried through
    S_final (or the scratch's state slot when no S_final is asked for)."""
    w = wl.make_chunk("gdn_bf16_long_b1_t8192_h16_d128", B=2, T=16384 + 37)
    assert w.H * ((w.T + 63) // 64) * UNIT(w.dv) > SCRATCH
    o, s = run_noalloc(w, want_state=want_state)
    ro, rs = run_ref(w, ldn.LDN_VARIANT_SPLIT, want_state=want_state)
    _same(o, ro)
    _same(s, rs)


# ---- variant choice and the paths that take no scratch ----
def test_auto_follows_the_cost_model():
    w = wl.make_chunk(GDN_BASE)
    chosen = ldn.ldn_chunk_fwd_select_ws(w.B, w.T, w.H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16, 1 << 62)
    assert chosen in (ldn.LDN_VARIANT_TENSOR, ldn.LDN_VARIANT_PAIR, ldn.LDN_VARIANT_SPLIT,
                      ldn.LDN_VARIANT_PRESOLVED)
    o, s = run_noalloc(w, ldn.LDN_VARIANT_AUTO)
    ro, rs = run_ref(w, chosen)
    _same(o, ro)
    _same(s, rs)


@pytest.mark.parametrize("variant", [ldn.LDN_VARIANT_TENSOR, ldn.LDN_VARIANT_SIMT])
def test_explicit_non_split_variants(variant):
    w = wl.make_chunk(GDN_BASE, B=1, T=300, H=2)
    o, s = run_noalloc(w, variant)
    ro, rs = run_ref(w, variant)
    _same(o, ro)
    _same(s, rs)


def test_fp32_auto_runs_simt():
    w = wl.make_chunk(BASE[0], B=2, T=130, H=2)
    o, s = run_noalloc(w, ldn.LDN_VARIANT_AUTO)
    ro, rs = run_ref(w, ldn.LDN_VARIANT_AUTO)
    _same(o, ro)
    _same(s, rs)


def test_fp32_split_is_unsupported():
    import torch
    w = wl.make_chunk(BASE[0], B=1, T=64, H=1)
    t = w.torch_inputs("cuda")
    out, sf = _outputs(t, w, True)
    st = ldn.ldn_chunk_fwd_noalloc(_p(t["q"]), _p(t["k"]), _p(t["v"]), _p(t["beta"]), None, None, _p(out),
                                   _p(sf), 1, 64, 1, w.dk, w.dv, 64, w.mode, ldn.LDN_F32,
                                   ldn.LDN_VARIANT_SPLIT, torch.cuda.current_stream().cuda_stream)
    assert st == ldn.LDN_ERR_UNSUPPORTED


def test_zero_length_copies_state():
    import torch
    S0 = torch.randn(2, 3, 128, 128, device="cuda")
    sf = torch.empty_like(S0)
    st = ldn.ldn_chunk_fwd_noalloc(None, None, None, None, None, S0.data_ptr(), None, sf.data_ptr(),
                                   2, 0, 3, 128, 128, 64, ldn.LDN_GDN, ldn.LDN_BF16, ldn.LDN_VARIANT_SPLIT,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == ldn.LDN_OK
    torch.cuda.synchronize()
    assert torch.equal(sf, S0)


# ---- sharing the scratch ----
def test_calls_on_two_streams_do_not_collide():
    """Two different problems enqueued on two streams back to back: the library
    orders their use of the shared scratch, so each equals its own lone run."""
    import torch
    w1 = wl.make_chunk(GDN_BASE, seed=1)
    w2 = wl.make_chunk(GDN_BASE, seed=2)
    lone1, lone2 = run_noalloc(w1), run_noalloc(w2)
    t1, t2 = w1.torch_inputs("cuda"), w2.torch_inputs("cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    res = []
    for _ in range(3):
        res.append(run_noalloc(w1, stream=s1, t=t1, sync=False))
        res.append(run_noalloc(w2, stream=s2, t=t2, sync=False))
    torch.cuda.synchronize()
    assert ldn.device_status() == ldn.LDN_OK
    for i, (o, s) in enumerate(res):
        lo, ls = lone1 if i % 2 == 0 else lone2
        _same(o, lo)
        _same(s, ls)


def test_no_device_memory_is_allocated_per_call():
    import torch
    w = wl.make_chunk("kda_bf16_b8_t4096_h16_d128", B=4, T=2048)
    t = w.torch_inputs("cuda")
    out, sf = _outputs(t, w, True)
    args = (_p(t["q"]), _p(t["k"]), _p(t["v"]), _p(t["beta"]), _p(t["gate"]), None, _p(out), _p(sf),
            w.B, w.T, w.H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16, ldn.LDN_VARIANT_SPLIT,
            torch.cuda.current_stream().cuda_stream)
    assert ldn.ldn_chunk_fwd_noalloc(*args) == ldn.LDN_OK
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for _ in range(5):
        assert ldn.ldn_chunk_fwd_noalloc(*args) == ldn.LDN_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0
    assert ldn.device_status() == ldn.LDN_OK


def test_graph_capture_and_replay():
    """The call captured into a CUDA graph replays to the eager result."""
    import torch
    w = wl.make_chunk(GDN_BASE, B=2, T=700, H=8, s0=True)
    t = w.torch_inputs("cuda")
    eager_o, eager_s = run_noalloc(w, t=t)
    out, sf = _outputs(t, w, True)
    args = (_p(t["q"]), _p(t["k"]), _p(t["v"]), _p(t["beta"]), _p(t["gate"]), _p(t["S0"]), _p(out), _p(sf),
            w.B, w.T, w.H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16, ldn.LDN_VARIANT_SPLIT)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
        st = ldn.ldn_chunk_fwd_noalloc(*args, side.cuda_stream)
    assert st == ldn.LDN_OK
    out.zero_()
    sf.zero_()
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert ldn.device_status() == ldn.LDN_OK
    _same(out, eager_o)
    _same(sf, eager_s)


_FIRST_CALL_UNDER_CAPTURE = r"""
import sys
sys.path.insert(0, sys.argv[1])
import torch
import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl
ldn.load()
torch.cuda.set_device(0)
w = wl.make_chunk("gdn_bf16_b4_t2048_h16_d128", B=1, T=200, H=2, s0=True)
t = w.torch_inputs("cuda")
out = torch.empty((w.B, w.T, w.H, w.dv), dtype=t["q"].dtype, device="cuda")
sf = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
args = (t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), t["beta"].data_ptr(), t["gate"].data_ptr(),
        t["S0"].data_ptr(), out.data_ptr(), sf.data_ptr(), w.B, w.T, w.H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16,
        ldn.LDN_VARIANT_SPLIT)
side = torch.cuda.Stream()
side.wait_stream(torch.cuda.current_stream())
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
    st_cap = ldn.ldn_chunk_fwd_noalloc(*args, side.cuda_stream)
torch.cuda.synchronize()
st_eager = ldn.ldn_chunk_fwd_noalloc(*args, torch.cuda.current_stream().cuda_stream)
torch.cuda.synchronize()
print(st_cap, st_eager, ldn.device_status())
"""


def test_first_call_under_capture_is_rejected_in_a_fresh_process():
    """In a fresh process, a first call made while its stream is being captured
    is refused (LDN_ERR_UNSUPPORTED, nothing enqueued: the capture still ends
    cleanly); the next call, made eagerly, sets the scratch up and runs."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_UNDER_CAPTURE, root], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    st_cap, st_eager, dev = (int(x) for x in r.stdout.strip().splitlines()[-1].split())
    assert st_cap == ldn.LDN_ERR_UNSUPPORTED
    assert st_eager == ldn.LDN_OK and dev == ldn.LDN_OK
