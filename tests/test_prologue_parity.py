"""GPU parity of the prologue (short causal convolution + SiLU, L2 norm, sigmoid
beta, decay gate) and the gated RMSNorm epilogue against the fp64 oracle.

Tolerances from the arithmetic: the kernels compute in fp32 (relative error a few
1e-7 per step), so fp32 outputs must agree to 1e-5 of the RMS and bf16 outputs
to 1e-4 of the RMS beyond the half-ulp rounding of the stored value."""
import numpy as np
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl
from oracle import prologue as op
from tests._helpers import BF16_HALF_ULP, rel_err

pytestmark = pytest.mark.gpu

EPS = 1e-6
TOL = {"f32": 1e-5, "bf16": 1e-4}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def _dev(x, dtype):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(device="cuda", dtype=dtype)


def _p(x):
    return None if x is None else x.data_ptr()


def run_prologue(p, eps=EPS):
    import torch
    el = torch.bfloat16 if p["dtype"] == "bf16" else torch.float32
    f32 = torch.float32
    B, T, H, dk, dv, mode = p["B"], p["T"], p["H"], p["dk"], p["dv"], p["mode"]
    qi, ki, vi = _dev(p["q_in"], el), _dev(p["k_in"], el), _dev(p["v_in"], el)
    cq, ck, cv = _dev(p["conv_q"], f32), _dev(p["conv_k"], f32), _dev(p["conv_v"], f32)
    bl, gz, ga, gb = _dev(p["beta_logit"], f32), _dev(p["gate_z"], f32), _dev(p["gate_a"], f32), _dev(p["gate_b"], f32)
    q = torch.empty((B, T, H, dk), dtype=el, device="cuda")
    k = torch.empty_like(q)
    v = torch.empty((B, T, H, dv), dtype=el, device="cuda")
    beta = torch.empty((B, T, H), dtype=f32, device="cuda")
    gate = None if mode == ldn.LDN_DELTANET else torch.empty(tuple(p["gate_z"].shape), dtype=f32, device="cuda")
    dt = ldn.LDN_BF16 if p["dtype"] == "bf16" else ldn.LDN_F32
    st = ldn.ldn_prologue(_p(qi), _p(ki), _p(vi), _p(cq), _p(ck), _p(cv), p["width"], _p(bl), _p(gz), _p(ga), _p(gb),
                          _p(q), _p(k), _p(v), _p(beta), _p(gate), B, T, H, dk, dv, mode, dt, eps,
                          torch.cuda.current_stream().cuda_stream)
    assert st == ldn.LDN_OK, ldn.ldn_status_string(st)
    torch.cuda.synchronize()
    cpu = lambda x: None if x is None else x.float().cpu().numpy()
    return cpu(q), cpu(k), cpu(v), cpu(beta), cpu(gate)


def check_prologue(p, eps=EPS):
    got = run_prologue(p, eps)
    ref = op.prologue(p["q_in"], p["k_in"], p["v_in"], p["conv_q"], p["conv_k"], p["conv_v"], p["beta_logit"],
                      p["gate_z"], p["gate_a"], p["gate_b"], mode=p["mode"], eps=eps)
    for name, g, r in zip(("q", "k", "v"), got[:3], ref[:3]):
        e = rel_err(g, r, BF16_HALF_ULP if p["dtype"] == "bf16" else 0.0)
        assert e <= TOL[p["dtype"]], f"{name}: {e:.3g}"
    assert rel_err(got[3], ref[3]) <= TOL["f32"], "beta"
    if ref[4] is None:
        assert got[4] is None
    else:
        assert rel_err(got[4], ref[4]) <= TOL["f32"], f"gate {rel_err(got[4], ref[4]):.3g}"
    return got


BASE = {0: "gdn_prologue_bf16_b4_t2048_h16_d128_w4", 1: "gdn_prologue_bf16_b4_t2048_h16_d128_w4",
        2: "kda_prologue_bf16_b8_t4096_h16_d128_w4"}


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_prologue_modes_dtypes_dims(mode, dtype, dk, dv):
    p = wl.make_prologue(BASE[mode], mode=mode, dtype=dtype, B=2, T=150, H=3, dk=dk, dv=dv)
    check_prologue(p)


@pytest.mark.parametrize("width", [1, 2, 3, 4, 5, 8])
def test_prologue_widths(width):
    check_prologue(wl.make_prologue(B=2, T=97, H=2, width=width))


@pytest.mark.parametrize("T", [1, 3, 63, 64, 65, 129])
def test_prologue_lengths(T):
    """Sequences shorter than the convolution, one token, exact and ragged runs."""
    check_prologue(wl.make_prologue(B=3, T=T, H=2, width=4))


def test_prologue_zero_rows_and_eps():
    """All-zero inputs: the convolution gives 0, SiLU(0) = 0 and the L2 norm keeps 0."""
    p = wl.make_prologue(B=1, T=70, H=2, dk=64, dv=64)
    p["q_in"][:] = 0.0
    q, *_ = check_prologue(p, eps=1e-6)
    assert np.all(q == 0.0)
    check_prologue(wl.make_prologue(B=1, T=70, H=2), eps=0.25)


def test_prologue_zero_length_is_a_no_op():
    import torch
    st = ldn.ldn_prologue(None, None, None, None, None, None, 4, None, None, None, None, None, None, None, None, None,
                          1, 0, 2, 128, 128, 1, ldn.LDN_BF16, EPS, torch.cuda.current_stream().cuda_stream)
    assert st == ldn.LDN_OK


def test_prologue_full_gdn_workload():
    check_prologue(wl.make_prologue("gdn_prologue_bf16_b4_t2048_h16_d128_w4"))


def test_prologue_full_kda_workload_sampled():
    """KDA B=8, T=4096, H=16 in the benchmark's launch; two whole sequences against
    the oracle (the convolution and the gates act per sequence and head)."""
    p = wl.make_prologue("kda_prologue_bf16_b8_t4096_h16_d128_w4")
    got = run_prologue(p)
    for b in (0, 7):
        sub = {k: (v[b:b + 1] if isinstance(v, np.ndarray) and v.ndim >= 3 and v.shape[0] == p["B"] else v)
               for k, v in p.items()}
        ref = op.prologue(sub["q_in"], sub["k_in"], sub["v_in"], p["conv_q"], p["conv_k"], p["conv_v"],
                          sub["beta_logit"], sub["gate_z"], p["gate_a"], p["gate_b"], mode=p["mode"], eps=EPS)
        for i, r in enumerate(ref):
            stored = BF16_HALF_ULP if i < 3 else 0.0
            tol = TOL["bf16"] if i < 3 else TOL["f32"]
            assert rel_err(got[i][b:b + 1], r, stored) <= tol, (b, i)


# ---- epilogue ----
def run_rmsnorm(p, eps=EPS, in_place=False):
    import torch
    el = torch.bfloat16 if p["dtype"] == "bf16" else torch.float32
    o, g, w = _dev(p["o"], el), _dev(p["g"], el), _dev(p["gain"], torch.float32)
    y = o if in_place else torch.empty_like(o)
    dt = ldn.LDN_BF16 if p["dtype"] == "bf16" else ldn.LDN_F32
    st = ldn.ldn_rmsnorm_gated(_p(o), _p(g), _p(w), _p(y), p["B"], p["T"], p["H"], p["dv"], dt, eps,
                               torch.cuda.current_stream().cuda_stream)
    assert st == ldn.LDN_OK, ldn.ldn_status_string(st)
    torch.cuda.synchronize()
    return y.float().cpu().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dv", [64, 128])
@pytest.mark.parametrize("in_place", [False, True])
def test_rmsnorm_gated_parity(dtype, dv, in_place):
    p = wl.make_prologue(dtype=dtype, B=2, T=77, H=3, dv=dv)
    y = run_rmsnorm(p, in_place=in_place)
    ref = op.rmsnorm_gated(p["o"], p["g"], p["gain"], EPS)
    assert rel_err(y, ref, BF16_HALF_ULP if dtype == "bf16" else 0.0) <= TOL[dtype]


def test_rmsnorm_gated_full_workload_and_tiny_rows():
    p = wl.make_prologue("gdn_prologue_bf16_b4_t2048_h16_d128_w4")
    assert rel_err(run_rmsnorm(p), op.rmsnorm_gated(p["o"], p["g"], p["gain"], EPS), BF16_HALF_ULP) <= TOL["bf16"]
    p = wl.make_prologue(B=1, T=1, H=1, dv=64)   # a single row (one walker, 63 idle rows)
    assert rel_err(run_rmsnorm(p), op.rmsnorm_gated(p["o"], p["g"], p["gain"], EPS), BF16_HALF_ULP) <= TOL["bf16"]
    p["o"][:] = 0.0
    assert np.all(run_rmsnorm(p) == 0.0)
