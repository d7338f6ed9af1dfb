"""GPU parity of ldn_chunk_fwd against the fp64 oracle, element by element.

Sizes span several 64-token chunks and a ragged tail; each case compares every
output and the final state with max|gpu - oracle| / RMS(oracle) within 1e-4
(fp32 inputs) or 2e-2 (bf16 inputs, fp32 state)."""
import numpy as np
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl
from tests._helpers import TOL, fmt_parity, oracle_chunk, out_err, parity, rel_err

pytestmark = pytest.mark.gpu

BASE = {0: "deltanet_fp32_b1_t256_h1_d64", 1: "gdn_bf16_b4_t2048_h16_d128", 2: "kda_bf16_b8_t4096_h16_d128"}
MODE_NAME = {0: "deltanet", 1: "gdn", 2: "kda"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def run_gpu(w, variant=ldn.LDN_VARIANT_AUTO, S0=True, want_state=True, workspace=False):
    """workspace=True: through ldn_chunk_fwd_ws with a workspace of
    ldn_chunk_fwd_workspace_size bytes, as the benchmark calls it (AUTO may then pick a
    workspace variant)."""
    import torch
    t = w.torch_inputs("cuda")
    ws = None
    if workspace:
        need = ldn.ldn_chunk_fwd_workspace_size(w.B, w.T, w.H, w.dk, w.dv, 64, w.mode,
                                                ldn.LDN_BF16 if w.dtype == "bf16" else ldn.LDN_F32)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    out, sf = ldn.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["gate"], t["S0"] if S0 else None,
                            mode=w.mode, variant=variant, want_state=want_state, workspace=ws)
    assert ldn.device_status() == ldn.LDN_OK
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), (None if sf is None else sf.cpu().numpy())


def check(w, variant=ldn.LDN_VARIANT_AUTO, tol=None):
    tol = tol or TOL[w.dtype]
    o, s = run_gpu(w, variant)
    ro, rs = oracle_chunk(w)
    eo, es = out_err(o, ro, w.dtype), rel_err(s, rs)
    assert eo <= tol and es <= tol, f"{w.name} {w.dtype} variant={variant}: out {eo:.3g} state {es:.3g} (tol {tol})"
    return eo, es


# ---- every mode x dtype x head size, ragged tails, with and without S0 ----
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_parity_modes_dtypes_dims(mode, dtype, dk, dv):
    w = wl.make_chunk(BASE[mode], B=2, T=200, H=3, dk=dk, dv=dv, mode=mode, dtype=dtype, s0=True)
    check(w)


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 129, 321])
@pytest.mark.parametrize("mode", [1, 2])
def test_parity_lengths(T, mode):
    w = wl.make_chunk(BASE[mode], B=1, T=T, H=2, s0=(T % 2 == 1))
    check(w)


@pytest.mark.parametrize("variant", [ldn.LDN_VARIANT_SIMT])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_simt_variant_on_bf16(variant, mode):
    w = wl.make_chunk(BASE[mode], B=2, T=150, H=2, mode=mode, dtype="bf16", s0=True)
    check(w, variant)


def test_config_deltanet_fp32_full():
    """The fp32 DeltaNet workload at its full size (B=1, T=256, H=1, d=64)."""
    w = wl.make_chunk("deltanet_fp32_b1_t256_h1_d64")
    check(w)


def test_zero_length_copies_state():
    import torch
    w = wl.make_chunk(BASE[1], B=2, T=3, H=2, s0=True)
    t = w.torch_inputs("cuda")
    S_final = torch.full_like(t["S0"], 7.0)
    st = ldn.ldn_chunk_fwd(0, 0, 0, 0, 0, t["S0"].data_ptr(), 0, S_final.data_ptr(), 2, 0, 2, 128, 128,
                           64, 1, 1, torch.cuda.current_stream().cuda_stream)
    assert st == ldn.LDN_OK
    torch.cuda.synchronize()
    assert torch.equal(S_final, t["S0"])
    st = ldn.ldn_chunk_fwd(0, 0, 0, 0, 0, 0, 0, S_final.data_ptr(), 2, 0, 2, 128, 128, 64, 1, 1,
                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == ldn.LDN_OK and float(S_final.abs().max()) == 0.0


def test_no_state_output_and_null_s0():
    w = wl.make_chunk(BASE[2], B=1, T=100, H=2, s0=False)
    o, s = run_gpu(w, want_state=False)
    assert s is None
    ro, _ = oracle_chunk(w)
    assert out_err(o, ro, "bf16") <= TOL["bf16"]


def test_state_output_may_alias_initial_state():
    import torch
    w = wl.make_chunk(BASE[1], B=2, T=130, H=2, s0=True)
    t = w.torch_inputs("cuda")
    S = t["S0"].clone()
    out, sf = ldn.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["gate"], S, mode=1, S_final=S)
    torch.cuda.synchronize()
    ro, rs = oracle_chunk(w)
    assert out_err(out.float().cpu().numpy(), ro, "bf16") <= TOL["bf16"]
    assert rel_err(S.cpu().numpy(), rs) <= TOL["bf16"]


@pytest.mark.parametrize("mode", [1, 2])
def test_state_passing_split_equals_full(mode):
    """Resume: S_final of the first part seeds the second part."""
    import torch
    w = wl.make_chunk(BASE[mode], B=2, T=300, H=2, s0=True)
    t = w.torch_inputs("cuda")
    cut = 130
    sl = lambda x, a, b: None if x is None else x[:, a:b].contiguous()
    o1, s1 = ldn.chunk_fwd(sl(t["q"], 0, cut), sl(t["k"], 0, cut), sl(t["v"], 0, cut), sl(t["beta"], 0, cut),
                           sl(t["gate"], 0, cut), t["S0"], mode=mode)
    o2, s2 = ldn.chunk_fwd(sl(t["q"], cut, None), sl(t["k"], cut, None), sl(t["v"], cut, None),
                           sl(t["beta"], cut, None), sl(t["gate"], cut, None), s1, mode=mode)
    torch.cuda.synchronize()
    ro, rs = oracle_chunk(w)
    o = torch.cat([o1, o2], dim=1).float().cpu().numpy()
    assert out_err(o, ro, "bf16") <= TOL["bf16"]
    assert rel_err(s2.cpu().numpy(), rs) <= TOL["bf16"]


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_degenerate_beta(mode):
    """beta = 0 (memory only decays) and beta = 1 (exact overwrite along k)."""
    for bval in (0.0, 1.0):
        w = wl.make_chunk(BASE[mode], B=1, T=140, H=2, mode=mode, s0=True)
        w.beta = np.full_like(w.beta, bval)
        check(w)


def test_strong_gdn_gates():
    """Large per-token decays (log alpha ~ -2): the decayed chunk products stay finite
    for a scalar gate because only e^{g_r - g_j}, r >= j, is ever needed."""
    w = wl.make_chunk(BASE[1], B=1, T=200, H=2, s0=True)
    w.gate = (w.gate * 20).astype(np.float32)
    check(w)


@pytest.mark.parametrize("variant", [ldn.LDN_VARIANT_TENSOR, ldn.LDN_VARIANT_SIMT])
def test_kda_tensor_and_simt_paths(variant):
    """KDA through the tensor-core kernel (per-channel decay split about the
    chunk's middle row) and through the CUDA-core kernel, on the same inputs."""
    w = wl.make_chunk(BASE[2], B=2, T=333, H=3, s0=True)
    check(w, variant)


def test_kda_strong_channel_gates_entrywise_chunks():
    """Per-channel decays strong enough (log a ~ -1.2 on a few channels, in some
    chunks only) that the fp16 decay factors would leave their range: those
    chunks are formed entry by entry, the others through the factored MMA."""
    w = wl.make_chunk(BASE[2], B=1, T=320, H=2, s0=True)
    g = w.gate.copy()
    g[:, 64:192, :, 5] = -1.2      # chunks 1 and 2, channel 5
    g[:, 256:300, 1, 100] = -0.9   # chunk 4, head 1, channel 100
    w.gate = g.astype(np.float32)
    check(w, ldn.LDN_VARIANT_TENSOR)


def test_kda_all_chunks_entrywise():
    """Every chunk beyond the factored range (log a = -0.6 on every channel)."""
    w = wl.make_chunk(BASE[2], B=1, T=200, H=2, s0=True)
    w.gate = np.full_like(w.gate, -0.6)
    check(w, ldn.LDN_VARIANT_TENSOR)


# ---- split variant: parallel chunk preparation into a workspace, then the state chain ----
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("B,T,H,dv,s0", [(2, 200, 3, 128, True), (1, 64, 2, 64, False), (1, 1, 1, 128, True),
                                         (1, 700, 1, 128, True), (2, 333, 2, 64, True)])
def test_split_variant_parity(mode, B, T, H, dv, s0):
    w = wl.make_chunk(BASE[mode], B=B, T=T, H=H, dk=128, dv=dv, mode=mode, dtype="bf16", s0=s0)
    check(w, ldn.LDN_VARIANT_SPLIT)


def test_split_variant_kda_strong_gates():
    """Entry-wise chunks (spans beyond the fp16 factors) through the split variant."""
    w = wl.make_chunk(BASE[2], B=1, T=320, H=2, s0=True)
    g = w.gate.copy()
    g[:, 64:192, :, 5] = -1.2
    g[:, 256:300, 1, 100] = -0.9
    w.gate = g.astype(np.float32)
    check(w, ldn.LDN_VARIANT_SPLIT)


def test_split_equals_fused_up_to_rounding():
    """Same inputs through both tensor-core variants: same result up to rounding."""
    w = wl.make_chunk(BASE[1], B=2, T=500, H=4, s0=True)
    o1, s1 = run_gpu(w, ldn.LDN_VARIANT_TENSOR)
    o2, s2 = run_gpu(w, ldn.LDN_VARIANT_SPLIT)
    # Both outputs are bf16-rounded independently, so they may differ by one bf16 ulp
    # (up to 2^-7 of the value) on top of the difference of the unrounded values.
    ulp_excess = np.maximum(np.abs(o2 - o1) - 2.0 ** -7 * np.abs(o1), 0.0).max() / np.sqrt(np.mean(o1 ** 2))
    assert ulp_excess < 1e-2 and rel_err(s2, s1) < 1e-2


# ---- split variant with the sequence split: long (b, h) cut into segments run side by side ----
def _segments(w, ws_bytes):
    return ldn.ldn_chunk_fwd_split_segments(w.B, w.T, w.H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16, ws_bytes)


def _base_bytes(w):
    """The operand images alone (no room for the segment states and maps)."""
    return w.B * w.H * ((w.T + 63) // 64) * (32768 + (w.dv // 64) * 16384 + 16896)


@pytest.mark.parametrize("mode,B,T,H,s0,nseg", [(1, 1, 8192 + 37, 1, True, 8), (1, 1, 64 * 60 + 5, 2, True, 3),
                                                (2, 1, 5000, 3, True, 4), (0, 2, 4000, 2, False, 3),
                                                (1, 1, 64 * 112, 1, False, 7)])
def test_sequence_split_parity(mode, B, T, H, s0, nseg):
    """Segment counts 3 .. 8, ragged last chunk and uneven last segment, with and without
    S0, every mode; the whole output and final state against the oracle."""
    w = wl.make_chunk(BASE[mode], B=B, T=T, H=H, dk=128, dv=128, mode=mode, dtype="bf16", s0=s0)
    need = ldn.ldn_chunk_fwd_workspace_size(w.B, w.T, w.H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16)
    assert need > _base_bytes(w) and _segments(w, need) == nseg
    o, s = run_gpu(w, ldn.LDN_VARIANT_SPLIT, S0=s0, workspace=True)
    ro, rs = oracle_chunk(w)
    eo, es = out_err(o, ro, w.dtype), rel_err(s, rs)
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], f"nseg {nseg}: out {eo:.3g} state {es:.3g}"


def test_sequence_split_matches_unsplit_recurrence():
    """The same call with a workspace of the operand images alone runs the recurrence
    unsplit: both forms agree up to rounding (the maps compose in fp32), and without a
    final state asked for."""
    import torch
    w = wl.make_chunk(BASE[1], B=1, T=6000, H=2, s0=True)
    t = w.torch_inputs("cuda")
    base = _base_bytes(w)
    need = ldn.ldn_chunk_fwd_workspace_size(w.B, w.T, w.H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16)
    assert _segments(w, need) >= 3 and _segments(w, base) == 1
    res = []
    for nbytes in (base, need):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        o, sf = ldn.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["gate"], t["S0"], mode=w.mode,
                              variant=ldn.LDN_VARIANT_SPLIT, workspace=ws)
        o2, sf2 = ldn.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["gate"], t["S0"], mode=w.mode,
                                variant=ldn.LDN_VARIANT_SPLIT, want_state=False, workspace=ws)
        torch.cuda.synchronize()
        assert ldn.device_status() == ldn.LDN_OK and sf2 is None
        assert torch.equal(o, o2)
        res.append((o.float().cpu().numpy(), sf.cpu().numpy()))
    (o1, s1), (o2, s2) = res
    ulp_excess = np.maximum(np.abs(o2 - o1) - 2.0 ** -7 * np.abs(o1), 0.0).max() / np.sqrt(np.mean(o1 ** 2))
    assert ulp_excess < 1e-2 and rel_err(s2, s1) < 1e-2


# ---- cluster-pair variant (two CTAs per (b, h) share the preparation) ----
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("B,T,H,s0", [(1, 64, 1, False), (2, 65, 3, True), (1, 1, 2, True), (2, 500, 4, True),
                                      (1, 1000, 2, False), (3, 128, 5, True)])
def test_pair_variant_parity(mode, B, T, H, s0):
    w = wl.make_chunk(BASE[mode], dtype="bf16", B=B, T=T, H=H, dk=128, dv=128, s0=s0)
    check(w, ldn.LDN_VARIANT_PAIR)


@pytest.mark.parametrize("mode", [0, 1])
def test_pair_equals_fused_bitwise(mode):
    """The pair's CTAs compute every chunk's operands with the fused kernel's arithmetic
    (the peer's copy is the same bits), so the results are identical."""
    w = wl.make_chunk(BASE[mode], dtype="bf16", B=2, T=777, H=3, dk=128, dv=128, s0=True)
    o1, s1 = run_gpu(w, ldn.LDN_VARIANT_TENSOR)
    o2, s2 = run_gpu(w, ldn.LDN_VARIANT_PAIR)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_pair_strong_gates_entrywise_chunks():
    """Gated DeltaNet chunks whose log-decay span exceeds the factored form, in both CTAs'
    chunks (even and odd)."""
    w = wl.make_chunk(BASE[1], B=1, T=256, H=2, s0=True)
    w.gate = (w.gate * 40.0).astype(np.float32)
    check(w, ldn.LDN_VARIANT_PAIR)


# ---- full-size workloads in the benchmark's launch configuration ----
def _sampled(name, picks, variant=ldn.LDN_VARIANT_AUTO, **over):
    import torch
    w = wl.make_chunk(name, **over)
    o, s = run_gpu(w, variant)
    for b, h in picks:
        sub = wl.Workload(name=w.name, mode=w.mode, dtype=w.dtype, B=1, T=w.T, H=1, dk=w.dk, dv=w.dv,
                          q=w.q[b:b + 1, :, h:h + 1], k=w.k[b:b + 1, :, h:h + 1], v=w.v[b:b + 1, :, h:h + 1],
                          beta=w.beta[b:b + 1, :, h:h + 1],
                          gate=None if w.gate is None else w.gate[b:b + 1, :, h:h + 1],
                          S0=None if w.S0 is None else w.S0[b:b + 1, h:h + 1])
        ro, rs = oracle_chunk(sub)
        eo = out_err(o[b:b + 1, :, h:h + 1], ro, w.dtype)
        es = rel_err(s[b:b + 1, h:h + 1], rs)
        assert eo <= TOL[w.dtype] and es <= TOL[w.dtype], f"{name} (b={b},h={h}): out {eo:.3g} state {es:.3g}"
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(s))


# Every output element and every final-state element of each full-size
# chunkwise workload (Gated DeltaNet B=4 T=2048; KDA B=8 T=4096; the long
# Gated DeltaNet sequences T = 8192, 32768, 65536 with S0), computed as the
# benchmark launches it (ldn_chunk_fwd_ws with a workspace, the variant the
# library picks), against the oracle over the whole tensor.
FULL_WORKLOADS = ["gdn_bf16_b4_t2048_h16_d128", "kda_bf16_b8_t4096_h16_d128", "gdn_bf16_long_b1_t8192_h16_d128",
                  "gdn_bf16_long_b1_t32768_h16_d128", "gdn_bf16_long_b1_t65536_h16_d128"]


@pytest.mark.parametrize("name", FULL_WORKLOADS)
def test_full_workload_whole_tensors(name):
    w = wl.make_chunk(name)
    o, s = run_gpu(w, workspace=True)
    ro, rs = oracle_chunk(w)
    po, ps = parity(o, ro, w.dtype), parity(s, rs, "f32", tol=TOL[w.dtype])
    print(f"\n{name}: output: {fmt_parity(po)}; final state: plain {ps['plain']:.3g} over {ps['n']} elements")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(s))
    assert po["excess"] <= TOL[w.dtype], f"{name}: output {fmt_parity(po)}"
    assert ps["plain"] <= TOL[w.dtype], f"{name}: final state {ps['plain']:.3g}"


@pytest.mark.parametrize("name,picks", [("gdn_bf16_b4_t2048_h16_d128", [(0, 0), (3, 15)]),
                                        ("kda_bf16_b8_t4096_h16_d128", [(7, 12)]),
                                        ("gdn_bf16_long_b1_t65536_h16_d128", [(0, 5)])])
def test_full_workloads_split_variant_sampled(name, picks):
    _sampled(name, picks, ldn.LDN_VARIANT_SPLIT)


@pytest.mark.parametrize("name,picks", [("kda_bf16_b8_t4096_h16_d128", [(0, 3), (7, 12)]),
                                        ("gdn_bf16_long_b1_t65536_h16_d128", [(0, 5)])])
def test_full_workloads_presolved_variant_sampled(name, picks):
    _sampled(name, picks, ldn.LDN_VARIANT_PRESOLVED)


@pytest.mark.parametrize("name,picks", [("gdn_bf16_b4_t2048_h16_d128", [(0, 0), (2, 9), (3, 15)]),
                                        ("gdn_bf16_long_b1_t8192_h16_d128", [(0, 5)])])
def test_full_workloads_pair_variant_sampled(name, picks):
    _sampled(name, picks, ldn.LDN_VARIANT_PAIR)
