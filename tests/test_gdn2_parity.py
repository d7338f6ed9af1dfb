"""GPU parity of the Gated DeltaNet-2 entry points (ldn_chunk_fwd_gdn2,
ldn_decode_step_gdn2) against the fp64 oracle, element by element, with the
tolerances of the other modes: max|gpu - oracle| / RMS(oracle) within 1e-4 for
fp32 inputs and 2e-2 for bf16 inputs (fp32 state).  Sizes span several
64-token chunks and a ragged tail."""
import numpy as np
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import workloads as wl
from tests._helpers import TOL, fmt_parity, out_err, parity, rel_err
import oracle

pytestmark = pytest.mark.gpu

CHUNK = "gdn2_bf16_b8_t4096_h16_d128"
DECODE = "gdn2_decode_b64_h16_dk128_dv128_steps1000"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def run_chunk(w, S0=True, variant=ldn.LDN_VARIANT_AUTO):
    import torch
    t = w.torch_inputs("cuda")
    out, sf = ldn.chunk_fwd_gdn2(t["q"], t["k"], t["v"], t["erase"], t["write"], t["gate"], t["S0"] if S0 else None,
                                 variant=variant)
    assert ldn.device_status() == ldn.LDN_OK
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), sf.cpu().numpy()


VARIANTS = [ldn.LDN_VARIANT_SIMT, ldn.LDN_VARIANT_TENSOR, ldn.LDN_VARIANT_SPLIT]


def check_chunk(w, variant=ldn.LDN_VARIANT_AUTO):
    o, s = run_chunk(w, variant=variant)
    ro, rs = oracle.fwd_gdn2(w.q, w.k, w.v, w.erase, w.write, w.gate, w.S0)
    eo, es = out_err(o, ro, w.dtype), rel_err(s, rs)
    assert eo <= TOL[w.dtype] and es <= TOL[w.dtype], f"out {eo:.3g} state {es:.3g}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_chunk_parity_dtypes_dims(dtype, dk, dv):
    w = wl.make_chunk(CHUNK, B=2, T=200, H=3, dk=dk, dv=dv, dtype=dtype, s0=True)
    check_chunk(w)
    check_chunk(w, ldn.LDN_VARIANT_SIMT)


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 129])
@pytest.mark.parametrize("variant", VARIANTS)
def test_chunk_parity_lengths(T, variant):
    check_chunk(wl.make_chunk(CHUNK, B=1, T=T, H=2, s0=(T % 2 == 1)), variant)


@pytest.mark.parametrize("variant", [ldn.LDN_VARIANT_TENSOR, ldn.LDN_VARIANT_SPLIT])
@pytest.mark.parametrize("B,T,H,dv,s0", [(2, 200, 3, 128, True), (1, 64, 2, 64, False), (1, 700, 1, 128, True),
                                         (2, 333, 2, 64, True), (1, 1, 1, 128, True)])
def test_chunk_tensor_core_variants(variant, B, T, H, dv, s0):
    """The tcgen05 kernels: K rows carry b * K, beta = 1, V enters as w * V."""
    check_chunk(wl.make_chunk(CHUNK, B=B, T=T, H=H, dv=dv, s0=s0), variant)


@pytest.mark.parametrize("variant", [ldn.LDN_VARIANT_TENSOR, ldn.LDN_VARIANT_SPLIT])
def test_chunk_strong_channel_gates_entrywise_chunks(variant):
    """Chunks whose per-channel decay span leaves the fp16 factors are formed entry
    by entry (erase gate applied per entry there); the others through the MMA."""
    w = wl.make_chunk(CHUNK, B=1, T=320, H=2, s0=True)
    g = w.gate.copy()
    g[:, 64:192, :, 5] = -1.2
    g[:, 256:300, 1, 100] = -0.9
    w.gate = g.astype(np.float32)
    check_chunk(w, variant)
    w.gate = np.full_like(w.gate, -0.6)   # every chunk entry by entry
    check_chunk(w, variant)


def test_chunk_tensor_core_erase_and_write_extremes():
    """b = 0 on some tokens (nothing erased), w = 0 on others (nothing written),
    b = w = 1 on the rest: the gates reach the operands they belong to."""
    w = wl.make_chunk(CHUNK, B=1, T=250, H=2, s0=True)
    w.erase[:, 10:80] = 0.0
    w.write[:, 60:140] = 0.0
    w.erase[:, 200:] = 1.0
    w.write[:, 200:] = 1.0
    for variant in VARIANTS:
        check_chunk(w, variant)


def test_chunk_tensor_core_with_both_gates_beta_matches_kda():
    """The same reduction through the tensor-core kernels (fused and split): the
    GDN2 and KDA builds differ only in where beta enters, so the two agree to the
    fp16 operand rounding."""
    import torch
    k = wl.make_chunk("kda_bf16_b8_t4096_h16_d128", B=2, T=260, H=2, s0=True)
    t = k.torch_inputs("cuda")
    erase = t["beta"][..., None].expand(*t["beta"].shape, k.dk).contiguous()
    write = t["beta"][..., None].expand(*t["beta"].shape, k.dv).contiguous()
    for variant in (ldn.LDN_VARIANT_TENSOR, ldn.LDN_VARIANT_SPLIT):
        o2, s2 = ldn.chunk_fwd_gdn2(t["q"], t["k"], t["v"], erase, write, t["gate"], t["S0"], variant=variant)
        ok, sk = ldn.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["gate"], t["S0"], mode=ldn.LDN_KDA,
                               variant=variant)
        torch.cuda.synchronize()
        ro, rs = oracle.fwd(k.q, k.k, k.v, k.beta, k.gate, k.S0, mode=oracle.MODE_KDA)
        assert out_err(o2.float().cpu().numpy(), ro, "bf16") <= TOL["bf16"]
        assert rel_err(s2.cpu().numpy(), rs) <= TOL["bf16"]
        # both outputs are rounded to bf16 independently: one bf16 ulp (2^-7 of the value)
        # apart at most, beyond the difference of the unrounded values
        a, c = o2.float().cpu().numpy(), ok.float().cpu().numpy()
        assert np.maximum(np.abs(a - c) - 2.0 ** -7 * np.abs(c), 0.0).max() / np.sqrt(np.mean(c ** 2)) <= 1e-2


def test_chunk_with_both_gates_beta_matches_the_kda_kernel():
    """b = beta 1 and w = beta 1 turn the rule into KDA: the GDN2 entry point must
    agree with the KDA path of ldn_chunk_fwd (SIMT kernel) on the same inputs."""
    import torch
    k = wl.make_chunk("kda_bf16_b8_t4096_h16_d128", B=2, T=150, H=2, dtype="f32", s0=True)
    t = k.torch_inputs("cuda")
    erase = t["beta"][..., None].expand(*t["beta"].shape, k.dk).contiguous()
    write = t["beta"][..., None].expand(*t["beta"].shape, k.dv).contiguous()
    o2, s2 = ldn.chunk_fwd_gdn2(t["q"], t["k"], t["v"], erase, write, t["gate"], t["S0"],
                                variant=ldn.LDN_VARIANT_SIMT)
    ok, sk = ldn.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["gate"], t["S0"], mode=ldn.LDN_KDA,
                           variant=ldn.LDN_VARIANT_SIMT)
    torch.cuda.synchronize()
    assert rel_err(o2.cpu().numpy(), ok.cpu().numpy()) <= 1e-5
    assert rel_err(s2.cpu().numpy(), sk.cpu().numpy()) <= 1e-5


def test_chunk_erase_off_is_additive():
    """b = 0: nothing is erased, the state only decays and accumulates w v k^T."""
    w = wl.make_chunk(CHUNK, B=1, T=130, H=2, dtype="f32", s0=True)
    w.erase = np.zeros_like(w.erase)
    check_chunk(w)


def test_chunk_zero_length_copies_state():
    import torch
    w = wl.make_chunk(CHUNK, B=2, T=3, H=2, s0=True)
    t = w.torch_inputs("cuda")
    S_final = torch.full_like(t["S0"], 7.0)
    st = ldn.ldn_chunk_fwd_gdn2(0, 0, 0, 0, 0, 0, t["S0"].data_ptr(), 0, S_final.data_ptr(), 2, 0, 2, 128, 128,
                                64, 1, ldn.LDN_VARIANT_AUTO, torch.cuda.current_stream().cuda_stream)
    assert st == ldn.LDN_OK
    torch.cuda.synchronize()
    assert torch.equal(S_final, t["S0"])


@pytest.mark.parametrize("variant", [ldn.LDN_VARIANT_TENSOR, ldn.LDN_VARIANT_SIMT])
def test_chunk_full_workload_sampled(variant):
    """B=8, T=4096, H=16, d=128 bf16 in one call; sampled (b, h) against the oracle."""
    w = wl.make_chunk(CHUNK)
    o, s = run_chunk(w, S0=False, variant=variant)
    for b, h in [(0, 0), (5, 11), (7, 15)]:
        sl = lambda a: a[b:b + 1, :, h:h + 1]
        ro, rs = oracle.fwd_gdn2(sl(w.q), sl(w.k), sl(w.v), sl(w.erase), sl(w.write), sl(w.gate), None)
        assert out_err(o[b:b + 1, :, h:h + 1], ro, "bf16") <= TOL["bf16"]
        assert rel_err(s[b:b + 1, h:h + 1], rs) <= TOL["bf16"]


def test_chunk_full_workload_whole_tensors():
    """B=8, T=4096, H=16, d=128 bf16 in one call with the variant the library
    picks: every output and final-state element against the oracle."""
    w = wl.make_chunk(CHUNK)
    o, s = run_chunk(w, S0=False, variant=ldn.LDN_VARIANT_AUTO)
    ro, rs = oracle.fwd_gdn2(w.q, w.k, w.v, w.erase, w.write, w.gate, None)
    po, ps = parity(o, ro, "bf16"), parity(s, rs, "f32", tol=TOL["bf16"])
    print(f"\n{CHUNK}: output: {fmt_parity(po)}; final state: plain {ps['plain']:.3g}")
    assert po["excess"] <= TOL["bf16"] and ps["plain"] <= TOL["bf16"]


def run_decode(w):
    import torch
    t = w.torch_inputs("cuda")
    S = t["S0"].clone()
    outs = [ldn.decode_step_gdn2(t["q"][i], t["k"][i], t["v"][i], t["erase"][i], t["write"][i], t["gate"][i], S)
            for i in range(w.T)]
    assert ldn.device_status() == ldn.LDN_OK
    return torch.stack(outs).float().cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (64, 64), (128, 64)])
def test_decode_parity(dtype, dk, dv):
    w = wl.make_decode(DECODE, B=3, H=5, dk=dk, dv=dv, steps=24, dtype=dtype)
    o, S = run_decode(w)
    ro, rs = oracle.decode_gdn2(w.q, w.k, w.v, w.erase, w.write, w.gate, w.S0)
    assert out_err(o, ro, dtype) <= TOL[dtype]
    assert rel_err(S, rs) <= TOL[dtype]


def test_decode_full_1000_steps_whole_tensors():
    """B=64 x H=16, 1000 consecutive tokens: every output of every step and the
    whole final state against the oracle."""
    w = wl.make_decode(DECODE)
    o, S = run_decode(w)
    ro, rs = oracle.decode_gdn2(w.q, w.k, w.v, w.erase, w.write, w.gate, w.S0)
    po, ps = parity(o, ro, "f32"), parity(S, rs, "f32")
    print(f"\n{DECODE}: outputs plain {po['plain']:.3g}; state plain {ps['plain']:.3g}")
    assert np.all(np.isfinite(o))
    assert po["plain"] <= TOL["f32"] and ps["plain"] <= TOL["f32"]


def test_chunk_split_through_the_library_scratch_in_pieces():
    """B=2, T=16384, H=16: the split variant's workspace (330 MB per sequence)
    exceeds the library's 256 MiB array, so the call is cut into token runs with
    the state carried between them; the erase and write gates must follow every
    piece's offset.  Sampled (b, h) against the oracle."""
    import torch
    w = wl.make_chunk(CHUNK, B=2, T=16384, H=16, s0=True)
    o, s = run_chunk(w, variant=ldn.LDN_VARIANT_SPLIT)
    for b, h in [(0, 3), (1, 14)]:
        sl = lambda a: a[b:b + 1, :, h:h + 1]
        ro, rs = oracle.fwd_gdn2(sl(w.q), sl(w.k), sl(w.v), sl(w.erase), sl(w.write), sl(w.gate),
                                 w.S0[b:b + 1, h:h + 1], nthreads=1)
        assert out_err(o[b:b + 1, :, h:h + 1], ro, "bf16") <= TOL["bf16"]
        assert rel_err(s[b:b + 1, h:h + 1], rs) <= TOL["bf16"]
    torch.cuda.empty_cache()
