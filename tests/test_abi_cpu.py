"""CPU-side checks of the C ABI: the library loads without a GPU, exports
every entry point include/ldn.h declares, and rejects bad arguments
synchronously (these paths run before any CUDA call)."""
import os
import re

import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from gated_delta_rule_chunkwise_gb300 import build as ldn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ldn_build.build()
    return ldn.load()


def _declared(header):
    txt = open(os.path.join(ROOT, "include", header)).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return set(re.findall(r"\b(ldn_\w+)\s*\(", txt))


def test_headers_are_the_two_libraries():
    assert sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")) == ["ldn.h",
                                                                                               "ldn_diag.h"]


def test_exports_every_declared_symbol(lib):
    declared = _declared("ldn.h")
    assert {"ldn_chunk_fwd", "ldn_decode_step"} <= declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ldn.h but not exported"
    assert set(ldn.EXPORTS) == declared


def test_diagnostics_live_in_their_own_library(lib):
    """include/ldn_diag.h is exported by the test-only libldn_diag.so and by
    nothing in the product library."""
    from tests import _diag
    declared = _declared("ldn_diag.h")
    assert {"ldn_diag_wait_timeout", "ldn_diag_get_device_status"} <= declared
    d = _diag.load()
    for name in declared:
        assert hasattr(d, name), f"{name} declared in include/ldn_diag.h but not exported"
        assert not hasattr(lib, name), f"{name} is exported by the product library"
    assert set(_diag.SIGNATURES) == declared


def test_version_and_status_strings(lib):
    assert ldn.ldn_version() == 7
    for st in range(5):
        assert isinstance(ldn.ldn_status_string(st), str) and ldn.ldn_status_string(st)
    assert "unknown" in ldn.ldn_status_string(99)


FAKE = 1 << 20          # a 16-byte aligned, never dereferenced address


def _chunk(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, beta=FAKE, gate=FAKE, S0=None, out=FAKE, S_final=None,
             B=1, T=64, H=1, dk=64, dv=64, chunk=64, mode=1, dtype=1, variant=0, stream=None)
    a.update(kw)
    return ldn.ldn_chunk_fwd_variant(a["q"], a["k"], a["v"], a["beta"], a["gate"], a["S0"], a["out"],
                                     a["S_final"], a["B"], a["T"], a["H"], a["dk"], a["dv"], a["chunk"],
                                     a["mode"], a["dtype"], a["variant"], a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(k=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(v=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(beta=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(out=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(gate=None, mode=1), ldn.LDN_ERR_INVALID_ARG),
    (dict(gate=None, mode=2), ldn.LDN_ERR_INVALID_ARG),
    (dict(q=FAKE + 4), ldn.LDN_ERR_INVALID_ARG),            # misaligned
    (dict(S0=FAKE + 8), ldn.LDN_ERR_INVALID_ARG),
    (dict(out=FAKE + 2), ldn.LDN_ERR_INVALID_ARG),
    (dict(beta=FAKE + 2), ldn.LDN_ERR_INVALID_ARG),
    (dict(gate=FAKE + 1), ldn.LDN_ERR_INVALID_ARG),
    (dict(mode=3), ldn.LDN_ERR_INVALID_ARG),
    (dict(mode=-1), ldn.LDN_ERR_INVALID_ARG),
    (dict(dtype=2), ldn.LDN_ERR_INVALID_ARG),
    (dict(B=0), ldn.LDN_ERR_INVALID_ARG),
    (dict(H=0), ldn.LDN_ERR_INVALID_ARG),
    (dict(T=-1), ldn.LDN_ERR_INVALID_ARG),
    (dict(variant=3), ldn.LDN_ERR_INVALID_ARG),
    (dict(dk=96), ldn.LDN_ERR_UNSUPPORTED),
    (dict(dv=32), ldn.LDN_ERR_UNSUPPORTED),
    (dict(dk=0), ldn.LDN_ERR_INVALID_ARG),
    (dict(chunk=32), ldn.LDN_ERR_UNSUPPORTED),
    (dict(variant=2, dtype=0), ldn.LDN_ERR_UNSUPPORTED),    # tensor cores need bf16
])
def test_chunk_rejects_bad_arguments(lib, kw, want):
    assert _chunk(**kw) == want


def _decode(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, beta=FAKE, gate=FAKE, S=FAKE, out=FAKE, B=1, H=1, dk=64, dv=64,
             mode=1, dtype=0, stream=None)
    a.update(kw)
    return ldn.ldn_decode_step(a["q"], a["k"], a["v"], a["beta"], a["gate"], a["S"], a["out"], a["B"],
                               a["H"], a["dk"], a["dv"], a["mode"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(S=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(q=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(gate=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(S=FAKE + 4), ldn.LDN_ERR_INVALID_ARG),
    (dict(q=FAKE + 2), ldn.LDN_ERR_INVALID_ARG),             # fp32 q needs 4-byte alignment
    (dict(beta=FAKE + 1), ldn.LDN_ERR_INVALID_ARG),
    (dict(B=0), ldn.LDN_ERR_INVALID_ARG),
    (dict(mode=7), ldn.LDN_ERR_INVALID_ARG),
    (dict(dk=32), ldn.LDN_ERR_UNSUPPORTED),
])
def test_decode_rejects_bad_arguments(lib, kw, want):
    assert _decode(**kw) == want


def _chunk_gdn2(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, erase=FAKE, write=FAKE, gate=FAKE, S0=None, out=FAKE, S_final=None,
             B=1, T=64, H=1, dk=64, dv=64, chunk=64, dtype=1, variant=0, stream=None)
    a.update(kw)
    return ldn.ldn_chunk_fwd_gdn2(a["q"], a["k"], a["v"], a["erase"], a["write"], a["gate"], a["S0"], a["out"],
                                  a["S_final"], a["B"], a["T"], a["H"], a["dk"], a["dv"], a["chunk"], a["dtype"],
                                  a["variant"], a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(erase=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(write=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(gate=None), ldn.LDN_ERR_INVALID_ARG),            # the decay is part of the rule
    (dict(out=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(q=FAKE + 4), ldn.LDN_ERR_INVALID_ARG),
    (dict(S_final=FAKE + 8), ldn.LDN_ERR_INVALID_ARG),
    (dict(erase=FAKE + 2), ldn.LDN_ERR_INVALID_ARG),
    (dict(write=FAKE + 1), ldn.LDN_ERR_INVALID_ARG),
    (dict(dtype=5), ldn.LDN_ERR_INVALID_ARG),
    (dict(B=0), ldn.LDN_ERR_INVALID_ARG),
    (dict(T=-1), ldn.LDN_ERR_INVALID_ARG),
    (dict(dk=96), ldn.LDN_ERR_UNSUPPORTED),
    (dict(chunk=128), ldn.LDN_ERR_UNSUPPORTED),
    (dict(T=0, q=None, erase=None, write=None, gate=None, out=None), ldn.LDN_OK),   # no state asked: nothing to do
    (dict(variant=7), ldn.LDN_ERR_INVALID_ARG),
    (dict(variant=ldn.LDN_VARIANT_PAIR, dk=128, dv=128), ldn.LDN_ERR_UNSUPPORTED),
    (dict(variant=ldn.LDN_VARIANT_TENSOR, dtype=0, dk=128), ldn.LDN_ERR_UNSUPPORTED),   # tensor cores: bf16
    (dict(variant=ldn.LDN_VARIANT_TENSOR, dk=128, erase=FAKE + 4), ldn.LDN_ERR_UNSUPPORTED),   # float4 gates
    (dict(variant=ldn.LDN_VARIANT_SPLIT, dk=64), ldn.LDN_ERR_UNSUPPORTED),
])
def test_chunk_gdn2_rejects_bad_arguments(lib, kw, want):
    assert _chunk_gdn2(**kw) == want


def _decode_gdn2(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, erase=FAKE, write=FAKE, gate=FAKE, S=FAKE, out=FAKE, B=1, H=1, dk=64,
             dv=64, dtype=0, stream=None)
    a.update(kw)
    return ldn.ldn_decode_step_gdn2(a["q"], a["k"], a["v"], a["erase"], a["write"], a["gate"], a["S"], a["out"],
                                    a["B"], a["H"], a["dk"], a["dv"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(S=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(erase=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(write=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(gate=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(S=FAKE + 4), ldn.LDN_ERR_INVALID_ARG),
    (dict(k=FAKE + 2), ldn.LDN_ERR_INVALID_ARG),
    (dict(write=FAKE + 2), ldn.LDN_ERR_INVALID_ARG),
    (dict(H=0), ldn.LDN_ERR_INVALID_ARG),
    (dict(dv=256), ldn.LDN_ERR_UNSUPPORTED),
])
def test_decode_gdn2_rejects_bad_arguments(lib, kw, want):
    assert _decode_gdn2(**kw) == want


def test_beta_gated_entry_points_reject_the_gdn2_mode(lib):
    assert _decode(mode=ldn.LDN_GDN2) == ldn.LDN_ERR_INVALID_ARG
    assert _chunk(mode=ldn.LDN_GDN2) == ldn.LDN_ERR_INVALID_ARG
    assert ldn.ldn_chunk_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, 1, 64, 1, 128, 128, 64,
                                     ldn.LDN_GDN2, 1, 0, None) == ldn.LDN_ERR_INVALID_ARG
    assert ldn.ldn_chunk_fwd_workspace_size(1, 64, 1, 128, 128, 64, ldn.LDN_GDN2, 1) == 0
    assert ldn.ldn_chunk_fwd_select(64, 64, 64, ldn.LDN_GDN2, 1) == -ldn.LDN_ERR_INVALID_ARG


def test_binding_without_library_fails_loudly(tmp_path, monkeypatch):
    import gated_delta_rule_chunkwise_gb300._native as nat
    monkeypatch.setattr(nat, "_lib", None)
    with pytest.raises(RuntimeError, match="libldn.so not found"):
        nat.load(str(tmp_path / "missing.so"))


def test_select_reports_kernel_family(lib):
    assert ldn.ldn_chunk_fwd_select(64, 64, 64, 0, ldn.LDN_F32) == ldn.LDN_VARIANT_SIMT
    assert ldn.ldn_chunk_fwd_select(128, 128, 64, 1, ldn.LDN_BF16) in (ldn.LDN_VARIANT_SIMT, ldn.LDN_VARIANT_TENSOR)
    assert ldn.ldn_chunk_fwd_select(96, 128, 64, 1, ldn.LDN_BF16) == -ldn.LDN_ERR_UNSUPPORTED
    assert ldn.ldn_chunk_fwd_select(128, 128, 32, 1, ldn.LDN_BF16) == -ldn.LDN_ERR_UNSUPPORTED
    assert ldn.ldn_chunk_fwd_select(128, 128, 64, 5, ldn.LDN_BF16) == -ldn.LDN_ERR_INVALID_ARG


def test_split_workspace_size_is_per_chunk_operands(lib):
    """[Q~;-W] 32 KiB + [P U';U'] 16 KiB per 64-column slice + K~ 16 KiB + e^{g_C} 512 B
    per (b, h, chunk); 0 where the split variant does not apply."""
    per = lambda dv: 32768 + (dv // 64) * 16384 + 16384 + 512
    assert ldn.ldn_chunk_fwd_workspace_size(4, 2048, 16, 128, 128, 64, 1, 1) == 4 * 16 * 32 * per(128)
    assert ldn.ldn_chunk_fwd_workspace_size(1, 65, 3, 128, 64, 64, 2, 1) == 3 * 2 * per(64)
    assert ldn.ldn_chunk_fwd_workspace_size(1, 64, 1, 128, 128, 64, 0, 0) == 0   # fp32: no tensor path
    assert ldn.ldn_chunk_fwd_workspace_size(1, 64, 1, 64, 128, 64, 1, 1) == 0    # dk = 64
    assert ldn.ldn_chunk_fwd_workspace_size(1, 0, 1, 128, 128, 64, 1, 1) == 0    # empty sequence
    assert ldn.ldn_chunk_fwd_workspace_size(1, 64, 1, 128, 128, 32, 1, 1) == 0   # chunk != 64


def test_split_segments_answers_without_a_device(lib):
    """With no device the SM count is unknown: the recurrence runs unsplit (1), the
    workspace is the operand images alone; 0 where the split variant does not apply,
    -LDN_ERR_* for rejected arguments."""
    big = (1 << 64) - 1
    assert ldn.ldn_chunk_fwd_split_segments(1, 65536, 16, 128, 128, 64, 1, 1, big) == 1
    assert ldn.ldn_chunk_fwd_workspace_size(1, 65536, 16, 128, 128, 64, 1, 1) == 16 * 1024 * (32768 + 2 * 16384 + 16896)
    assert ldn.ldn_chunk_fwd_split_segments(1, 64, 1, 128, 128, 64, 0, 0, big) == 0    # fp32: no split variant
    assert ldn.ldn_chunk_fwd_split_segments(1, 64, 1, 128, 128, 32, 1, 1, big) == -ldn.LDN_ERR_UNSUPPORTED
    assert ldn.ldn_chunk_fwd_split_segments(0, 64, 1, 128, 128, 64, 1, 1, big) == -ldn.LDN_ERR_INVALID_ARG
    assert ldn.ldn_chunk_fwd_split_segments(1, 64, 1, 128, 128, 64, 7, 1, big) == -ldn.LDN_ERR_INVALID_ARG


def test_split_without_workspace_is_rejected(lib):
    """The split variant needs a workspace: without one (or with too small a one) the
    call is rejected before anything is enqueued."""
    fake = 1 << 20   # never dereferenced: the checks come first
    args = [fake] * 5 + [0, fake, 0, 1, 64, 1, 128, 128, 64, 1, 1]
    assert ldn.ldn_chunk_fwd_variant(*args, ldn.LDN_VARIANT_SPLIT, 0) == ldn.LDN_ERR_INVALID_ARG
    assert ldn.ldn_chunk_fwd_ws(*args, ldn.LDN_VARIANT_SPLIT, 0, 0, 0) == ldn.LDN_ERR_INVALID_ARG
    assert ldn.ldn_chunk_fwd_ws(*args, ldn.LDN_VARIANT_SPLIT, 1 << 20, 16, 0) == ldn.LDN_ERR_INVALID_ARG
    assert ldn.ldn_chunk_fwd_ws(*args, ldn.LDN_VARIANT_SPLIT, (1 << 20) + 8, 1 << 30, 0) == ldn.LDN_ERR_INVALID_ARG


def _noalloc(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, beta=FAKE, gate=FAKE, S0=None, out=FAKE, S_final=None,
             B=1, T=64, H=1, dk=64, dv=64, chunk=64, mode=1, dtype=1, variant=0, stream=None)
    a.update(kw)
    return ldn.ldn_chunk_fwd_noalloc(a["q"], a["k"], a["v"], a["beta"], a["gate"], a["S0"], a["out"],
                                     a["S_final"], a["B"], a["T"], a["H"], a["dk"], a["dv"], a["chunk"],
                                     a["mode"], a["dtype"], a["variant"], a["stream"])


@pytest.mark.parametrize("variant", [ldn.LDN_VARIANT_AUTO, ldn.LDN_VARIANT_SPLIT])
@pytest.mark.parametrize("kw,want", [
    (dict(q=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(out=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(gate=None, mode=2), ldn.LDN_ERR_INVALID_ARG),
    (dict(q=FAKE + 4), ldn.LDN_ERR_INVALID_ARG),
    (dict(S_final=FAKE + 8), ldn.LDN_ERR_INVALID_ARG),
    (dict(beta=FAKE + 2), ldn.LDN_ERR_INVALID_ARG),
    (dict(mode=3), ldn.LDN_ERR_INVALID_ARG),
    (dict(dtype=2), ldn.LDN_ERR_INVALID_ARG),
    (dict(B=0), ldn.LDN_ERR_INVALID_ARG),
    (dict(T=-1), ldn.LDN_ERR_INVALID_ARG),
    (dict(dk=96), ldn.LDN_ERR_UNSUPPORTED),
    (dict(chunk=32), ldn.LDN_ERR_UNSUPPORTED),
])
def test_noalloc_rejects_bad_arguments(lib, kw, want, variant):
    """The no-allocation entry checks its arguments like the others, before it takes
    the scratch or enqueues anything."""
    assert _noalloc(variant=variant, **kw) == want


def test_noalloc_split_outside_the_tensor_kernels_is_unsupported(lib):
    assert _noalloc(variant=ldn.LDN_VARIANT_SPLIT, dk=64) == ldn.LDN_ERR_UNSUPPORTED   # dk = 64
    assert _noalloc(variant=ldn.LDN_VARIANT_SPLIT, dk=128, dtype=0) == ldn.LDN_ERR_UNSUPPORTED   # fp32
    assert _noalloc(variant=ldn.LDN_VARIANT_SPLIT, dk=128, mode=2, gate=FAKE + 4) == ldn.LDN_ERR_UNSUPPORTED
    assert _noalloc(variant=ldn.LDN_VARIANT_PRESOLVED, dk=64) == ldn.LDN_ERR_UNSUPPORTED
    assert _noalloc(variant=ldn.LDN_VARIANT_PRESOLVED, dk=128, dtype=0) == ldn.LDN_ERR_UNSUPPORTED
    assert _noalloc(variant=6) == ldn.LDN_ERR_INVALID_ARG


def test_presolved_variant_needs_a_workspace_and_the_tensor_kernels(lib):
    """The pre-solved variant runs through a workspace of 16 KiB per (b, h, chunk): without
    one (ldn_chunk_fwd_variant) or with too small a one it is refused before any CUDA call;
    outside the tensor-core sizes it is unsupported."""
    assert _chunk(variant=ldn.LDN_VARIANT_PRESOLVED, dk=128, dv=128) == ldn.LDN_ERR_INVALID_ARG   # no workspace
    big = 1 << 30
    for dk, dv, dtype in ((64, 64, 1), (128, 128, 0)):   # not the tensor-core sizes / fp32
        assert ldn.ldn_chunk_fwd_ws(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, 1, 64, 1, dk, dv, 64, 1, dtype,
                                    ldn.LDN_VARIANT_PRESOLVED, FAKE, big, None) == ldn.LDN_ERR_UNSUPPORTED
    B, T, H = 2, 200, 3
    need = B * H * ((T + 63) // 64) * 16384
    assert ldn.ldn_chunk_fwd_workspace_size(B, T, H, 128, 128, 64, 1, 1) >= need   # enough for either variant
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, B, T, H, 128, 128, 64, 1, 1,
            ldn.LDN_VARIANT_PRESOLVED)
    assert ldn.ldn_chunk_fwd_ws(*args, FAKE, need - 256, None) == ldn.LDN_ERR_INVALID_ARG      # too small
    assert ldn.ldn_chunk_fwd_ws(*args, FAKE + 16, need, None) == ldn.LDN_ERR_INVALID_ARG       # not 256-aligned


def test_pair_variant_outside_its_sizes_is_unsupported(lib):
    """The cluster-pair kernel takes DeltaNet / Gated DeltaNet, bf16, dk = dv = 128."""
    assert _chunk(variant=ldn.LDN_VARIANT_PAIR, dk=128, dv=128, mode=2) == ldn.LDN_ERR_UNSUPPORTED   # KDA
    assert _chunk(variant=ldn.LDN_VARIANT_PAIR, dk=128, dv=64) == ldn.LDN_ERR_UNSUPPORTED            # one slice
    assert _chunk(variant=ldn.LDN_VARIANT_PAIR, dk=64, dv=128) == ldn.LDN_ERR_UNSUPPORTED
    assert _chunk(variant=ldn.LDN_VARIANT_PAIR, dk=128, dv=128, dtype=0) == ldn.LDN_ERR_UNSUPPORTED  # fp32
    assert _chunk(variant=6) == ldn.LDN_ERR_INVALID_ARG


def _prologue(**kw):
    a = dict(q_in=FAKE, k_in=FAKE + (1 << 22), v_in=FAKE + (2 << 22), conv_q=FAKE + (3 << 22), conv_k=FAKE + (3 << 22),
             conv_v=FAKE + (3 << 22), width=4, beta_logit=FAKE + (4 << 22), gate_z=FAKE + (5 << 22),
             gate_a=FAKE + (6 << 22), gate_b=FAKE + (6 << 22), q=FAKE + (8 << 22), k=FAKE + (9 << 22),
             v=FAKE + (10 << 22), beta=FAKE + (11 << 22), gate=FAKE + (12 << 22), B=1, T=64, H=2, dk=128, dv=128,
             mode=1, dtype=1, eps=1e-6, stream=None)
    a.update(kw)
    return ldn.ldn_prologue(a["q_in"], a["k_in"], a["v_in"], a["conv_q"], a["conv_k"], a["conv_v"], a["width"],
                            a["beta_logit"], a["gate_z"], a["gate_a"], a["gate_b"], a["q"], a["k"], a["v"],
                            a["beta"], a["gate"], a["B"], a["T"], a["H"], a["dk"], a["dv"], a["mode"], a["dtype"],
                            a["eps"], a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(width=0), ldn.LDN_ERR_INVALID_ARG),
    (dict(width=9), ldn.LDN_ERR_UNSUPPORTED),
    (dict(eps=-1.0), ldn.LDN_ERR_INVALID_ARG),
    (dict(eps=float("nan")), ldn.LDN_ERR_INVALID_ARG),
    (dict(dk=96), ldn.LDN_ERR_UNSUPPORTED),
    (dict(mode=4), ldn.LDN_ERR_INVALID_ARG),
    (dict(q_in=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(conv_v=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(beta=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(gate_z=None), ldn.LDN_ERR_INVALID_ARG),          # GDN needs its gate inputs
    (dict(gate=None, mode=2), ldn.LDN_ERR_INVALID_ARG),
    (dict(q=FAKE + (8 << 22) + 8), ldn.LDN_ERR_INVALID_ARG),   # misaligned row
    (dict(gate_z=FAKE + (5 << 22) + 4, mode=2), ldn.LDN_ERR_INVALID_ARG),   # KDA gates move as float4
    (dict(q=FAKE), ldn.LDN_ERR_INVALID_ARG),                # output over its own input
    (dict(v=FAKE + (1 << 22) + 64), ldn.LDN_ERR_INVALID_ARG),   # output inside another input
    (dict(k=FAKE + (8 << 22) + 1024), ldn.LDN_ERR_INVALID_ARG),  # outputs overlapping each other
    (dict(B=0), ldn.LDN_ERR_INVALID_ARG),
])
def test_prologue_rejects_bad_arguments(lib, kw, want):
    assert _prologue(**kw) == want


def test_prologue_zero_length_and_deltanet_gates_need_no_pointers(lib):
    assert _prologue(T=0, q_in=None, q=None) == ldn.LDN_OK   # nothing to do, nothing launched
    # DeltaNet ignores the gate pointers: NULL gate inputs pass the checks (the rejection
    # tested here is the misaligned q, which comes after them)
    assert _prologue(mode=0, gate_z=None, gate_a=None, gate_b=None, gate=None, q=FAKE + (8 << 22) + 8) == \
        ldn.LDN_ERR_INVALID_ARG


def _rms(**kw):
    a = dict(o=FAKE, g=FAKE + (1 << 22), weight=FAKE + (2 << 22), y=FAKE + (3 << 22), B=1, T=64, H=2, dv=128,
             dtype=1, eps=1e-6, stream=None)
    a.update(kw)
    return ldn.ldn_rmsnorm_gated(a["o"], a["g"], a["weight"], a["y"], a["B"], a["T"], a["H"], a["dv"], a["dtype"],
                                 a["eps"], a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(y=FAKE + (1 << 22)), ldn.LDN_ERR_INVALID_ARG),     # y over the gate
    (dict(y=FAKE + 512), ldn.LDN_ERR_INVALID_ARG),           # y partly over o
    (dict(o=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(o=FAKE + 8), ldn.LDN_ERR_INVALID_ARG),
    (dict(dv=96), ldn.LDN_ERR_UNSUPPORTED),
    (dict(dtype=3), ldn.LDN_ERR_INVALID_ARG),
    (dict(eps=-0.5), ldn.LDN_ERR_INVALID_ARG),
    (dict(T=-1), ldn.LDN_ERR_INVALID_ARG),
])
def test_rmsnorm_gated_rejects_bad_arguments(lib, kw, want):
    assert _rms(**kw) == want


def test_select_answers_for_gdn2(lib):
    """The kernel family ldn_chunk_fwd_gdn2 runs: tensor-core families for bf16 with
    dk = 128, the CUDA-core kernel otherwise; never the pair kernel."""
    big = (1 << 64) - 1
    assert ldn.ldn_chunk_fwd_select_ws(1, 64, 1, 64, 64, 64, ldn.LDN_GDN2, 1, big) == ldn.LDN_VARIANT_SIMT
    assert ldn.ldn_chunk_fwd_select_ws(1, 64, 1, 128, 128, 64, ldn.LDN_GDN2, 0, big) == ldn.LDN_VARIANT_SIMT
    fam = ldn.ldn_chunk_fwd_select_ws(8, 4096, 16, 128, 128, 64, ldn.LDN_GDN2, 1, big)
    assert fam in (ldn.LDN_VARIANT_TENSOR, ldn.LDN_VARIANT_SPLIT)


def _bwd(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, beta=FAKE, gate=FAKE, S0=None, dout=FAKE, dsf=None, dq=FAKE, dk=FAKE,
             dv=FAKE, dbeta=FAKE, dgate=FAKE, dS0=FAKE, B=1, T=64, H=1, dkd=64, dvd=64, mode=1, dtype=1,
             ws=FAKE, wsb=1 << 40, stream=None)
    a.update(kw)
    return ldn.ldn_backward(a["q"], a["k"], a["v"], a["beta"], a["gate"], a["S0"], a["dout"], a["dsf"], a["dq"],
                            a["dk"], a["dv"], a["dbeta"], a["dgate"], a["dS0"], a["B"], a["T"], a["H"], a["dkd"],
                            a["dvd"], a["mode"], a["dtype"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(dout=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(dS0=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(dgate=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(gate=None, mode=2), ldn.LDN_ERR_INVALID_ARG),
    (dict(ws=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(wsb=1024), ldn.LDN_ERR_INVALID_ARG),              # workspace too small
    (dict(ws=FAKE + 8), ldn.LDN_ERR_INVALID_ARG),
    (dict(q=FAKE + 1), ldn.LDN_ERR_INVALID_ARG),
    (dict(dbeta=FAKE + 2), ldn.LDN_ERR_INVALID_ARG),
    (dict(mode=ldn.LDN_GDN2), ldn.LDN_ERR_INVALID_ARG),
    (dict(dtype=3), ldn.LDN_ERR_INVALID_ARG),
    (dict(B=0), ldn.LDN_ERR_INVALID_ARG),
    (dict(dkd=32), ldn.LDN_ERR_UNSUPPORTED),
    (dict(mode=0, gate=None, dgate=None, q=None), ldn.LDN_ERR_INVALID_ARG),
])
def test_backward_rejects_bad_arguments(lib, kw, want):
    assert _bwd(**kw) == want


def test_chunkwise_backward_wants_aligned_tensors_and_its_workspace(lib):
    """bf16 Gated DeltaNet at dk = dv = 128 takes the chunkwise backward: 16-byte aligned
    tensors, a 256-byte aligned workspace of its size; anything less is refused before any
    CUDA call."""
    need = ldn.ldn_backward_workspace_size(1, 64, 1, 128, 128, 1, ldn.LDN_BF16)
    base = dict(dkd=128, dvd=128, dtype=ldn.LDN_BF16, wsb=need)
    assert _bwd(q=FAKE + 2, **base) == ldn.LDN_ERR_INVALID_ARG
    assert _bwd(dk=FAKE + 4, **base) == ldn.LDN_ERR_INVALID_ARG
    assert _bwd(ws=FAKE + 16, **base) == ldn.LDN_ERR_INVALID_ARG
    assert _bwd(**dict(base, wsb=need - 1)) == ldn.LDN_ERR_INVALID_ARG


def test_backward_workspace_size(lib):
    """Recurrent form: state copies (every eighth state of every column) plus
    per-32-column partial sums of dq, dk, the gate gradient and dbeta.  Chunkwise form
    (bf16 DeltaNet / GDN, dk = dv = 128), per chunk: the solve X (16 KiB), the state
    entering and the state gradient leaving it and the chain's two terms M and Bc (fp16
    images of 128 x 136), P (64 x 72) and -W (64 x 136); and the forward's output."""
    B, T, H, dk, dv = 2, 70, 3, 128, 64
    n, nsub, sl = B * T * H, (T + 7) // 8, dv // 32
    for dtype in (ldn.LDN_F32, ldn.LDN_BF16):
        for mode, gw in ((0, 0), (1, 1), (2, dk)):
            want = 4 * (B * H * dv * nsub * dk + sl * n * (2 * dk + gw + 1))
            assert ldn.ldn_backward_workspace_size(B, T, H, dk, dv, mode, dtype) == want
    nch = (T + 63) // 64
    chunked = B * H * nch * (16384 + 4 * 128 * 136 * 2 + 64 * 72 * 2 + 64 * 136 * 2) + n * 128 * 2
    for mode in (0, 1):
        assert ldn.ldn_backward_workspace_size(B, T, H, 128, 128, mode, ldn.LDN_BF16) == chunked
    n, nsub, sl = B * T * H, (T + 7) // 8, 128 // 32
    assert ldn.ldn_backward_workspace_size(B, T, H, 128, 128, 2, ldn.LDN_BF16) == \
        4 * (B * H * 128 * nsub * 128 + sl * n * (2 * 128 + 128 + 1))   # KDA: recurrent
    assert ldn.ldn_backward_workspace_size(B, T, H, 96, dv, 1, 1) == 0
    assert ldn.ldn_backward_workspace_size(B, T, H, dk, dv, ldn.LDN_GDN2, 1) == 0


def _rla(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, beta=FAKE, gamma=FAKE, gate=FAKE, clip=1.0, S0=None, R0=None, out=FAKE,
             sf=None, rf=None, B=1, T=64, H=1, dk=64, dv=64, delta=1, dtype=1, stream=None)
    a.update(kw)
    return ldn.ldn_rla_fwd(a["q"], a["k"], a["v"], a["beta"], a["gamma"], a["gate"], a["clip"], a["S0"], a["R0"],
                           a["out"], a["sf"], a["rf"], a["B"], a["T"], a["H"], a["dk"], a["dv"], a["delta"],
                           a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(gamma=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(gate=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(clip=0.0), ldn.LDN_ERR_INVALID_ARG),
    (dict(clip=-1.0), ldn.LDN_ERR_INVALID_ARG),
    (dict(clip=float("nan")), ldn.LDN_ERR_INVALID_ARG),
    (dict(delta=2), ldn.LDN_ERR_INVALID_ARG),
    (dict(out=FAKE + 4), ldn.LDN_ERR_INVALID_ARG),
    (dict(R0=FAKE + 4), ldn.LDN_ERR_INVALID_ARG),
    (dict(gamma=FAKE + 2), ldn.LDN_ERR_INVALID_ARG),
    (dict(dk=96), ldn.LDN_ERR_UNSUPPORTED),
    (dict(dtype=4), ldn.LDN_ERR_INVALID_ARG),
    (dict(T=0, q=None, out=None), ldn.LDN_OK),              # no state asked: nothing to do
])
def test_rla_rejects_bad_arguments(lib, kw, want):
    assert _rla(**kw) == want


def test_rla_workspace_size(lib):
    """Chunk form (bf16, dk = dv = 128): Residual DeltaNet's two solves, 16 KiB per
    (b, h, chunk) each; Residual Linear Attention and the recurrent shapes need none."""
    B, T, H = 2, 130, 3
    nch = (T + 63) // 64
    assert ldn.ldn_rla_fwd_workspace_size(B, T, H, 128, 128, 1, ldn.LDN_BF16) == 2 * B * H * nch * 16384
    assert ldn.ldn_rla_fwd_workspace_size(B, T, H, 128, 128, 0, ldn.LDN_BF16) == 0
    assert ldn.ldn_rla_fwd_workspace_size(B, T, H, 128, 128, 1, ldn.LDN_F32) == 0
    assert ldn.ldn_rla_fwd_workspace_size(B, T, H, 64, 128, 1, ldn.LDN_BF16) == 0
    assert ldn.ldn_rla_fwd_workspace_size(B, 0, H, 128, 128, 1, ldn.LDN_BF16) == 0
    assert ldn.ldn_rla_fwd_workspace_size(B, T, H, 128, 128, 2, ldn.LDN_BF16) == 0


def test_rla_ws_wants_an_aligned_workspace(lib):
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, None, None, FAKE, None, None, 1, 64, 1, 128, 128, 1,
            ldn.LDN_BF16)
    assert ldn.ldn_rla_fwd_ws(*args, FAKE + 16, 1 << 20, None) == ldn.LDN_ERR_INVALID_ARG
    assert ldn.ldn_rla_fwd_ws(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, None, None, FAKE, None, None, 1, 64, 1, 128,
                              128, 1, ldn.LDN_BF16, FAKE, 1 << 20, None) == ldn.LDN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(S=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(S=FAKE + 8), ldn.LDN_ERR_INVALID_ARG),
    (dict(gate=None), ldn.LDN_ERR_INVALID_ARG),
    (dict(n=-1), ldn.LDN_ERR_INVALID_ARG),
    (dict(mode=ldn.LDN_GDN2), ldn.LDN_ERR_UNSUPPORTED),
    (dict(dk=96), ldn.LDN_ERR_UNSUPPORTED),
    (dict(n=0, q=None, v=None, out=None), ldn.LDN_OK),   # nothing to do
])
def test_decode_steps_rejects_bad_arguments(lib, kw, want):
    a = dict(q=FAKE, k=FAKE, v=FAKE, beta=FAKE, gate=FAKE, S=FAKE, out=FAKE, n=4, B=1, H=1, dk=64, dv=64,
             mode=ldn.LDN_GDN, dtype=ldn.LDN_F32)
    a.update(kw)
    assert ldn.ldn_decode_steps(a["q"], a["k"], a["v"], a["beta"], a["gate"], a["S"], a["out"], a["n"], a["B"],
                                a["H"], a["dk"], a["dv"], a["mode"], a["dtype"], None) == want
