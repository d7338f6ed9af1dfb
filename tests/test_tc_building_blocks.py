"""The tensor-core building blocks, pinned on tiny matrices (GPU).

ldn_diag_tma_sw128 checks that a TMA load with 128-byte swizzle places element
(row, col) of a 64-column box at byte 128*row + 16*((col/8) XOR (row%8)) +
2*(col%8) of the tile (the SWIZZLE_128B pattern of the PTX ISA), and that
rows past the end read as zero.  ldn_diag_umma checks one tcgen05.mma chain
(bf16 in, fp32 out) for K-major and MN-major operands against A @ B^T and
records which TMEM lane holds which accumulator row: M = 128 uses lane = row,
M = 64 uses lanes 0-15 of each 32-lane quarter (row r -> 32*(r//16) + r%16).
"""
import numpy as np
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from tests import _diag

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def sw128_offset(row, col):
    return row * 128 + (((col >> 3) ^ (row & 7)) * 16) + (col & 7) * 2


@pytest.mark.parametrize("row0,col0", [(0, 0), (40, 64), (64, 0)])
def test_tma_swizzle_128b_placement(row0, col0):
    import torch
    rows, cols = 100, 128
    src = torch.arange(rows * cols, dtype=torch.int32).remainder(30000).to(torch.int16).view(torch.bfloat16)
    src = src.reshape(rows, cols).cuda().contiguous()
    dst = torch.zeros(8192, dtype=torch.uint8, device="cuda")
    assert _diag.load().ldn_diag_tma_sw128(src.data_ptr(), dst.data_ptr(), rows, cols, row0, col0, _stream()) == ldn.LDN_OK
    assert _diag.status() == ldn.LDN_OK
    got = dst.cpu().numpy().view(np.uint16)
    s = src.view(torch.int16).cpu().numpy().view(np.uint16)
    want = np.zeros(4096, np.uint16)
    for r in range(64):
        for c in range(64):
            if row0 + r < rows:
                want[sw128_offset(r, c) // 2] = s[row0 + r, col0 + c]
    np.testing.assert_array_equal(got, want)


CASES = [  # M, N, K, a_mn, b_mn, fmt (0 fp16, 1 bf16)
    (128, 64, 128, 0, 0, 1), (128, 128, 64, 0, 1, 1), (128, 64, 64, 1, 1, 1), (128, 128, 128, 1, 0, 1),
    (128, 256, 64, 0, 1, 1), (64, 128, 64, 0, 1, 1), (64, 64, 128, 0, 0, 1), (64, 128, 64, 1, 1, 1),
    (128, 16, 32, 0, 0, 1),
    (128, 64, 128, 0, 0, 0), (128, 128, 64, 0, 1, 0), (128, 64, 64, 1, 1, 0), (128, 128, 128, 1, 0, 0),
]


@pytest.mark.parametrize("M,N,K,a_mn,b_mn,fmt", CASES)
def test_umma_f16kind_layouts(M, N, K, a_mn, b_mn, fmt):
    import torch
    g = torch.Generator().manual_seed(M * 1000 + N + K + 7 * a_mn + 13 * b_mn + 17 * fmt)
    dt = torch.bfloat16 if fmt == 1 else torch.float16
    A = torch.randn(M, K, generator=g).to(dt)
    B = torch.randn(N, K, generator=g).to(dt)
    D = torch.empty(128, N, dtype=torch.float32, device="cuda")
    Ad, Bd = A.cuda(), B.cuda()
    st = _diag.load().ldn_diag_umma(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, a_mn, b_mn, fmt, _stream())
    assert st == ldn.LDN_OK
    assert _diag.status() == ldn.LDN_OK
    got = D.cpu().numpy().astype(np.float64)
    ref = A.double().numpy() @ B.double().numpy().T
    lane_of = (lambda r: r) if M == 128 else (lambda r: 32 * (r // 16) + r % 16)
    # locate every reference row among the lanes, to report the layout on failure
    found = {}
    for r in range(M):
        d = np.max(np.abs(got - ref[r][None, :]), axis=1)
        found[r] = int(np.argmin(d)) if np.min(d) < 1e-3 * (1 + np.abs(ref[r]).max()) else None
    expected = {r: lane_of(r) for r in range(M)}
    assert found == expected, f"row -> lane found {found}"
    used = {lane_of(r) for r in range(M)}
    for lane in range(128):
        if lane not in used and M == 128:
            raise AssertionError("M=128 must use every lane")


TMEM_A_CASES = [  # N, K, b_mn, fmt
    (64, 128, 1, 0), (128, 64, 0, 0), (64, 64, 1, 1), (256, 128, 0, 1), (16, 32, 0, 0),
]


@pytest.mark.parametrize("N,K,b_mn,fmt", TMEM_A_CASES)
def test_umma_a_operand_in_tmem(N, K, b_mn, fmt):
    """A (M = 128) read from TMEM as 16-bit pairs: element k of row r in lane r,
    column k // 2, low half for even k.  On failure, say whether the pairs were
    read the other way round."""
    import torch
    g = torch.Generator().manual_seed(N * 7 + K + 3 * b_mn + 11 * fmt)
    dt = torch.bfloat16 if fmt == 1 else torch.float16
    A = torch.randn(128, K, generator=g).to(dt)
    B = torch.randn(N, K, generator=g).to(dt)
    D = torch.empty(128, N, dtype=torch.float32, device="cuda")
    Ad, Bd = A.cuda(), B.cuda()
    assert _diag.load().ldn_diag_umma_tmem_a(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), N, K, b_mn, fmt, _stream()) == ldn.LDN_OK
    assert _diag.status() == ldn.LDN_OK
    got = D.cpu().numpy().astype(np.float64)
    a, b = A.double().numpy(), B.double().numpy()
    ref = a @ b.T
    swapped = a.reshape(128, K // 2, 2)[:, :, ::-1].reshape(128, K) @ b.T
    err = np.max(np.abs(got - ref)) / (1 + np.abs(ref).max())
    err_sw = np.max(np.abs(got - swapped)) / (1 + np.abs(ref).max())
    assert err < 1e-5, f"max rel err {err:.3g} (pair-swapped reading: {err_sw:.3g})"
