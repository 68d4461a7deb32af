"""The tensor-core engine (tcgen05 + TMEM + TMA, 128-byte swizzle) on a dense bf16 GEMM
against torch.matmul: pins its smem/instruction descriptors, K stepping, B box layout,
double-buffered accumulators and epilogue row mapping before any MoE kernel relies on it."""
import ctypes
import os

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def selftest_lib():
    path = os.path.join(HERE, "libtc_selftest.so")
    if not os.path.exists(path):
        pytest.fail("tests/libtc_selftest.so is missing: run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    lib.tc_selftest_gemm.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 2
    lib.tc_selftest_gemm.restype = ctypes.c_int
    lib.tc_selftest_gemm_ex.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 6 + [ctypes.c_void_p] * 2
    lib.tc_selftest_gemm_ex.restype = ctypes.c_int
    return lib


ROWS, COLUMNS = 0, 1


@pytest.mark.parametrize("mode", [ROWS, COLUMNS])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 1024), (200, 256, 2048), (1000, 1024, 512),
                                   (16, 256, 128), (131, 256, 256)])
def test_tc_gemm_matches_torch(M, N, K, mode):
    lib = selftest_lib()
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N + K)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = (torch.randn(K, N, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    D = torch.full((M, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.tc_selftest_gemm(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, mode, status.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = A.float() @ B.float()
    assert torch.isfinite(D).all()
    err = (D - ref).abs().max().item()
    assert err <= 1e-3 * ref.abs().max().item() + 1e-4, err


@pytest.mark.parametrize("rows_per_tile", [16, 48, 112, 256])
def test_tc_gemm_columns_row_groups(rows_per_tile):
    """COLUMNS tiles whose row groups are smaller than the 256-row maximum: the MMA's N takes
    every multiple of 16 the grouped GEMMs use, with ragged groups at the end."""
    lib = selftest_lib()
    M, N, K = 1000, 512, 2048
    g = torch.Generator(device="cuda").manual_seed(rows_per_tile)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = (torch.randn(K, N, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    D = torch.full((M, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.tc_selftest_gemm_ex(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, COLUMNS, rows_per_tile, 0,
                                 status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = A.float() @ B.float()
    assert torch.isfinite(D).all()
    assert (D - ref).abs().max().item() <= 1e-3 * ref.abs().max().item() + 1e-4
