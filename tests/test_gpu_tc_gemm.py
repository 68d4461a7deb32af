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
    lib.tc_selftest_gemm.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2
    lib.tc_selftest_gemm.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 1024), (200, 256, 2048), (1000, 1024, 512)])
def test_tc_gemm_matches_torch(M, N, K):
    lib = selftest_lib()
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N + K)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = (torch.randn(K, N, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    D = torch.full((M, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.tc_selftest_gemm(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, status.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = A.float() @ B.float()
    assert torch.isfinite(D).all()
    err = (D - ref).abs().max().item()
    assert err <= 1e-3 * ref.abs().max().item() + 1e-4, err
