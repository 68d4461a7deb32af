"""The dense SwiGLU MLP layers (flint_dense_*, width 6144) against the fp64 oracle, through the
C ABI: the decode-size kernel (T <= 256, the shared-expert steps at this width, whose down
inputs are staged in windows of 2048) and the tensor-core GEMMs (T > 256), every token checked,
with ragged sizes, pre-norm + residual in place and bitwise run-to-run determinism.  Tolerance:
the layer's, max |y - y_ref| <= 2e-2 max |y_ref| and relative L1 <= 5e-3."""
import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_moe_layer_15_b300 as fm
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
EPS = 1e-6


@pytest.fixture(scope="module")
def wd():
    return synth.dense_weights(seed=7, device=DEV)


@pytest.fixture(scope="module")
def host_w(wd):
    return {k: parity.to_np_bf16(v) for k, v in wd.items()}


def reference(host_w, x, eps=None, residual=False):
    x64 = oracle.bf16_to_f64(parity.to_np_bf16(x))
    xin = x64 if eps is None else oracle.prenorm_input(x64, eps)
    y = oracle.dense(xin, host_w["w_gate"], host_w["w_up"], host_w["w_down"], nthreads=parity.ORACLE_THREADS)
    return x64 + y if residual else y


def check(y, ref):
    g = oracle.bf16_to_f64(parity.to_np_bf16(y))
    d = np.abs(g - ref)
    max_rel = d.max() / np.abs(ref).max()
    rel_l1 = d.sum() / np.abs(ref).sum()
    assert max_rel <= parity.MAX_ABS_REL and rel_l1 <= parity.REL_L1, (max_rel, rel_l1)


@pytest.mark.parametrize("T", [1, 3, 16, 64, 65, 256, 257, 1000])
def test_dense_layer_all_tokens(wd, host_w, T):
    layer = fm.FlintDense(wd, max_tokens=T)
    x = synth.torch_normal_bf16((T, fm.HIDDEN), 600 + T, synth.TAG_X, 1.0, device=DEV)
    y = layer.forward(x)
    torch.cuda.synchronize()
    assert layer.poll_device_status() == 0
    check(y, reference(host_w, x))
    y2 = layer.forward(x)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    layer.close()


def test_dense_layer_full_prefill_size_sampled(wd, host_w):
    # the bench's dense workload at T = 8192 (weights seed 7, x seed 600 + T as there): every 16th
    # token, which samples every 256-row group of the GEMM tiles
    T = 8192
    layer = fm.FlintDense(wd, max_tokens=T)
    x = synth.torch_normal_bf16((T, fm.HIDDEN), 600 + T, synth.TAG_X, 1.0, device=DEV)
    y = layer.forward(x)
    torch.cuda.synchronize()
    assert layer.poll_device_status() == 0
    rows = torch.arange(0, T, 16, device=DEV)
    check(y[rows], reference(host_w, x[rows]))
    layer.close()


@pytest.mark.parametrize("T", [4, 512])
def test_dense_layer_prenorm_residual_in_place(wd, host_w, T):
    flags = fm.FLAG_PRE_RMSNORM | fm.FLAG_RESIDUAL
    layer = fm.FlintDense(wd, max_tokens=T, flags=flags, rms_eps=EPS)
    x = synth.torch_normal_bf16((T, fm.HIDDEN), 700 + T, synth.TAG_X, 1.0, device=DEV)
    ref = reference(host_w, x, eps=EPS, residual=True)
    y = layer.forward(x)
    x2 = x.clone()
    layer.forward(x2, y=x2)
    torch.cuda.synchronize()
    assert layer.poll_device_status() == 0
    check(y, ref)
    assert torch.equal(x2.view(torch.int16), y.view(torch.int16))
    layer.close()


def test_dense_layer_rejects_other_widths(wd):
    import ctypes
    L = fm.load_library()
    cfg = fm._DenseConfig(fm.HIDDEN, 4096, 16, 0, 1e-6)
    n = ctypes.c_size_t(0)
    assert L.flint_dense_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)) == 2  # unsupported
