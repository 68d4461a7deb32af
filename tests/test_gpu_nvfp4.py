"""The Flint MoE layer on NVFP4 expert weights (flint_moe_create_nvfp4, decode sizes) against the
fp64 oracle of the dequantised layer, through the C ABI: the decode sweep T = 1..64 (routing and
outputs on every token, the parity rule of tests/parity.py), pre-norm + residual in place,
bitwise run-to-run determinism, route/forward agreement, and the size limit."""
import numpy as np
import pytest
import torch

import synth
import sparse_moe_layer_15_b300 as fm
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def wq():
    w = synth.flint_weights(seed=0, device=DEV)
    q = synth.nvfp4_weights(w)
    return w, q


@pytest.fixture(scope="module")
def layer(wq):
    w, q = wq
    lay = fm.FlintMoE.nvfp4(w["w_router"], q, max_tokens=64)
    yield lay
    lay.close()


def run(layer, x):
    T = x.shape[0]
    idx = torch.full((T, fm.TOP_K), -1, dtype=torch.int32, device=DEV)
    gw = torch.zeros((T, fm.TOP_K), dtype=torch.float32, device=DEV)
    y = layer.forward(x, topk_idx=idx, topk_w=gw)
    torch.cuda.synchronize()
    assert layer.poll_device_status() == 0
    return y, idx, gw


@pytest.mark.parametrize("T", [1, 2, 4, 8, 16, 32, 64])
def test_nvfp4_decode_sweep_matches_oracle(wq, layer, T):
    w, q = wq
    x = synth.torch_normal_bf16((T, fm.HIDDEN), 1000 + T, synth.TAG_X, 1.0, device=DEV)
    y, idx, gw = run(layer, x)
    ref = parity.oracle_reference_nvfp4(w, q, x, range(T))
    rep = parity.compare(ref, y, idx, gw)
    assert rep["ok"], rep
    y2, _, _ = run(layer, x)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    idx3, gw3, counts = layer.route(x)
    torch.cuda.synchronize()
    assert torch.equal(idx3, idx) and torch.equal(gw3, gw)
    assert np.array_equal(counts.cpu().numpy(), np.bincount(idx.cpu().numpy().reshape(-1), minlength=256))


def test_nvfp4_prenorm_residual_in_place(wq):
    w, q = wq
    flags = fm.FLAG_PRE_RMSNORM | fm.FLAG_RESIDUAL
    lay = fm.FlintMoE.nvfp4(w["w_router"], q, max_tokens=16, flags=flags, rms_eps=1e-6)
    x = synth.torch_normal_bf16((16, fm.HIDDEN), 77, synth.TAG_X, 1.0, device=DEV)
    y, idx, gw = run(lay, x)
    ref = parity.oracle_reference_nvfp4(w, q, x, range(16), eps=1e-6, residual=True)
    assert parity.compare(ref, y, idx, gw)["ok"]
    x2 = x.clone()
    lay.forward(x2, y=x2)
    torch.cuda.synchronize()
    assert torch.equal(x2.view(torch.int16), y.view(torch.int16))
    lay.close()


def test_nvfp4_rejects_prefill_sizes(wq):
    w, q = wq
    with pytest.raises(fm.FlintMoEError) as e:
        fm.FlintMoE.nvfp4(w["w_router"], q, max_tokens=65)
    assert e.value.code == 2
