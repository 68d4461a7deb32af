"""The layer stack (flint_moe_stack_*: one launch of decode_stack for all layers) against
successive single-layer calls on the same weights: the results, and
every layer's routing, must be bitwise equal (the stack kernel runs each layer's steps with the
same arithmetic; the single-layer path is itself checked against the oracle in
test_gpu_parity.py and test_gpu_stack.py)."""
import pytest
import torch

import synth
import sparse_moe_layer_15_b300 as fm
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
EPS = 1e-6
N_LAYERS = 3


@pytest.fixture(scope="module")
def layer_weights():
    return [synth.flint_weights(seed=100 + l, device=DEV) for l in range(N_LAYERS)]


def per_layer(weights, x0, flags, T):
    ws = torch.empty(fm.workspace_bytes(T, flags, EPS), dtype=torch.uint8, device=DEV)
    layers = [fm.FlintMoE(w, max_tokens=T, flags=flags, rms_eps=EPS, workspace=ws) for w in weights]
    x = x0.clone()
    idx = torch.full((len(weights), T, fm.TOP_K), -1, dtype=torch.int32, device=DEV)
    gw = torch.zeros((len(weights), T, fm.TOP_K), dtype=torch.float32, device=DEV)
    for l, lay in enumerate(layers):
        lay.forward(x, y=x, topk_idx=idx[l], topk_w=gw[l])
    torch.cuda.synchronize()
    for lay in layers:
        assert lay.poll_device_status() == 0
        lay.close()
    return x, idx, gw


@pytest.mark.parametrize("T", [1, 3, 16, 64, 256])
def test_stack_equals_layer_calls_prenorm_residual(layer_weights, T):
    flags = fm.FLAG_PRE_RMSNORM | fm.FLAG_RESIDUAL
    x0 = synth.torch_normal_bf16((T, fm.HIDDEN), 4000 + T, synth.TAG_X, 1.0, device=DEV)
    ref, ref_idx, ref_gw = per_layer(layer_weights, x0, flags, T)
    stack = fm.FlintMoEStack(layer_weights, max_tokens=256, flags=flags, rms_eps=EPS)
    idx = torch.full((N_LAYERS, T, fm.TOP_K), -1, dtype=torch.int32, device=DEV)
    gw = torch.zeros((N_LAYERS, T, fm.TOP_K), dtype=torch.float32, device=DEV)
    x = x0.clone()
    stack.forward(x, topk_idx=idx, topk_w=gw)
    torch.cuda.synchronize()
    assert stack.poll_device_status() == 0
    assert torch.equal(idx, ref_idx)
    assert torch.equal(gw.view(torch.int32), ref_gw.view(torch.int32))
    assert torch.equal(x.view(torch.int16), ref.view(torch.int16))
    # a second call on the same handle (counters back at zero) repeats the result
    x2 = x0.clone()
    stack.forward(x2)
    torch.cuda.synchronize()
    assert torch.equal(x2.view(torch.int16), ref.view(torch.int16))
    stack.close()


@pytest.mark.parametrize("T", [1, 64])
def test_stack_with_a_router_bias_per_layer(T):
    # each layer has its own N(0, 0.5) router bias (the prefill workload's kind): the stack must
    # take layer l's bias from its table, so the routing and outputs equal the layer calls', and
    # the last layer meets the parity rule against the oracle on the stack's own input to it
    flags = fm.FLAG_PRE_RMSNORM | fm.FLAG_RESIDUAL
    weights = [synth.flint_weights(seed=100 + l, device=DEV, bias="normal", bias_seed=300 + l)
               for l in range(N_LAYERS)]
    x0 = synth.torch_normal_bf16((T, fm.HIDDEN), 4300 + T, synth.TAG_X, 1.0, device=DEV)
    ref, ref_idx, ref_gw = per_layer(weights, x0, flags, T)
    prefix, _, _ = per_layer(weights[:-1], x0, flags, T)
    stack = fm.FlintMoEStack(weights, max_tokens=T, flags=flags, rms_eps=EPS)
    idx = torch.full((N_LAYERS, T, fm.TOP_K), -1, dtype=torch.int32, device=DEV)
    gw = torch.zeros((N_LAYERS, T, fm.TOP_K), dtype=torch.float32, device=DEV)
    x = x0.clone()
    stack.forward(x, topk_idx=idx, topk_w=gw)
    torch.cuda.synchronize()
    assert stack.poll_device_status() == 0
    assert torch.equal(idx, ref_idx)
    assert torch.equal(x.view(torch.int16), ref.view(torch.int16))
    stack.close()
    rep = parity.compare(parity.oracle_reference(weights[-1], prefix, range(T), eps=EPS, residual=True), x,
                         idx[-1], gw[-1])
    assert rep["ok"], rep


@pytest.mark.parametrize("T", [16, 64, 256])
def test_stack_equals_layer_calls_without_norm_or_residual(layer_weights, T):
    # no pre-norm copy: the router and gate/up read x directly, and the combine overwrites it
    x0 = synth.torch_normal_bf16((T, fm.HIDDEN), 4100, synth.TAG_X, 1.0, device=DEV)
    ref, _, _ = per_layer(layer_weights[:2], x0, 0, T)
    stack = fm.FlintMoEStack(layer_weights[:2], max_tokens=T, flags=0)
    x = x0.clone()
    stack.forward(x)
    torch.cuda.synchronize()
    assert stack.poll_device_status() == 0
    assert torch.equal(x.view(torch.int16), ref.view(torch.int16))
    stack.close()


def test_stack_rejects_too_many_tokens(layer_weights):
    stack = fm.FlintMoEStack(layer_weights[:1], max_tokens=8)
    x = torch.zeros((9, fm.HIDDEN), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fm.FlintMoEError) as e:
        stack.forward(x)
    assert e.value.code == 1
    stack.close()
