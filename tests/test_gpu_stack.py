"""The 47-layer stack workload (T = 256 tokens, x <- x + MoE_l(RMSNorm(x)), eps 1e-6, weights
seed 100 + l, about 76 GB resident), checked layer by layer with teacher forcing: the oracle's
layer l takes the GPU's bf16 input to layer l, on sampled layers 0, 23 and 46 -- routing and
outputs on all 256 tokens.  A routing flip in an early layer would make
an end-to-end comparison meaningless, so the end-to-end output is only checked to be finite and
bitwise deterministic, and the stack handle (one launch for the 47 layers) must reproduce the per-layer
results bitwise."""
import pytest
import torch

import synth
import sparse_moe_layer_15_b300 as fm
from sparse_moe_layer_15_b300 import accounting as acc
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
EPS = 1e-6
CHECKED = (0, 23, 46)


def test_stack_47_layers_teacher_forced_parity():
    L, T = acc.N_MOE_LAYERS, 256
    flags = fm.FLAG_PRE_RMSNORM | fm.FLAG_RESIDUAL
    ws = torch.empty(fm.workspace_bytes(T, flags, EPS), dtype=torch.uint8, device=DEV)
    weights = [synth.flint_weights(seed=100 + l, device=DEV) for l in range(L)]
    layers = [fm.FlintMoE(weights[l], max_tokens=T, flags=flags, rms_eps=EPS, workspace=ws) for l in range(L)]
    x0 = synth.torch_normal_bf16((T, fm.HIDDEN), 4, synth.TAG_X, 1.0, device=DEV)

    def run(keep):
        x = x0.clone()
        seen = {}
        for l, lay in enumerate(layers):
            if l in keep:
                idx = torch.full((T, fm.TOP_K), -1, dtype=torch.int32, device=DEV)
                gw = torch.zeros((T, fm.TOP_K), dtype=torch.float32, device=DEV)
                xin = x.clone()
                lay.forward(x, y=x, topk_idx=idx, topk_w=gw)
                seen[l] = (xin, x.clone(), idx, gw)
            else:
                lay.forward(x, y=x)
        torch.cuda.synchronize()
        for lay in layers:
            assert lay.poll_device_status() == 0
        return x, seen

    y1, seen = run(CHECKED)
    y2, _ = run(())
    assert torch.isfinite(y1.float()).all()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    for l in CHECKED:
        xin, yout, idx, gw = seen[l]
        rep = parity.check_routing_all(weights[l], xin, idx, gw, eps=EPS)
        assert rep["ok"], (l, {k: v for k, v in rep.items() if k != "oracle_counts"})
        ref = parity.oracle_reference(weights[l], xin, range(T), eps=EPS, residual=True)
        rep = parity.compare(ref, yout, idx, gw)
        assert rep["ok"], (l, rep)
    for lay in layers:
        lay.close()
    # the stack handle (all 47 layers in one launch): bitwise the per-layer result, at T = 256 and
    # at 16 tokens
    stack = fm.FlintMoEStack(weights, max_tokens=T, flags=flags, rms_eps=EPS)
    x = x0.clone()
    stack.forward(x)
    torch.cuda.synchronize()
    assert stack.poll_device_status() == 0
    assert torch.equal(x.view(torch.int16), y2.view(torch.int16))
    xs = x0[:16].clone()
    stack.forward(xs)
    small = [fm.FlintMoE(weights[l], max_tokens=16, flags=flags, rms_eps=EPS) for l in range(L)]
    xr = x0[:16].clone()
    for lay in small:
        lay.forward(xr, y=xr)
    torch.cuda.synchronize()
    assert stack.poll_device_status() == 0
    assert torch.equal(xs.view(torch.int16), xr.view(torch.int16))
    for lay in small:
        lay.close()
    stack.close()
