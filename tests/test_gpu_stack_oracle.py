"""The one-launch layer stack (decode_stack) against the fp64 oracle directly,
layer by layer with teacher forcing.

Stacks of 1, 2 and 3 layers (weights seed 100 + l; x <- x + MoE_l(RMSNorm(x)), eps 1e-6) run on
the same input; the output of the n-layer stack is the input of layer n, so every layer's bf16
input and output come from the kernel itself.  The oracle's layer l takes the kernel's input to
layer l (the 47-layer workload's teacher forcing, serving-kit post "The architecture, from the
config": the MoE layers run back to back) and the parity rule is applied to every token's routing
and output.
"""
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


@pytest.mark.parametrize("T", [1, 16, 256])
def test_stack_prefixes_teacher_forced_against_oracle(layer_weights, T):
    flags = fm.FLAG_PRE_RMSNORM | fm.FLAG_RESIDUAL
    x0 = synth.torch_normal_bf16((T, fm.HIDDEN), 4200 + T, synth.TAG_X, 1.0, device=DEV)
    outs, routes = [x0.clone()], []
    for n in range(1, N_LAYERS + 1):
        stack = fm.FlintMoEStack(layer_weights[:n], max_tokens=T, flags=flags, rms_eps=EPS)
        idx = torch.full((n, T, fm.TOP_K), -1, dtype=torch.int32, device=DEV)
        gw = torch.zeros((n, T, fm.TOP_K), dtype=torch.float32, device=DEV)
        x = x0.clone()
        stack.forward(x, topk_idx=idx, topk_w=gw)
        torch.cuda.synchronize()
        assert stack.poll_device_status() == 0
        stack.close()
        outs.append(x)
        routes.append((idx[n - 1], gw[n - 1]))
        # the shorter stacks' routing is repeated by the longer ones
        if n > 1:
            assert torch.equal(idx[n - 2], routes[n - 2][0])
    for l in range(N_LAYERS):
        xin, yout = outs[l], outs[l + 1]
        idx, gw = routes[l]
        ref = parity.oracle_reference(layer_weights[l], xin, range(T), eps=EPS, residual=True)
        rep = parity.compare(ref, yout, idx, gw)
        assert rep["ok"], (l, rep)
        rep = parity.check_routing_all(layer_weights[l], xin, idx, gw, eps=EPS)
        assert rep["ok"], (l, {k: v for k, v in rep.items() if k != "oracle_counts"})
