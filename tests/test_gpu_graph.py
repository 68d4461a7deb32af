"""route / forward make no host synchronisation and no allocation, so they can be captured in a
CUDA graph and replayed: a captured forward (the decode-size kernel, and the tensor-core path's
kernels chained by programmatic dependent launch) and a captured one-launch layer stack replay
bitwise the outputs of the same calls made directly, several times in a row (every call leaves
the workspace's counters at zero)."""
import pytest
import torch

import synth
import sparse_moe_layer_15_b300 as fm

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def capture(fn):
    # torch's recipe: warm up on a side stream, then capture on it
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("T", [16, 300])
def test_forward_replays_from_a_cuda_graph(T):
    w = synth.flint_weights(seed=0, device=DEV)
    layer = fm.FlintMoE(w, max_tokens=T)
    x = synth.torch_normal_bf16((T, fm.HIDDEN), 7000 + T, synth.TAG_X, 1.0, device=DEV)
    ref = layer.forward(x)
    torch.cuda.synchronize()
    y = torch.empty_like(x)
    g = capture(lambda: layer.forward(x, y))
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    assert layer.poll_device_status() == 0
    layer.close()


def test_stack_replays_from_a_cuda_graph():
    T, L = 8, 3
    flags = fm.FLAG_PRE_RMSNORM | fm.FLAG_RESIDUAL
    weights = [synth.flint_weights(seed=100 + l, device=DEV) for l in range(L)]
    stack = fm.FlintMoEStack(weights, max_tokens=T, flags=flags)
    x0 = synth.torch_normal_bf16((T, fm.HIDDEN), 7100, synth.TAG_X, 1.0, device=DEV)
    ref = x0.clone()
    stack.forward(ref)
    torch.cuda.synchronize()
    x = x0.clone()
    g = capture(lambda: stack.forward(x))
    for _ in range(3):
        x.copy_(x0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(x.view(torch.int16), ref.view(torch.int16))
    assert stack.poll_device_status() == 0
    stack.close()
