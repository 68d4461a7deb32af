"""The allocation-free entry point, flint_moe_forward_noalloc, against flint_moe_forward.

Some callers cannot allocate device memory where they run the layer: a host program that owns
all device memory and gives plugins no allocator, a runtime that plans its memory at start-up
and forbids allocation afterwards, or a latency path that cannot take cudaMalloc's implicit
synchronisation.  They call the layer with weights, input and output only; the library takes
its scratch space from a fixed array of its own (at most 4 tokens per call).

The entry point runs the same kernel on the same grid as flint_moe_forward, so its outputs and
routing must be bitwise those of flint_moe_forward; they are also checked against the fp64
oracle, and its own status word (read through flint_moe_noalloc_poll_device_status) must be
clear.  This file is collected last so that a run stopping at the first failure has run every
other test; it passes alone in a fresh process as well.
"""
import pytest
import torch

import synth
import sparse_moe_layer_15_b300 as fm
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def test_noalloc_matches_forward_on_two_calls_in_a_row():
    w = synth.flint_weights(seed=0, device=DEV)
    layer = fm.FlintMoE(w, max_tokens=fm.NOALLOC_MAX_TOKENS)
    for T, seed in ((fm.NOALLOC_MAX_TOKENS, 31), (3, 32)):  # two calls in a row, different sizes
        x = synth.torch_normal_bf16((T, fm.HIDDEN), seed, synth.TAG_X, 1.0, device=DEV)
        idx_ref = torch.empty((T, fm.TOP_K), dtype=torch.int32, device=DEV)
        gw_ref = torch.empty((T, fm.TOP_K), dtype=torch.float32, device=DEV)
        y_ref = layer.forward(x, topk_idx=idx_ref, topk_w=gw_ref)
        idx = torch.full((T, fm.TOP_K), -1, dtype=torch.int32, device=DEV)
        gw = torch.zeros((T, fm.TOP_K), dtype=torch.float32, device=DEV)
        y = fm.forward_noalloc(w, x, topk_idx=idx, topk_w=gw)
        torch.cuda.synchronize()
        assert layer.poll_device_status() == 0
        assert fm.noalloc_poll_device_status() == 0
        # same kernel, grid and arithmetic: bitwise equal to flint_moe_forward
        assert torch.equal(idx, idx_ref)
        assert torch.equal(gw.view(torch.int32), gw_ref.view(torch.int32))
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
        # and within the parity rule of the fp64 oracle
        ref = parity.oracle_reference(w, x, range(T))
        rep = parity.compare(ref, y, idx, gw)
        assert rep["ok"], rep
    layer.close()


def test_noalloc_rejects_sizes_beyond_its_array():
    w = synth.flint_weights(seed=0, device=DEV)
    x = synth.torch_normal_bf16((fm.NOALLOC_MAX_TOKENS + 1, fm.HIDDEN), 5, synth.TAG_X, 1.0, device=DEV)
    with pytest.raises(fm.FlintMoEError) as e:
        fm.forward_noalloc(w, x)
    assert e.value.code == 2  # FLINT_MOE_ERR_UNSUPPORTED
    assert fm.noalloc_poll_device_status() == 0
