"""The allocation-free entry point, flint_moe_forward_noalloc, against flint_moe_forward.

Callers that cannot allocate device memory where they run the layer (a host program that
owns all device memory, a runtime that forbids allocation after start-up, a path that cannot
take cudaMalloc's implicit synchronisation) call the layer with weights, input and output
only; the library takes its scratch space from a fixed array of its own.  This file is
collected last so that a run stopping at the first failure has run every other test.
"""
import numpy as np
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
        # routing: identical; outputs: within the parity tolerance of the other tests
        assert torch.equal(idx, idx_ref) and torch.equal(gw, gw_ref)
        a = parity.oracle.bf16_to_f64(parity.to_np_bf16(y))
        b = parity.oracle.bf16_to_f64(parity.to_np_bf16(y_ref))
        d = np.abs(a - b)
        assert d.max() <= parity.MAX_ABS_REL * np.abs(b).max()
        assert d.sum() <= parity.REL_L1 * np.abs(b).sum()
    layer.close()


def test_noalloc_rejects_sizes_beyond_its_array():
    w = synth.flint_weights(seed=0, device=DEV)
    x = synth.torch_normal_bf16((fm.NOALLOC_MAX_TOKENS + 1, fm.HIDDEN), 5, synth.TAG_X, 1.0, device=DEV)
    with pytest.raises(fm.FlintMoEError) as e:
        fm.forward_noalloc(w, x)
    assert e.value.code == 2  # FLINT_MOE_ERR_UNSUPPORTED
