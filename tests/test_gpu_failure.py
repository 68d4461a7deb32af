"""The device-timeout path, exercised without a GPU fault: a handle created with the test-only
flag FLINT_MOE_FLAG_TEST_WAIT_TIMEOUT makes one bounded device wait per call on a workspace word
that nothing writes.  The wait must give up (about 0.25 s), the status word must report
FLINT_MOE_ERR_DEVICE_TIMEOUT through flint_moe_poll_device_status, the call's results must be
unaffected, and the context must stay usable for the next call."""
import time

import numpy as np
import pytest
import torch

import synth
import sparse_moe_layer_15_b300 as fm
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ERR_DEVICE_TIMEOUT = 5


@pytest.mark.parametrize("T,max_tokens", [(4, 16), (300, 512)], ids=["decode_path", "prefill_path"])
def test_device_wait_timeout_reported_and_context_survives(T, max_tokens):
    w = synth.flint_weights(seed=0, device=DEV)
    x = synth.torch_normal_bf16((T, fm.HIDDEN), 900 + T, synth.TAG_X, 1.0, device=DEV)
    normal = fm.FlintMoE(w, max_tokens=max_tokens)
    y_ok = normal.forward(x)
    torch.cuda.synchronize()
    assert normal.poll_device_status() == 0

    stalled = fm.FlintMoE(w, max_tokens=max_tokens, flags=fm.FLAG_TEST_WAIT_TIMEOUT)
    idx = torch.full((T, fm.TOP_K), -1, dtype=torch.int32, device=DEV)
    gw = torch.zeros((T, fm.TOP_K), dtype=torch.float32, device=DEV)
    t0 = time.perf_counter()
    y = stalled.forward(x, topk_idx=idx, topk_w=gw)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert 0.2 <= waited < 5.0, waited
    assert stalled.poll_device_status() == ERR_DEVICE_TIMEOUT
    assert stalled.poll_device_status() == 0  # the poll cleared it
    # the wait only delayed the call: same bits as the normal handle, and oracle parity
    assert torch.equal(y.view(torch.int16), y_ok.view(torch.int16))
    tokens = sorted(set(np.linspace(0, T - 1, 8).astype(int).tolist()))
    rep = parity.compare(parity.oracle_reference(w, x, tokens), y, idx, gw)
    assert rep["ok"], rep
    # routing alone takes the same wait
    stalled.route(x)
    assert stalled.poll_device_status() == ERR_DEVICE_TIMEOUT
    stalled.close()

    # the context is still usable
    y2 = normal.forward(x)
    torch.cuda.synchronize()
    assert normal.poll_device_status() == 0
    assert torch.equal(y2.view(torch.int16), y_ok.view(torch.int16))
    normal.close()
