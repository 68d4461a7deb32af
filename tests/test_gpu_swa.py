"""Sliding-window decode attention with learned sinks (flint_swa_*) against the fp64 oracle,
through the C ABI: every sequence and head, batches from 1 to 256 with the length mix of the
input recipe (sequences shorter than the window, exactly one slot, full windows), a sink of
-inf (plain softmax), bitwise run-to-run determinism, a reused workspace (its tickets return
to zero) and the bounds check of a negative position.  Tolerance: the layer's, max |o - o_ref|
<= 2e-2 max |o_ref| and relative L1 <= 5e-3."""
import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_moe_layer_15_b300 as fm
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def reference(inp):
    h = {k: parity.to_np_bf16(v) for k, v in inp.items() if k in ("q", "k", "v")}
    return oracle.swa_decode(h["q"], h["k"], h["v"], inp["sinks"].cpu().numpy(), inp["pos"].cpu().numpy(),
                             nthreads=parity.ORACLE_THREADS)


def check(out, ref):
    g = oracle.bf16_to_f64(parity.to_np_bf16(out))
    d = np.abs(g - ref)
    max_rel, rel_l1 = d.max() / np.abs(ref).max(), d.sum() / np.abs(ref).sum()
    assert max_rel <= parity.MAX_ABS_REL and rel_l1 <= parity.REL_L1, (max_rel, rel_l1)


@pytest.mark.parametrize("B", [1, 3, 8, 64, 256])
def test_swa_decode_matches_oracle(B):
    attn = fm.SwaAttention(max_batch=256, device=DEV)
    inp = synth.swa_inputs(B, seed=900 + B, device=DEV)
    out = attn.decode(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["pos"])
    out2 = attn.decode(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["pos"])
    torch.cuda.synchronize()
    assert attn.poll_device_status() == 0
    check(out, reference(inp))
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_swa_decode_without_sink_and_single_slot():
    attn = fm.SwaAttention(max_batch=8, device=DEV)
    inp = synth.swa_inputs(8, seed=950, device=DEV)
    inp["sinks"] = torch.full((32,), float("-inf"), device=DEV)
    inp["pos"] = torch.tensor([0, 1, 56, 57, 58, 511, 512, 100000], dtype=torch.int32, device=DEV)
    out = attn.decode(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["pos"])
    torch.cuda.synchronize()
    assert attn.poll_device_status() == 0
    check(out, reference(inp))
    # one valid slot and no sink: the output is that slot's value row
    v0 = inp["v"][0, 0].float()  # [4, 128]
    assert torch.allclose(out[0].float(), v0.repeat_interleave(8, dim=0), atol=0, rtol=2 ** -8)


def test_swa_decode_negative_position_is_a_bounds_error():
    attn = fm.SwaAttention(max_batch=2, device=DEV)
    inp = synth.swa_inputs(2, seed=960, device=DEV)
    inp["pos"][1] = -5
    attn.decode(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["pos"])
    torch.cuda.synchronize()
    assert attn.poll_device_status() == 6  # FLINT_MOE_ERR_DEVICE_BOUNDS, then cleared
    inp["pos"][1] = 7
    attn.decode(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["pos"])
    assert attn.poll_device_status() == 0


def test_swa_decode_rejects_a_batch_beyond_the_workspace():
    attn = fm.SwaAttention(max_batch=4, device=DEV)
    inp = synth.swa_inputs(5, seed=970, device=DEV)
    with pytest.raises(fm.FlintMoEError) as e:
        attn.decode(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["pos"])
    assert e.value.code == 3  # FLINT_MOE_ERR_WORKSPACE
