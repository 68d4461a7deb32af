"""Pins of the sliding-window decode attention oracle (oracle_swa_decode) to things other than
itself: torch's scaled_dot_product_attention (a library routine) when the sink is -inf, closed
forms with a sink, the GQA head mapping, and the ring's slot order.  A plausible slip -- the
sink carrying a value, a missing 1/sqrt(d), h % 4 instead of h / 8 for the KV head, attending
to invalid slots of a short sequence -- fails one of them."""
import math

import numpy as np
import torch

import oracle
import synth

NH, NKV, D, W = 32, 4, 128, 513


def rnd(shape, seed, tag, sigma=1.0):
    return synth.normal_bf16(seed, tag, int(np.prod(shape)), sigma).reshape(shape)


def inputs(B, seed):
    q = rnd((B, NH, D), seed, synth.TAG_Q)
    k = rnd((B, W, NKV, D), seed, synth.TAG_K)
    v = rnd((B, W, NKV, D), seed, synth.TAG_V)
    sinks = oracle.bf16_to_f64(rnd((NH,), seed, synth.TAG_SINK)).astype(np.float32)
    pos = np.array([synth.SWA_POSITIONS[b % len(synth.SWA_POSITIONS)] for b in range(B)], np.int32)
    return q, k, v, sinks, pos


def sdpa_reference(q, k, v, pos):
    """torch SDPA in float64, KV heads repeated to the query heads (h -> h // 8), invalid ring
    slots masked out; no sink."""
    B = q.shape[0]
    Q = torch.from_numpy(oracle.bf16_to_f64(q)).unsqueeze(2)                          # [B, NH, 1, D]
    K = torch.from_numpy(oracle.bf16_to_f64(k)).permute(0, 2, 1, 3).repeat_interleave(NH // NKV, dim=1)
    V = torch.from_numpy(oracle.bf16_to_f64(v)).permute(0, 2, 1, 3).repeat_interleave(NH // NKV, dim=1)
    n = np.minimum(pos.astype(np.int64) + 1, W)
    mask = torch.from_numpy(np.arange(W)[None, :] < n[:, None]).view(B, 1, 1, W)
    o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask)
    return o.squeeze(2).numpy()


def test_without_sink_matches_torch_sdpa_with_gqa_and_short_sequences():
    q, k, v, _, pos = inputs(8, 3)
    sinks = np.full(NH, -np.inf, np.float32)
    out = oracle.swa_decode(q, k, v, sinks, pos, nthreads=4)
    np.testing.assert_allclose(out, sdpa_reference(q, k, v, pos), rtol=1e-10, atol=1e-12)


def test_zero_keys_closed_form_with_sink():
    # every score is 0: out = sum_{j < n} v_j / (n + e^sink)
    q, k, v, sinks, pos = inputs(8, 4)
    k = np.zeros_like(k)
    out = oracle.swa_decode(q, k, v, sinks, pos)
    V = oracle.bf16_to_f64(v)
    for b in range(8):
        n = min(int(pos[b]) + 1, W)
        for h in range(NH):
            ref = V[b, :n, h // 8].sum(0) / (n + math.exp(float(sinks[h])))
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-14)


def test_single_cached_token_closed_form():
    # pos = 0: one key; out = v_0 / (1 + e^(sink - s_0)), s_0 = q.k_0 / sqrt(128)
    q, k, v, sinks, _ = inputs(1, 5)
    pos = np.zeros(1, np.int32)
    out = oracle.swa_decode(q, k, v, sinks, pos)
    Q, K, V = (oracle.bf16_to_f64(a) for a in (q, k, v))
    for h in range(NH):
        s0 = float(Q[0, h] @ K[0, 0, h // 8]) / math.sqrt(D)
        np.testing.assert_allclose(out[0, h], V[0, 0, h // 8] / (1.0 + math.exp(float(sinks[h]) - s0)), rtol=1e-12)


def test_large_sink_takes_the_attention():
    q, k, v, _, pos = inputs(2, 6)
    out = oracle.swa_decode(q, k, v, np.full(NH, 60.0, np.float32), pos)
    assert np.abs(out).max() < 1e-10


def test_ring_slot_order_does_not_matter_for_a_full_window():
    q, k, v, sinks, _ = inputs(2, 7)
    pos = np.array([4095, 700], np.int32)  # both windows full: all 513 slots valid
    perm = np.random.default_rng(0).permutation(W)
    a = oracle.swa_decode(q, k, v, sinks, pos)
    b = oracle.swa_decode(q, k[:, perm].copy(), v[:, perm].copy(), sinks, pos)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_kv_head_mapping_groups_eight_query_heads():
    # changing KV head 1 changes query heads 8..15 only
    q, k, v, sinks, pos = inputs(1, 8)
    a = oracle.swa_decode(q, k, v, sinks, pos)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 1] = rnd(k2[:, :, 1].shape, 9, synth.TAG_K)
    v2[:, :, 1] = rnd(v2[:, :, 1].shape, 9, synth.TAG_V)
    b = oracle.swa_decode(q, k2, v2, sinks, pos)
    changed = np.abs(a - b).max(axis=2)[0] > 0
    assert changed.tolist() == [8 <= h < 16 for h in range(NH)]
