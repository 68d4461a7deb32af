"""The parity rule's own logic (CPU): exact-tie order, gap segments."""
import numpy as np

from tests import parity


def test_tied_pair_keeps_relative_order_even_if_a_close_expert_moves():
    # oracle: 252 just above the tied pair (29, 203); fp32 may merge 252 into the tie
    idx_r = np.array([252, 29, 203, 168, 104, 110])
    gaps = np.array([2.2e-9, 0.0, 8.8e-5, 3.3e-5, 0.0, 7.9e-5])
    assert not parity.tie_broken_wrong(np.array([29, 203, 252, 168, 104, 110]), idx_r, gaps)
    assert parity.tie_broken_wrong(np.array([203, 29, 252, 168, 104, 110]), idx_r, gaps)
    assert parity.tie_broken_wrong(np.array([252, 29, 203, 168, 110, 104]), idx_r, gaps)


def test_no_tie_no_error():
    idx_r = np.array([1, 2, 3, 4, 5, 6])
    gaps = np.array([0.1, 0.1, 0.1, 0.1, 0.1, 0.1])
    assert not parity.tie_broken_wrong(np.array([6, 5, 4, 3, 2, 1]), idx_r, gaps)


# ---------------------------------------------------------------- exempt tokens: only near ties
def test_near_tie_choice_accepts_a_swap_across_the_gap():
    s = np.linspace(1.0, 0.5, 16)
    s[6] = s[5] - 5e-5  # the 7th expert is within the gap of the 6th
    assert parity.near_tie_choice_valid(np.array([0, 1, 2, 3, 4, 6]), s)
    assert parity.near_tie_choice_valid(np.array([0, 1, 2, 3, 4, 5]), s)


def test_near_tie_choice_rejects_a_wild_pick_a_duplicate_and_a_dropped_top_expert():
    s = np.linspace(1.0, 0.5, 16)
    s[6] = s[5] - 5e-5
    assert not parity.near_tie_choice_valid(np.array([0, 1, 2, 3, 4, 15]), s)  # far below the cut
    assert not parity.near_tie_choice_valid(np.array([0, 1, 2, 3, 4, 4]), s)   # duplicate
    assert not parity.near_tie_choice_valid(np.array([1, 2, 3, 4, 5, 6]), s)   # drops the best
    assert not parity.near_tie_choice_valid(np.array([0, 1, 2, 3, 4, 16]), s)  # out of range
    assert not parity.near_tie_choice_valid(np.array([5, 1, 2, 3, 4, 0]), s)   # not descending


def test_routing_verdict_categories():
    s = np.linspace(1.0, 0.5, 16)
    idx_r = np.arange(6)
    gaps = np.array([s[j] - s[j + 1] for j in range(6)])
    assert parity.routing_verdict(np.arange(6), idx_r, gaps, s) == "ok"
    assert parity.routing_verdict(np.array([0, 1, 2, 3, 4, 6]), idx_r, gaps, s) == "set"
    assert parity.routing_verdict(np.array([1, 0, 2, 3, 4, 5]), idx_r, gaps, s) == "order"
    s2 = s.copy()
    s2[6] = s2[5]
    gaps2 = gaps.copy()
    gaps2[5] = 0.0
    assert parity.routing_verdict(np.array([0, 1, 2, 3, 4, 6]), idx_r, gaps2, s2) == "ok"
    assert parity.routing_verdict(np.array([0, 1, 2, 3, 4, 12]), idx_r, gaps2, s2) == "near_tie"


def test_check_routing_all_fails_a_wrong_pick_on_an_exempt_token():
    # Real router shape; two duplicated, biased columns make exact 6th/7th ties on many tokens.
    import torch
    import synth
    import oracle
    H, E, T = 2048, 256, 48
    Wr = synth.normal_bf16(0, synth.TAG_ROUTER, H * E, 1.0 / np.sqrt(H)).reshape(H, E).copy()
    Wr[:, 201] = Wr[:, 17]
    bias = np.zeros(E, np.float32)
    bias[[17, 201]] = 1.5
    x = synth.normal_bf16(7, synth.TAG_X, T * H, 1.0).reshape(T, H)
    w = {"w_router": torch.from_numpy(Wr.view(np.int16)).view(torch.bfloat16),
         "router_bias": torch.from_numpy(bias)}
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    _, s = oracle.router(oracle.bf16_to_f64(x), Wr, bias)
    idx, g, gaps = oracle.select(s, 6)
    order = np.lexsort((np.broadcast_to(np.arange(E), s.shape), -s), axis=1)
    ex = [t for t in range(T) if gaps[t, 5] <= parity.GAP]
    assert ex, "the duplicated column must make exempt tokens"
    t = ex[0]

    def run(idx_g):
        sc = np.take_along_axis(s, idx_g.astype(np.int64), axis=1)
        gw = sc / sc.sum(1, keepdims=True)
        return parity.check_routing_all(w, xt, torch.from_numpy(idx_g.astype(np.int32)),
                                        torch.from_numpy(gw.astype(np.float32)))

    assert run(idx)["ok"]
    legit = idx.copy()
    legit[t, 5] = order[t, 6]  # the near-tied 7th expert instead of the 6th
    assert run(legit)["ok"]
    wild = idx.copy()
    wild[t, 5] = order[t, E - 1]  # the lowest-scoring expert
    rep = run(wild)
    assert not rep["ok"] and t in rep["set_mismatch"]
    dropped_best = idx.copy()
    dropped_best[t, 0] = order[t, 6]  # keeps the 6th, drops the best
    assert not run(dropped_best)["ok"]
