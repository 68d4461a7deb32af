"""Pins of the fp64 oracle to things other than itself.

Each test ties one part of the oracle to a library routine, a closed form, an invariant,
a brute-force evaluation or a value printed on the pages, chosen so that a plausible slip
(a dropped bias, softmax for sigmoid, a swapped gate/up, a transposed matrix, a wrong
tie-break, un-normalised gates, a summation over the wrong experts) fails one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
import synth
from sparse_moe_layer_15_b300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(shape, seed, tag, sigma):
    n = int(np.prod(shape))
    return synth.normal_bf16(seed, tag, n, sigma).reshape(shape)


def tiny_layer(seed=0, H=64, E=16, k=4, I=32, Is=48, bias=False):
    Wr = bf16((H, E), seed, synth.TAG_ROUTER, 1.0 / math.sqrt(H))
    Wg = bf16((E, H, I), seed, synth.TAG_GATE, 0.2)
    Wu = bf16((E, H, I), seed, synth.TAG_UP, 0.2)
    Wd = bf16((E, I, H), seed, synth.TAG_DOWN, 0.2)
    Wsg = bf16((H, Is), seed, synth.TAG_SGATE, 0.2)
    Wsu = bf16((H, Is), seed, synth.TAG_SUP, 0.2)
    Wsd = bf16((Is, H), seed, synth.TAG_SDOWN, 0.2)
    b = None
    if bias:
        b = oracle.bf16_to_f64(bf16((E,), seed, synth.TAG_BIAS, 0.7)).astype(np.float32)
    return dict(Wr=Wr, Wg=Wg, Wu=Wu, Wd=Wd, Wsg=Wsg, Wsu=Wsu, Wsd=Wsd, b=b, k=k)


def to_layer(p):
    return oracle.Layer(p["Wr"], p["Wg"], p["Wu"], p["Wd"], p["Wsg"], p["Wsu"], p["Wsd"],
                        router_bias=p["b"], k=p["k"])


def x_rows(T, H, seed=1):
    return oracle.bf16_to_f64(bf16((T, H), seed, synth.TAG_X, 1.0))


# ---------------------------------------------------------------- independent brute force

def f64(bits):
    return oracle.bf16_to_f64(bits)


def brute_force(p, x):
    """Dense evaluation of every expert, masked by a top-k taken from a full lexicographic
    sort on (score desc, index asc).  numpy only; shares no code with the C oracle."""
    Wr, Wg, Wu, Wd = f64(p["Wr"]), f64(p["Wg"]), f64(p["Wu"]), f64(p["Wd"])
    Wsg, Wsu, Wsd = f64(p["Wsg"]), f64(p["Wsu"]), f64(p["Wsd"])
    T = x.shape[0]
    E = Wr.shape[1]
    b = np.zeros(E) if p["b"] is None else p["b"].astype(np.float64)
    s = expit(x @ Wr + b)
    eidx = np.broadcast_to(np.arange(E), s.shape)
    order = np.lexsort((eidx, -s), axis=1)
    chosen = order[:, : p["k"]]
    mask = np.zeros_like(s)
    np.put_along_axis(mask, chosen, 1.0, axis=1)
    w = mask * s
    w = w / w.sum(axis=1, keepdims=True)

    def mlp(a, g, u, d):
        zg = a @ g
        return (zg * expit(zg) * (a @ u)) @ d

    y = mlp(x, Wsg, Wsu, Wsd)
    for e in range(E):
        y = y + w[:, e : e + 1] * mlp(x, Wg[e], Wu[e], Wd[e])
    return y, chosen, s


# ---------------------------------------------------------------- router and selection

def test_router_matches_torch_float64():
    p = tiny_layer(bias=True)
    x = x_rows(9, 64)
    lg, s = oracle.router(x, p["Wr"], p["b"])
    ref_l = torch.from_numpy(x) @ torch.from_numpy(f64(p["Wr"])) + torch.from_numpy(p["b"].astype(np.float64))
    np.testing.assert_allclose(lg, ref_l.numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(s, torch.sigmoid(ref_l).numpy(), rtol=1e-13, atol=0)


def test_router_real_shape_non_square():
    # 2048 x 256 is not square: a transposed router would not even index the same entries.
    H, E = 2048, 256
    Wr = bf16((H, E), 0, synth.TAG_ROUTER, 1.0 / math.sqrt(H))
    x = x_rows(3, H, seed=7)
    _, s = oracle.router(x, Wr)
    ref = torch.sigmoid(torch.from_numpy(x) @ torch.from_numpy(f64(Wr))).numpy()
    np.testing.assert_allclose(s, ref, rtol=1e-12)


def test_zero_input_scores_are_sigmoid_of_bias():
    p = tiny_layer(bias=True)
    x = np.zeros((2, 64))
    lg, s = oracle.router(x, p["Wr"], p["b"])
    for e in range(16):
        b = float(p["b"][e])
        assert lg[0, e] == b
        assert s[0, e] == 1.0 / (1.0 + math.exp(-b))


def test_all_tied_scores_pick_lowest_indices_with_equal_gates():
    # x = 0, no bias: every score is sigmoid(0) = 1/2 exactly, so the choice is decided by
    # the tie-break alone, and the gates are 0.5 / 3.0 = 1/6 exactly.
    s = np.full((1, 256), 0.5)
    idx, g, gaps = oracle.select(s, 6)
    assert idx[0].tolist() == [0, 1, 2, 3, 4, 5]
    assert all(v == 1.0 / 6.0 for v in g[0])
    assert all(v == 0.0 for v in gaps[0])


def test_duplicated_router_column_breaks_tie_to_lower_index():
    H, E = 2048, 256
    Wr = bf16((H, E), 0, synth.TAG_ROUTER, 1.0 / math.sqrt(H)).copy()
    a, b = 17, 200
    Wr[:, b] = Wr[:, a]
    bias = np.zeros(E, np.float32)
    bias[a] = bias[b] = 2.0  # make the pair likely to be chosen
    x = x_rows(64, H, seed=11)
    _, s = oracle.router(x, Wr, bias)
    assert np.array_equal(s[:, a], s[:, b])
    idx, _, _ = oracle.select(s, 6)
    hits = 0
    for t in range(64):
        row = idx[t].tolist()
        if b in row:
            hits += 1
            assert a in row and row.index(a) == row.index(b) - 1
    assert hits > 0


def test_selection_matches_full_sort_bruteforce():
    rng = np.random.default_rng(3)
    s = rng.random((200, 256))
    s[:, 10] = s[:, 3]  # exact ties
    s[:, 250] = s[:, 3]
    idx, g, gaps = oracle.select(s, 6)
    eidx = np.broadcast_to(np.arange(256), s.shape)
    order = np.lexsort((eidx, -s), axis=1)
    assert np.array_equal(idx, order[:, :6])
    top = np.take_along_axis(s, order[:, :7], axis=1)
    np.testing.assert_array_equal(gaps[:, 5], top[:, 5] - top[:, 6])
    np.testing.assert_allclose(g, top[:, :6] / top[:, :6].sum(1, keepdims=True), rtol=1e-15)


def test_gates_sum_to_one():
    rng = np.random.default_rng(4)
    s = expit(rng.normal(size=(500, 256)) * 3)
    _, g, _ = oracle.select(s, 6)
    assert np.max(np.abs(g.sum(1) - 1.0)) <= 1e-12


def test_k_equals_E_gates_are_scores_over_their_sum():
    rng = np.random.default_rng(5)
    s = rng.random((4, 12))
    idx, g, gaps = oracle.select(s, 12)
    for t in range(4):
        np.testing.assert_allclose(g[t], s[t, idx[t]] / s[t].sum(), rtol=1e-15)
    assert np.isinf(gaps[:, -1]).all()


# ---------------------------------------------------------------- layer forward

def test_forward_matches_dense_masked_bruteforce_tiny():
    p = tiny_layer(bias=True)
    x = x_rows(16, 64)
    out = oracle.forward(to_layer(p), x)
    y_bf, chosen, _ = brute_force(p, x)
    assert np.array_equal(out["idx"], chosen)
    np.testing.assert_allclose(out["y"], y_bf, rtol=1e-11, atol=1e-12)


def test_forward_matches_bruteforce_real_widths():
    # Real hidden / expert / shared widths and k=6, with 16 experts so that the dense
    # brute force stays cheap.
    p = tiny_layer(seed=2, H=2048, E=16, k=6, I=512, Is=1024, bias=False)
    p["Wg"] = bf16((16, 2048, 512), 2, synth.TAG_GATE, 0.02)
    p["Wu"] = bf16((16, 2048, 512), 2, synth.TAG_UP, 0.02)
    p["Wd"] = bf16((16, 512, 2048), 2, synth.TAG_DOWN, 0.02)
    p["Wsg"] = bf16((2048, 1024), 2, synth.TAG_SGATE, 0.02)
    p["Wsu"] = bf16((2048, 1024), 2, synth.TAG_SUP, 0.02)
    p["Wsd"] = bf16((1024, 2048), 2, synth.TAG_SDOWN, 0.02)
    x = x_rows(4, 2048, seed=9)
    out = oracle.forward(to_layer(p), x)
    y_bf, chosen, _ = brute_force(p, x)
    assert np.array_equal(out["idx"], chosen)
    np.testing.assert_allclose(out["y"], y_bf, rtol=1e-10, atol=1e-12)


def test_k_equals_E_is_dense_sigmoid_weighted_mixture_torch():
    p = tiny_layer(seed=3, E=8, k=8)
    x = x_rows(5, 64, seed=4)
    out = oracle.forward(to_layer(p), x)
    X = torch.from_numpy(x)
    Wr = torch.from_numpy(f64(p["Wr"]))
    s = torch.sigmoid(X @ Wr)
    w = s / s.sum(1, keepdim=True)
    G = torch.einsum("th,ehi->tei", X, torch.from_numpy(f64(p["Wg"])))
    U = torch.einsum("th,ehi->tei", X, torch.from_numpy(f64(p["Wu"])))
    Y = torch.einsum("tei,eih->teh", torch.nn.functional.silu(G) * U, torch.from_numpy(f64(p["Wd"])))
    S = (torch.nn.functional.silu(X @ torch.from_numpy(f64(p["Wsg"]))) * (X @ torch.from_numpy(f64(p["Wsu"])))) \
        @ torch.from_numpy(f64(p["Wsd"]))
    ref = S + torch.einsum("te,teh->th", w, Y)
    np.testing.assert_allclose(out["y"], ref.numpy(), rtol=1e-11, atol=1e-13)


def test_single_expert_is_sum_of_two_swiglu_mlps_torch():
    # E = 1, k = 1: the gate is s/s = 1 and y = shared(x) + E_0(x).
    p = tiny_layer(seed=4, E=1, k=1, I=24, Is=40)
    x = x_rows(6, 64, seed=5)
    out = oracle.forward(to_layer(p), x)
    X = torch.from_numpy(x)
    F = torch.nn.functional

    def swiglu(g, u, d):
        return (F.silu(X @ torch.from_numpy(f64(g))) * (X @ torch.from_numpy(f64(u)))) @ torch.from_numpy(f64(d))

    ref = swiglu(p["Wsg"], p["Wsu"], p["Wsd"]) + swiglu(p["Wg"][0], p["Wu"][0], p["Wd"][0])
    assert np.all(out["gates"] == 1.0)
    np.testing.assert_allclose(out["y"], ref.numpy(), rtol=1e-12, atol=1e-14)


def test_gate_and_up_are_not_interchangeable():
    # silu(x Wg) * (x Wu) differs from silu(x Wu) * (x Wg); the oracle must follow the first.
    p = tiny_layer(seed=5, E=1, k=1)
    x = x_rows(3, 64, seed=6)
    y = oracle.forward(to_layer(p), x)["y"]
    q = dict(p)
    q["Wg"], q["Wu"] = p["Wu"], p["Wg"]
    y_swapped = oracle.forward(to_layer(q), x)["y"]
    assert np.max(np.abs(y - y_swapped)) > 1e-3


def test_zero_routed_down_gives_shared_expert_alone():
    p = tiny_layer(seed=6, bias=True)
    p["Wd"] = np.zeros_like(p["Wd"])
    x = x_rows(7, 64, seed=8)
    y = oracle.forward(to_layer(p), x)["y"]
    X = torch.from_numpy(x)
    F = torch.nn.functional
    ref = (F.silu(X @ torch.from_numpy(f64(p["Wsg"]))) * (X @ torch.from_numpy(f64(p["Wsu"])))) \
        @ torch.from_numpy(f64(p["Wsd"]))
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-14)


def test_zero_routed_gate_weights_contribute_nothing():
    p = tiny_layer(seed=7)
    x = x_rows(5, 64, seed=2)
    q = dict(p)
    q["Wg"] = np.zeros_like(p["Wg"])
    y0 = oracle.forward(to_layer(q), x)["y"]
    q["Wd"] = np.zeros_like(p["Wd"])
    y_shared = oracle.forward(to_layer(q), x)["y"]
    assert np.array_equal(y0, y_shared)


def test_zero_input_gives_zero_output():
    p = tiny_layer(seed=8, bias=True)
    y = oracle.forward(to_layer(p), np.zeros((3, 64)))["y"]
    assert np.all(y == 0.0)


def test_forward_given_equals_forward_on_its_own_choice():
    p = tiny_layer(seed=9, bias=True)
    x = x_rows(10, 64, seed=3)
    out = oracle.forward(to_layer(p), x)
    y2 = oracle.forward_given(to_layer(p), x, out["idx"])
    np.testing.assert_array_equal(out["y"], y2)


def brute_force_given(p, x, chosen):
    """Dense evaluation of every expert masked by a GIVEN expert set per row (``chosen``
    [T, k]), the gates being the fp64 sigmoid scores of that set normalised over it.  numpy
    only; shares no code with the C oracle."""
    Wr, Wg, Wu, Wd = f64(p["Wr"]), f64(p["Wg"]), f64(p["Wu"]), f64(p["Wd"])
    Wsg, Wsu, Wsd = f64(p["Wsg"]), f64(p["Wsu"]), f64(p["Wsd"])
    E = Wr.shape[1]
    b = np.zeros(E) if p["b"] is None else p["b"].astype(np.float64)
    s = expit(x @ Wr + b)
    mask = np.zeros_like(s)
    np.put_along_axis(mask, np.asarray(chosen, dtype=np.int64), 1.0, axis=1)
    w = mask * s
    w = w / w.sum(axis=1, keepdims=True)

    def mlp(a, g, u, d):
        zg = a @ g
        return (zg * expit(zg) * (a @ u)) @ d

    y = mlp(x, Wsg, Wsu, Wsd)
    for e in range(E):
        y = y + w[:, e : e + 1] * mlp(x, Wg[e], Wu[e], Wd[e])
    return y


def non_top_sets(s, k, rng):
    """Per row, two sets that are NOT the top-k: ranks 2..k+1 of the (score desc, index asc)
    order (the best expert dropped, the (k+1)-th taken in), and a random k-subset, each listed
    in a scrambled order (the result must not depend on the listing order)."""
    E = s.shape[1]
    order = np.lexsort((np.broadcast_to(np.arange(E), s.shape), -s), axis=1)
    shifted = order[:, 1 : k + 1].copy()
    rand = np.stack([rng.choice(E, size=k, replace=False) for _ in range(s.shape[0])])
    for row in shifted:
        rng.shuffle(row)
    return shifted.astype(np.int32), rand.astype(np.int32), order[:, :k]


def test_forward_given_matches_bruteforce_on_sets_that_are_not_the_top_k():
    # A re-evaluation that ignored the given set (re-selecting the top-k), or normalised the
    # gates over the wrong experts (all, or the true top-k), fails here: the given sets are
    # never the top-k.
    rng = np.random.default_rng(21)
    p = tiny_layer(seed=13, E=16, k=4, bias=True)
    x = x_rows(12, 64, seed=14)
    _, s = oracle.router(x, p["Wr"], p["b"])
    shifted, rand, top = non_top_sets(s, 4, rng)
    L = to_layer(p)
    for given in (shifted, rand):
        assert all(set(g.tolist()) != set(t.tolist()) for g, t in zip(given, top))
        y = oracle.forward_given(L, x, given)
        np.testing.assert_allclose(y, brute_force_given(p, x, given), rtol=1e-11, atol=1e-12)
        assert np.max(np.abs(y - oracle.forward(L, x)["y"])) > 1e-3


def test_forward_given_matches_bruteforce_real_widths():
    # Real hidden / expert / shared widths and k = 6, 16 experts, a given set of ranks 2..7.
    rng = np.random.default_rng(22)
    p = tiny_layer(seed=14, H=2048, E=16, k=6, I=512, Is=1024, bias=True)
    p["Wg"] = bf16((16, 2048, 512), 14, synth.TAG_GATE, 0.02)
    p["Wu"] = bf16((16, 2048, 512), 14, synth.TAG_UP, 0.02)
    p["Wd"] = bf16((16, 512, 2048), 14, synth.TAG_DOWN, 0.02)
    p["Wsg"] = bf16((2048, 1024), 14, synth.TAG_SGATE, 0.02)
    p["Wsu"] = bf16((2048, 1024), 14, synth.TAG_SUP, 0.02)
    p["Wsd"] = bf16((1024, 2048), 14, synth.TAG_SDOWN, 0.02)
    x = x_rows(3, 2048, seed=15)
    _, s = oracle.router(x, p["Wr"], p["b"])
    shifted, _, _ = non_top_sets(s, 6, rng)
    y = oracle.forward_given(to_layer(p), x, shifted)
    np.testing.assert_allclose(y, brute_force_given(p, x, shifted), rtol=1e-10, atol=1e-12)


def test_forward_given_rejects_out_of_range_experts():
    p = tiny_layer(seed=15)
    x = x_rows(1, 64)
    with pytest.raises(RuntimeError):
        oracle.forward_given(to_layer(p), x, np.array([[0, 1, 2, 16]], np.int32))


def test_missing_expert_is_reported():
    p = tiny_layer(seed=10)
    L = oracle.Layer(p["Wr"], {0: p["Wg"][0]}, {0: p["Wu"][0]}, {0: p["Wd"][0]}, p["Wsg"], p["Wsu"], p["Wsd"], k=4)
    with pytest.raises(RuntimeError):
        oracle.forward(L, x_rows(2, 64))


def test_threaded_forward_is_identical():
    p = tiny_layer(seed=11, bias=True)
    x = x_rows(13, 64, seed=12)
    a = oracle.forward(to_layer(p), x)
    b = oracle.forward(to_layer(p), x, nthreads=4)
    for key in ("y", "idx", "gates", "gaps"):
        assert np.array_equal(a[key], b[key])


# ---------------------------------------------------------------- permutation, norm

def test_permute_is_stable_counting_sort():
    rng = np.random.default_rng(6)
    idx = rng.integers(0, 256, size=(300, 6)).astype(np.int32)
    counts, offsets, perm, inv = oracle.permute(idx, 256)
    flat = idx.reshape(-1)
    assert np.array_equal(counts, np.bincount(flat, minlength=256))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(inv[perm], np.arange(flat.size))


def test_rmsnorm_closed_form_and_numpy():
    eps = 1e-6
    x = np.full((1, 2048), 3.0)
    r = oracle.rmsnorm(x, eps)
    assert np.allclose(r, 3.0 / math.sqrt(9.0 + eps), rtol=1e-15, atol=0)
    rng = np.random.default_rng(7)
    x = rng.normal(size=(5, 2048))
    r = oracle.rmsnorm(x, eps)
    ref = x / np.sqrt((x * x).mean(axis=1, keepdims=True) + eps)
    np.testing.assert_allclose(r, ref, rtol=1e-14)


def test_round_bf16_matches_float32_rounding():
    # Every float32 value rounds to bf16 in a single step, so the float32 bit trick of the
    # generator (round to nearest even on the low 16 bits) is an independent check.
    rng = np.random.default_rng(8)
    v = np.concatenate([rng.normal(size=4000).astype(np.float32),
                        np.array([1.00390625, 1.01171875, -2.5, 3.0e-3, 65504.0, 1e-20], np.float32)])
    # half-way cases between bf16 neighbours: low 16 bits exactly 0x8000
    halves = (rng.integers(0x3F00, 0x4100, size=200).astype(np.uint32) << 16) | np.uint32(0x8000)
    v = np.concatenate([v, halves.view(np.float32)])
    want = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(v)).astype(np.float64)
    got = oracle.round_bf16(v.astype(np.float64))
    assert np.array_equal(got, want)


def test_prenorm_residual_composition():
    p = tiny_layer(seed=12)
    x = x_rows(4, 64, seed=13) * 3.0
    out = oracle.prenorm_residual(to_layer(p), x, 1e-6)
    r = oracle.round_bf16(x / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-6))
    y_bf, _, _ = brute_force(p, r)
    np.testing.assert_allclose(out["y"], x + y_bf, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- page-printed constants

def test_accounting_reproduces_page_counts():
    with open(os.path.join(GOLDEN, "flint_layer_config.json")) as f:
        g = json.load(f)
    assert acc.HIDDEN == g["hidden_size"]["value"]
    assert acc.N_EXPERTS == g["n_routed_experts"]["value"]
    assert acc.TOP_K == g["top_k"]["value"]
    assert acc.EXPERT_INTER == g["expert_intermediate"]["value"]
    assert acc.SHARED_INTER == g["shared_intermediate"]["value"]
    L = g["n_moe_layers"]["value"]
    routed = L * acc.N_EXPERTS * acc.expert_params() / 1e9
    assert abs(routed / g["routed_params_total_billions"]["value"] - 1) <= g["routed_params_total_billions"]["rel_tol"]
    active = L * acc.active_params_per_token() / 1e9
    assert abs(active / g["moe_active_params_per_token_billions"]["value"] - 1) <= \
        g["moe_active_params_per_token_billions"]["rel_tol"]
    # the 47 MoE layers in bf16 must fit inside the page's whole-model checkpoint size
    assert L * acc.layer_weight_bytes() / 1e9 < g["bf16_checkpoint_gb"]["value"]


def test_flop_and_byte_formulas():
    assert acc.flops_per_token() == 51_380_224
    assert acc.touched_weight_bytes(6) == 6 * 6_291_456 + 12_582_912 + 1_048_576
    assert acc.layer_weight_bytes() == 1_624_244_224
    assert abs(acc.expected_touched_experts(16) - 80.8) < 0.05


# ---------------------------------------------------------------- dense MLP layers

def test_dense_layer_real_width_matches_textbook_swiglu_torch():
    # The dense layers' width 6144 (2 x 3 x 2048 x 6144 = 75.5M parameters, the pages' "about
    # 75M" for the two), against torch's silu on the same bf16 weights, and not the swapped
    # gate/up.
    H, Id = 2048, 6144
    wg = bf16((H, Id), 3, synth.TAG_DGATE, 0.02)
    wu = bf16((H, Id), 3, synth.TAG_DUP, 0.02)
    wd = bf16((Id, H), 3, synth.TAG_DDOWN, 0.02)
    x = x_rows(3, H, seed=17)
    y = oracle.dense(x, wg, wu, wd, nthreads=2)
    X = torch.from_numpy(x)
    F = torch.nn.functional
    G, U, D = (torch.from_numpy(f64(a)) for a in (wg, wu, wd))
    ref = (F.silu(X @ G) * (X @ U)) @ D
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-11, atol=1e-13)
    swapped = (F.silu(X @ U) * (X @ G)) @ D
    assert np.max(np.abs(y - swapped.numpy())) > 1e-3
    assert 2 * (3 * H * Id) == 75_497_472
