"""Parity rule between the CUDA layer and the fp64 oracle (test infrastructure).

Routing: on every token whose oracle gap between the 6th and 7th score exceeds 1e-4 the GPU
must choose the same expert set; inside the chosen list, the GPU order must equal the oracle
order across every adjacent pair whose oracle gap exceeds 1e-4, and every exactly tied pair
(equal fp64 scores) must keep its relative order, lower index first.  Tokens at or below the gap are exempt:
their fp32 scores may legitimately pick the other near-tied expert, but only a near-tied one:
the GPU's list must hold 6 distinct experts, every chosen expert must score within the gap of
every expert left out (min over the chosen >= max over the rest - 1e-4, oracle fp64 scores),
and the list must descend in score up to the gap.  The oracle then re-evaluates such a token
with the GPU's choice (gates = its fp64 scores renormalised).

Outputs (bf16): max |y_gpu - y_ref| <= 2e-2 * max |y_ref| and
sum |y_gpu - y_ref| / sum |y_ref| <= 5e-3 (relative L1).
Gates: |g_gpu - g_ref| <= 2e-5 per chosen expert, and the GPU's gates sum to 1 within 1e-5.
"""
from __future__ import annotations

import os

import numpy as np

import oracle
import synth

GAP = 1e-4
MAX_ABS_REL = 2e-2
REL_L1 = 5e-3
GATE_TOL = 2e-5
# threads for full-batch oracle references (each token is the same single-threaded computation)
ORACLE_THREADS = max(1, min(os.cpu_count() or 8, 64))


def tie_broken_wrong(idx_g, idx_r, gaps):
    """True if an exactly tied pair of the oracle's ranking (gap 0: equal fp64 scores, the
    lower index listed first) appears in the GPU's list in the other relative order.  Experts
    that are merely close (gap <= GAP) may move across the pair; that is the gap rule's job."""
    pos = {int(e): k for k, e in enumerate(idx_g)}
    for j in range(len(idx_r) - 1):
        if gaps[j] == 0.0:
            a, b = int(idx_r[j]), int(idx_r[j + 1])
            if a in pos and b in pos and pos[a] > pos[b]:
                return True
    return False


def near_tie_choice_valid(idx_g, s):
    """The GPU's expert list ``idx_g`` for one exempt token is a top-k of the oracle's fp64
    scores ``s`` [E] perturbed by less than the gap: distinct experts in range, every chosen
    expert scoring no less than every expert left out minus GAP (so an expert the GPU took in
    is near the oracle's k-th score, and an oracle expert it dropped is near the (k+1)-th),
    and the list descending in score up to GAP."""
    E = s.shape[0]
    g = [int(e) for e in idx_g]
    if len(set(g)) != len(g) or any(e < 0 or e >= E for e in g):
        return False
    chosen = np.zeros(E, bool)
    chosen[g] = True
    if chosen.all():
        return True
    if s[chosen].min() < s[~chosen].max() - GAP:
        return False
    return all(s[g[j]] >= s[g[j + 1]] - GAP for j in range(len(g) - 1))


def routing_verdict(idx_g, idx_r, gaps, s):
    """The routing rule on one token: "ok", "set" (a non-exempt token chose another set),
    "near_tie" (an exempt token's other choice is not a near-tied one), "order" (a segment
    of the ranking between gaps > GAP holds other experts) or "tie" (an exact tie in the
    wrong order).  ``s``: the oracle's fp64 scores of the token (all experts)."""
    same = set(int(e) for e in idx_g) == set(int(e) for e in idx_r)
    if not same:
        if gaps[5] > GAP:
            return "set"
        return "ok" if near_tie_choice_valid(idx_g, s) else "near_tie"
    a = 0
    for j in range(6):
        if j == 5 or gaps[j] > GAP:
            if set(int(e) for e in idx_g[a:j + 1]) != set(int(e) for e in idx_r[a:j + 1]):
                return "order"
            a = j + 1
    if tie_broken_wrong(idx_g, idx_r, gaps):
        return "tie"
    return "ok"


def to_np_bf16(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_layer(w, experts=None):
    hw = synth.weights_to_host(w, experts=experts)
    return oracle.Layer(hw["w_router"], hw["w_gate"], hw["w_up"], hw["w_down"], hw["ws_gate"], hw["ws_up"],
                        hw["ws_down"], router_bias=hw["router_bias"], k=6)


def touched_experts(w, xin64, tokens):
    """Experts the oracle's routing picks for these token rows, plus every expert whose score
    is within twice the exemption gap of the 6th (so that a re-evaluation with the GPU's
    choice of a near-tied expert finds its weights)."""
    wr = to_np_bf16(w["w_router"])
    b = None if w.get("router_bias") is None else w["router_bias"].detach().float().cpu().numpy()
    _, s = oracle.router(xin64[tokens], wr, b)
    idx, _, _ = oracle.select(s, 6)
    need = set(idx.reshape(-1).tolist())
    sixth = -np.sort(-s, axis=1)[:, 5]
    for t in range(s.shape[0]):
        need.update(np.nonzero(s[t] >= sixth[t] - 2 * GAP)[0].tolist())
    return sorted(need)


def oracle_reference(w, x, tokens, xin64=None, nthreads=ORACLE_THREADS, residual=False, eps=None):
    """Oracle outputs for the token rows ``tokens`` of x (bf16 torch tensor).  With ``eps``
    the layer is pre-normed (x' = rms(x)) and, with ``residual``, y = x + MoE(x')."""
    x64 = oracle.bf16_to_f64(to_np_bf16(x))
    tokens = np.asarray(tokens, dtype=np.int64)
    xin = x64 if eps is None else oracle.prenorm_input(x64, eps)
    experts = touched_experts(w, xin, tokens)
    layer = oracle_layer(w, experts=experts)
    out = oracle.forward(layer, xin[tokens], nthreads=nthreads, want_scores=True)
    if residual:
        out["y"] = x64[tokens] + out["y"]
    out["tokens"] = tokens
    out["layer"] = layer
    out["xin"] = xin[tokens]
    out["xres"] = x64[tokens] if residual else None
    return out


def compare(ref, y, idx, gw, counts=None, full_T=None):
    """Apply the parity rule to GPU results (torch tensors over all T rows) on ref's tokens."""
    tokens = ref["tokens"]
    y_g = oracle.bf16_to_f64(to_np_bf16(y))[tokens]
    idx_g = idx.detach().cpu().numpy()[tokens]
    w_g = gw.detach().cpu().numpy().astype(np.float64)[tokens]
    idx_r, gaps, g_r, s_r = ref["idx"], ref["gaps"], ref["gates"], ref["scores"]
    n = len(tokens)
    exempt = gaps[:, 5] <= GAP
    set_mismatch, order_err, tie_err = [], [], []
    for i in range(n):
        v = routing_verdict(idx_g[i], idx_r[i], gaps[i], s_r[i])
        if v in ("set", "near_tie"):
            set_mismatch.append(int(tokens[i]))
        elif v == "order":
            order_err.append(int(tokens[i]))
        elif v == "tie":
            tie_err.append(int(tokens[i]))
    # re-evaluate exempt tokens whose set differs, with the GPU's choice
    y_ref = ref["y"].copy()
    reeval = [i for i in range(n) if set(idx_g[i].tolist()) != set(idx_r[i].tolist()) and exempt[i]
              and int(tokens[i]) not in set_mismatch]
    missing = []
    if reeval:
        try:
            yy = oracle.forward_given(ref["layer"], ref["xin"][reeval], idx_g[reeval])
            if ref.get("xres") is not None:
                yy = ref["xres"][reeval] + yy
            y_ref[reeval] = yy
        except RuntimeError:
            missing = [int(tokens[i]) for i in reeval]
    d = np.abs(y_g - y_ref)
    ymax = float(np.max(np.abs(y_ref))) if y_ref.size else 0.0
    max_rel = float(d.max() / ymax) if ymax > 0 else float(d.max())
    rel_l1 = float(d.sum() / max(np.abs(y_ref).sum(), 1e-300))
    # gates by expert id
    gate_err = 0.0
    for i in range(n):
        sg = dict(zip(idx_g[i].tolist(), w_g[i].tolist()))
        if set(sg) == set(idx_r[i].tolist()):
            for e, g in zip(idx_r[i].tolist(), g_r[i].tolist()):
                gate_err = max(gate_err, abs(sg[e] - g))
        else:
            sc = s_r[i, idx_g[i]]
            for e, g in zip(idx_g[i].tolist(), (sc / sc.sum()).tolist()):
                gate_err = max(gate_err, abs(sg[e] - g))
    gate_sum_err = float(np.max(np.abs(w_g.sum(1) - 1.0))) if n else 0.0
    rep = dict(n_tokens=n, n_exempt=int(exempt.sum()), set_mismatch=set_mismatch, order_err=order_err,
               tie_err=tie_err, reevaluated=len(reeval), missing=missing, max_abs_err_rel=max_rel,
               rel_l1=rel_l1, gate_err=gate_err, gate_sum_err=gate_sum_err,
               routing_mismatch=len(set_mismatch) + len(order_err) + len(tie_err))
    rep["ok"] = (not set_mismatch and not order_err and not tie_err and not missing and max_rel <= MAX_ABS_REL
                 and rel_l1 <= REL_L1 and gate_err <= GATE_TOL and gate_sum_err <= 1e-5)
    return rep


def check_routing_all(w, x, idx_gpu, gw_gpu, eps=None):
    """The routing rule on every token (oracle fp64 scores of all tokens; no expert weights
    needed).  Returns a report with the mismatches, the exempt count and the oracle counts."""
    x64 = oracle.bf16_to_f64(to_np_bf16(x))
    xin = x64 if eps is None else oracle.prenorm_input(x64, eps)
    wr = to_np_bf16(w["w_router"])
    b = None if w.get("router_bias") is None else w["router_bias"].detach().float().cpu().numpy()
    _, s = oracle.router(xin, wr, b)
    idx_r, g_r, gaps = oracle.select(s, 6)
    idx_g = idx_gpu.detach().cpu().numpy()
    w_g = gw_gpu.detach().cpu().numpy().astype(np.float64)
    exempt = gaps[:, 5] <= GAP
    set_mm, order_err, tie_err = [], [], []
    gate_err = 0.0
    for t in range(idx_r.shape[0]):
        v = routing_verdict(idx_g[t], idx_r[t], gaps[t], s[t])
        if v in ("set", "near_tie"):
            set_mm.append(t)
            continue
        if v == "order":
            order_err.append(t)
        elif v == "tie":
            tie_err.append(t)
        # gates against the oracle's fp64 scores of the experts the GPU chose
        sc = s[t, idx_g[t]]
        for g, ref in zip(w_g[t].tolist(), (sc / sc.sum()).tolist()):
            gate_err = max(gate_err, abs(g - ref))
    rep = dict(n=int(idx_r.shape[0]), n_exempt=int(exempt.sum()), set_mismatch=set_mm[:10], n_set_mismatch=len(set_mm),
               order_err=order_err[:10], tie_err=tie_err[:10], gate_err=gate_err,
               oracle_counts=np.bincount(idx_r.reshape(-1), minlength=256), exempt_any=bool(exempt.any()))
    rep["ok"] = not set_mm and not order_err and not tie_err and gate_err <= GATE_TOL
    return rep


def check_counts(ref_all, idx_gpu, counts_gpu):
    """Counts: exactly the oracle's when no token is exempt; in general exactly the counts
    of the GPU's own choices, which must agree with the oracle's on every non-exempt token
    (checked by compare)."""
    idx_g = idx_gpu.detach().cpu().numpy()
    c_g = counts_gpu.detach().cpu().numpy()
    own = np.bincount(idx_g.reshape(-1), minlength=256)
    ok = np.array_equal(c_g, own)
    if ref_all is not None and not (ref_all["gaps"][:, 5] <= GAP).any():
        ok = ok and np.array_equal(c_g, np.bincount(ref_all["idx"].reshape(-1), minlength=256))
    return ok


def nvfp4_host_layer(w, q, experts):
    """The oracle's layer for NVFP4 expert weights: the router and bias of ``w`` (bf16 weights
    dict) and, for the given routed experts and the shared expert, the dequantised NVFP4 values
    (oracle.nvfp4_dequant; bf16-exact with the generator's power-of-two tensor scales)."""
    def dq(codes, scales, ts):
        return oracle.f64_to_bf16_exact(oracle.nvfp4_dequant(codes.cpu().numpy(), scales.cpu().numpy(), float(ts)))

    wr = to_np_bf16(w["w_router"])
    b = None if w.get("router_bias") is None else w["router_bias"].detach().float().cpu().numpy()
    routed = {}
    for name in ("w_gate", "w_up", "w_down"):
        c, s, t = q[name]
        routed[name] = {int(e): dq(c[int(e)], s[int(e)], t[int(e)].item()) for e in experts}
    shared = {name: dq(*q[name]) for name in ("ws_gate", "ws_up", "ws_down")}
    return oracle.Layer(wr, routed["w_gate"], routed["w_up"], routed["w_down"], shared["ws_gate"], shared["ws_up"],
                        shared["ws_down"], router_bias=b, k=6)


def oracle_reference_nvfp4(w, q, x, tokens, nthreads=ORACLE_THREADS, residual=False, eps=None):
    """oracle_reference for a layer on NVFP4 expert weights ``q`` (router from ``w``)."""
    x64 = oracle.bf16_to_f64(to_np_bf16(x))
    tokens = np.asarray(tokens, dtype=np.int64)
    xin = x64 if eps is None else oracle.prenorm_input(x64, eps)
    experts = touched_experts(w, xin, tokens)
    layer = nvfp4_host_layer(w, q, experts)
    out = oracle.forward(layer, xin[tokens], nthreads=nthreads, want_scores=True)
    if residual:
        out["y"] = x64[tokens] + out["y"]
    out["tokens"] = tokens
    out["layer"] = layer
    out["xin"] = xin[tokens]
    out["xres"] = x64[tokens] if residual else None
    return out
