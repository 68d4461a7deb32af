"""Algorithmic byte and FLOP accounting of one Flint-shaped MoE layer.

Shapes: hidden 2048, 256 routed experts with 6 chosen per token, expert width 512,
shared expert width 1024 (Recursive Flint serving-kit post, section "The architecture,
from the config").  Every expert and the shared expert is a SwiGLU MLP with three
matrices (gate, up: hidden x width; down: width x hidden); the router is hidden x experts.

Algorithmic bytes count what the layer must read at least once (the router, the shared
expert and every expert that received at least one token, in bf16) plus the bf16 input
and output rows; intermediates are implementation traffic and are not counted.
"""
from __future__ import annotations

HIDDEN = 2048
N_EXPERTS = 256
TOP_K = 6
EXPERT_INTER = 512
SHARED_INTER = 1024
N_MOE_LAYERS = 47
BF16 = 2


def expert_params(hidden=HIDDEN, inter=EXPERT_INTER):
    return 3 * hidden * inter


def shared_params(hidden=HIDDEN, inter=SHARED_INTER):
    return 3 * hidden * inter


def router_params(hidden=HIDDEN, experts=N_EXPERTS):
    return hidden * experts


def layer_params(hidden=HIDDEN, experts=N_EXPERTS, inter=EXPERT_INTER, shared_inter=SHARED_INTER):
    return experts * expert_params(hidden, inter) + shared_params(hidden, shared_inter) + router_params(hidden, experts)


def layer_weight_bytes(**kw):
    return BF16 * layer_params(**kw)


def active_params_per_token(hidden=HIDDEN, experts=N_EXPERTS, top_k=TOP_K, inter=EXPERT_INTER,
                            shared_inter=SHARED_INTER):
    return top_k * expert_params(hidden, inter) + shared_params(hidden, shared_inter) + router_params(hidden, experts)


def touched_weight_bytes(n_touched_experts, hidden=HIDDEN, experts=N_EXPERTS, inter=EXPERT_INTER,
                         shared_inter=SHARED_INTER):
    """Weights a layer call must stream: every touched expert, the shared expert, the router."""
    return BF16 * (n_touched_experts * expert_params(hidden, inter) + shared_params(hidden, shared_inter)
                   + router_params(hidden, experts))


def algorithmic_bytes(n_touched_experts, tokens, hidden=HIDDEN, **kw):
    """Touched weights plus the bf16 input read and bf16 output write."""
    return touched_weight_bytes(n_touched_experts, hidden=hidden, **kw) + 2 * BF16 * hidden * tokens


def flops_per_token(hidden=HIDDEN, experts=N_EXPERTS, top_k=TOP_K, inter=EXPERT_INTER,
                    shared_inter=SHARED_INTER):
    """2 FLOP per multiply-add: router, k routed SwiGLU experts, the shared SwiGLU expert."""
    return 2 * (router_params(hidden, experts) + top_k * expert_params(hidden, inter)
                + shared_params(hidden, shared_inter))


def expected_touched_experts(tokens, experts=N_EXPERTS, top_k=TOP_K):
    """Mean number of distinct experts hit by ``tokens`` tokens under uniform routing."""
    p_miss = 1.0 - top_k / experts
    return experts * (1.0 - p_miss ** tokens)
