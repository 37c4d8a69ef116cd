"""The oracle against its pins, and the pins against planted oracle mistakes.

CPU only. A planted mistake is made in a private copy of the oracle module;
each one must make at least one pin fail, which shows the pins would catch
that kind of error in the oracle itself.
"""
import importlib.util
import math
import os

import numpy as np
import pytest

from tests import oracle_pins as P
from oracle import moe_oracle

ORACLE_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "moe_oracle.py")


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(moe_oracle)


def fresh_oracle():
    spec = importlib.util.spec_from_file_location("moe_oracle_mutant", ORACLE_PATH)
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _mut_silu_sign(m):
    m.silu = lambda a: np.asarray(a, float) / (1.0 + np.exp(np.asarray(a, float)))


def _mut_gate_up_swapped(m):
    orig = m.swiglu_hidden
    m.swiglu_hidden = lambda x, Wg, Wu: orig(x, Wu, Wg)


def _mut_down_transposed(m):
    def ffn(x, Wg, Wu, Wd):
        h = m.swiglu_hidden(x, Wg, Wu)
        Wd = np.asarray(Wd, float)
        return h @ (Wd.T if Wd.shape[0] == Wd.shape[1] else Wd[::-1])
    m.swiglu_ffn = ffn


def _mut_softmax_over_all(m):
    orig = m.route_from_logits

    def route(r, bias, gate, K, renormalize=False, routed_scale=1.0):
        out = orig(r, bias, gate, K, renormalize, routed_scale)
        if gate == m.GATE_SOFTMAX_TOPK:
            c = np.asarray(r, float) + (0 if bias is None else np.asarray(bias, float))
            ez = np.exp(c - c.max())
            out["w"] = (ez / ez.sum())[out["idx"]]
        return out
    m.route_from_logits = route


def _mut_tie_to_higher(m):
    def rank(c):
        c = np.asarray(c, float)
        n = c.shape[-1]
        return (n - 1 - np.argsort(-c[..., ::-1], axis=-1, kind="stable"))
    m.rank_experts = rank


def _mut_dispatch_unstable(m):
    orig = m.dispatch

    def dispatch(idx, E):
        dp = orig(idx, E)
        order = dp["order"].copy()
        for e in range(E):
            a, b = dp["offsets"][e], dp["offsets"][e + 1]
            order[a:b] = order[a:b][::-1]
        K = np.asarray(idx).shape[1]
        dp["order"], dp["sorted_token"] = order, order // K
        return dp
    m.dispatch = dispatch


def _mut_drop_shared(m):
    orig = m.moe_forward_token

    def tok(xt, idx_t, w_t, params, cache=None):
        p = dict(params, Ws_gate=None)
        return orig(xt, idx_t, w_t, p, None)
    m.moe_forward_token = tok


def _mut_sigmoid_corrected_weights(m):
    orig = m.route_from_logits

    def route(r, bias, gate, K, renormalize=False, routed_scale=1.0):
        out = orig(r, bias, gate, K, renormalize, routed_scale)
        if gate == m.GATE_SIGMOID:
            out["w"] = out["score"][out["idx"]]
        return out
    m.route_from_logits = route


def _mut_quantile_lower(m):
    m.quantile_rank = lambda T, E, K: int(math.floor(K / E * (T - 1)))


def _mut_quantile_no_centre(m):
    orig = m.quantile_bias_update

    def upd(top, s, K):
        b = orig(top, s, K)
        return (b + np.float32(0.25)).astype(np.float32)
    m.quantile_bias_update = upd


def _mut_latent_no_up(m):
    orig = m.moe_forward_token

    def tok(xt, idx_t, w_t, params, cache=None):
        if params.get("W_up_latent") is not None:
            params = dict(params, W_up_latent=np.eye(params["W_up_latent"].shape[0],
                                                     params["W_up_latent"].shape[1]))
        return orig(xt, idx_t, w_t, params, None)
    m.moe_forward_token = tok


def _mut_sign_bias_flipped(m):
    orig = m.sign_bias_update
    m.sign_bias_update = lambda c, N, K, b, a: orig(c, N, K, b, -a)


def _mut_aux_share_over_tokens(m):
    orig = m.routing_stats

    def stats(r, idx, E):
        st = orig(r, idx, E)
        K = np.asarray(idx).shape[1]
        st["aux"] = st["aux"] * K  # f normalised by T instead of T*K
        return st
    m.routing_stats = stats


def _mut_z_not_squared(m):
    orig = m.routing_stats

    def stats(r, idx, E):
        st = orig(r, idx, E)
        rr = np.asarray(r, float)
        st["z"] = float(np.mean(np.log(np.exp(rr).sum(axis=1))))
        return st
    m.routing_stats = stats


def _mut_bwd_silu_grad_short(m):
    m.silu_grad = lambda a: m.sigmoid(a)


def _mut_bwd_gate_grad_sign(m):
    orig = m.gate_logit_grad
    m.gate_logit_grad = lambda *a, **k: -orig(*a, **k)


def _mut_bwd_no_router_grad(m):
    m.gate_logit_grad = lambda r, *a, **k: np.zeros_like(np.asarray(r, float))


def _mut_bwd_gate_up_swapped(m):
    orig = m.moe_backward

    def bwd(*a, **k):
        g = orig(*a, **k)
        g["dW_gate"], g["dW_up"] = g["dW_up"], g["dW_gate"]
        return g
    m.moe_backward = bwd


def _mut_bwd_renorm_ignored(m):
    orig = m.gate_logit_grad

    def ggrad(r, bias, gate, idx, dw, renormalize=False, routed_scale=1.0):
        return orig(r, bias, gate, idx, dw, False, routed_scale)
    m.gate_logit_grad = ggrad


MUTANTS = [_mut_silu_sign, _mut_gate_up_swapped, _mut_down_transposed, _mut_softmax_over_all,
           _mut_tie_to_higher, _mut_dispatch_unstable, _mut_drop_shared,
           _mut_sigmoid_corrected_weights, _mut_quantile_lower, _mut_quantile_no_centre,
           _mut_latent_no_up, _mut_sign_bias_flipped, _mut_aux_share_over_tokens,
           _mut_z_not_squared, _mut_bwd_silu_grad_short, _mut_bwd_gate_grad_sign,
           _mut_bwd_no_router_grad, _mut_bwd_gate_up_swapped, _mut_bwd_renorm_ignored]


@pytest.mark.parametrize("mutate", MUTANTS, ids=lambda f: f.__name__)
def test_planted_mistake_is_caught(mutate):
    m = fresh_oracle()
    pin_ok = [True]
    for pin in P.ALL_PINS:
        mm = fresh_oracle()
        mutate(mm)
        try:
            pin(mm)
        except (AssertionError, ValueError, IndexError):
            pin_ok[0] = False
            break
    assert not pin_ok[0], f"no pin caught {mutate.__name__}"
    del m
