"""Plain CPU oracle for the forward pass of a top-K routed Mixture-of-Experts
SwiGLU FFN layer with always-on shared experts.

TEST INFRASTRUCTURE ONLY. The product path never imports, calls or runs this
module; only the tests, the smoke check in ``__graft_entry__`` and the
``cpu_baseline`` / reference leg of ``bench.py`` use it. It shares no code
with the CUDA library (no kernels, headers, tables or helpers).

Arithmetic is float64 on the exact input values (BF16 and FP32 inputs convert
to float64 without rounding), with NumPy's matmul and sort as the only library
steps. The exception is the quantile bias update, whose page works on FP32
scores; it is written in FP32 where the page computes in FP32.

Sources, cited as page title + section:

* [APEX-MoE] APEX-1 docs "10 - Mixture of Experts", class ``MoEFFN``: router
  Linear without bias, expert bias added to the scores, top-K, softmax over
  the selected scores, per-expert dispatch, shared experts on every token.
* [APEX-M3] APEX-1 Mathematical Reference Part 3: section 12 (SwiGLU FFN,
  SiLU), section 13 (MoE output, router, routing weights), section 14
  (bias-based load balancing).
* [K3-SLM] kimi_k3 "StableLatentMoE and QuantileBalancer": FP32 sigmoid router,
  top-(K+1) of bias-corrected scores, weights from uncorrected scores, stable
  argsort dispatch, latent down/up projections, quantile balancer update.
* [MoE-FS] "MoE from scratch" tutorial ("A working MoE layer in PyTorch"):
  ``SwiGLU``, ``MoELayer`` (softmax over all experts, top-K, renormalise,
  sorted dispatch, Switch load-balancing loss) and its ``naive_forward``
  reference.
* [BOOK-MoE] book-ai "Mixture of Experts" chapter, class ``MoELoss``:
  ``router_z_loss`` (ST-MoE z-loss).

Readings where the pages are silent or disagree:
ties in top-K go to the lower expert index; slot k holds the k-th largest
score; in the softmax modes the balance bias is added to the logits before
the score; the quantile rank is computed in FP32 as the FP32 quantile would;
the mean in the bias update is a sequential float64 sum rounded once to FP32.

Every function here is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import math

import numpy as np

GATE_SOFTMAX_TOPK = "softmax_topk"
GATE_SOFTMAX_ALL_RENORM = "softmax_all_renorm"
GATE_SIGMOID = "sigmoid"


def f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# SwiGLU expert  [APEX-M3] section 12.2-12.3; [MoE-FS] class SwiGLU
# --------------------------------------------------------------------------

def sigmoid(a):
    """sigma(a) = 1 / (1 + e^-a)."""
    a = f64(a)
    return 1.0 / (1.0 + np.exp(-a))


def silu(a):
    """SiLU(a) = a * sigma(a) = a / (1 + e^-a)  ([APEX-M3] section 12.3)."""
    a = f64(a)
    return a / (1.0 + np.exp(-a))


def swiglu_hidden(x, W_gate, W_up):
    """SiLU(x W_gate) (elementwise *) (x W_up): the gated hidden vector of
    section 12.2, for one token x [d] or a row block x [n, d]."""
    x = f64(x)
    return silu(x @ f64(W_gate)) * (x @ f64(W_up))


def swiglu_ffn(x, W_gate, W_up, W_down):
    """FFN(x) = W_down( SiLU(x W_gate) * (x W_up) )  ([APEX-M3] section 12.2).

    W_gate, W_up are [d, d_ff]; W_down is [d_ff, d]; x is [d] or [n, d].
    """
    return swiglu_hidden(x, W_gate, W_up) @ f64(W_down)


# --------------------------------------------------------------------------
# Router  [APEX-MoE] steps 2-3; [APEX-M3] section 13.2 and 13.5;
#         [MoE-FS] MoELayer.forward; [K3-SLM] "FP32 router and training-only QB update"
# --------------------------------------------------------------------------

def rank_experts(c):
    """Expert ids ordered by score descending; among equal scores the lower
    expert id comes first (the tie-break the library and this oracle share)."""
    c = f64(c)
    return np.argsort(-c, axis=-1, kind="stable")


def route_from_logits(r, bias, gate, K, renormalize=False, routed_scale=1.0):
    """Route one token from its router logits r [E].

    Returns a dict with
      idx [K]        selected experts, slot k = k-th largest selection score
      w [K]          gate weights
      margin         c_(K) - c_(K+1): selection score at rank K minus rank K+1
                     (1-based; +inf when K == E)
      min_gap        smallest gap between consecutive ranked scores among the
                     first min(K+1, E): how close the selection or the slot
                     order came to a tie
      score [E]      the selection score c the ranking used
      s [E]          sigmoid scores (sigmoid mode only)
      top_scores     [K+1] the K+1 largest c, descending (sigmoid mode only)

    Modes:
      softmax_topk        c = r + b; top-K of c; g = softmax over the K selected
                          c ([APEX-MoE] step 3, [APEX-M3] section 13.2)
      softmax_all_renorm  p = softmax over all E of (r + b); top-K of p;
                          g = p_sel / sum p_sel ([MoE-FS] MoELayer)
      sigmoid             s = sigma(r); c = s + b; top-(K+1) of c, the first K
                          used; g = s at the selected experts (uncorrected),
                          optionally divided by its sum, times routed_scale
                          ([K3-SLM] "FP32 router ..." and "Flatten routing ...")
    """
    r = f64(r)
    E = r.shape[0]
    b = np.zeros(E) if bias is None else f64(bias)
    out = {}
    if gate == GATE_SOFTMAX_TOPK:
        c = r + b
        order = rank_experts(c)
        idx = order[:K]
        sel = c[idx]
        ex = np.exp(sel - sel[0])
        w = ex / ex.sum()
    elif gate == GATE_SOFTMAX_ALL_RENORM:
        z = r + b
        ez = np.exp(z - z.max())
        p = ez / ez.sum()
        c = p
        order = rank_experts(c)
        idx = order[:K]
        w = p[idx] / p[idx].sum()
    elif gate == GATE_SIGMOID:
        s = sigmoid(r)
        c = s + b
        order = rank_experts(c)
        top = order[:K + 1]
        out["top_scores"] = c[top]
        out["s"] = s
        idx = top[:K]
        w = s[idx].copy()
        if renormalize:
            w = w / w.sum()
        w = w * routed_scale
    else:
        raise ValueError(f"unknown gate mode {gate!r}")
    out["idx"] = idx.astype(np.int64)
    out["w"] = w
    out["score"] = c
    out["margin"] = (c[order[K - 1]] - c[order[K]]) if K < E else math.inf
    top = c[order[:min(K + 1, E)]]
    out["min_gap"] = float(np.min(top[:-1] - top[1:])) if top.shape[0] > 1 else math.inf
    return out


def router_logits(x, W_router):
    """r = x W_router, FP32 inputs taken exactly, summed in float64
    ([APEX-M3] section 13.2; [K3-SLM] F.linear on FP32 copies)."""
    return f64(x) @ f64(W_router)


def route(x, W_router, bias, gate, K, renormalize=False, routed_scale=1.0):
    """Route every token of x [T, d]. Returns stacked arrays:
    idx [T, K] int64, w [T, K], margin [T], and for sigmoid mode
    top_scores [T, K+1] and s [T, E]."""
    r = router_logits(x, W_router)
    T = r.shape[0]
    per = [route_from_logits(r[t], bias, gate, K, renormalize, routed_scale)
           for t in range(T)]
    res = {
        "logits": r,
        "idx": np.stack([p["idx"] for p in per]) if T else np.zeros((0, K), np.int64),
        "w": np.stack([p["w"] for p in per]) if T else np.zeros((0, K)),
        "margin": np.array([p["margin"] for p in per], dtype=np.float64),
        "min_gap": np.array([p["min_gap"] for p in per], dtype=np.float64),
    }
    if gate == GATE_SIGMOID:
        res["top_scores"] = np.stack([p["top_scores"] for p in per])
        res["s"] = np.stack([p["s"] for p in per])
    return res


def gates_for(r, bias, gate, idx, renormalize=False, routed_scale=1.0):
    """Gate weights of one token for a GIVEN expert selection idx [K] (in slot
    order). Used when the oracle adopts another router's selection for a
    near-tie token: the weights follow the same formulas as route_from_logits."""
    r = f64(r)
    E = r.shape[0]
    b = np.zeros(E) if bias is None else f64(bias)
    idx = np.asarray(idx, dtype=np.int64)
    if gate == GATE_SOFTMAX_TOPK:
        sel = (r + b)[idx]
        ex = np.exp(sel - sel.max())
        return ex / ex.sum()
    if gate == GATE_SOFTMAX_ALL_RENORM:
        z = r + b
        ez = np.exp(z - z.max())
        p = ez / ez.sum()
        return p[idx] / p[idx].sum()
    if gate == GATE_SIGMOID:
        w = sigmoid(r)[idx]
        if renormalize:
            w = w / w.sum()
        return w * routed_scale
    raise ValueError(gate)


# --------------------------------------------------------------------------
# Sorted dispatch  [K3-SLM] "Flatten routing and recover original token order",
#                  "Dispatch is a stable permutation"; [MoE-FS] MoELayer.forward
# --------------------------------------------------------------------------

def dispatch(idx, E):
    """Stable grouping of the T*K assignments by expert id.

    Flat assignment j = t*K + k has expert idx[t, k]. A stable argsort of the
    flat ids, written as a counting sort over j in ascending order, gives
    order[pos] = j. Returns
      counts [E]        assignments per expert (the bincount)
      offsets [E+1]     exclusive prefix sum of counts (offsets[E] = T*K)
      order [T*K]       flat index j placed at each sorted position
      sorted_token [T*K] = order // K
      sorted_slot [T*K]  = order %  K
      inv [T, K]        sorted position of assignment (t, k)
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, K = idx.shape
    flat = idx.reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:E].copy()
    order = np.empty(T * K, dtype=np.int64)
    inv = np.empty(T * K, dtype=np.int64)
    for j in range(T * K):
        e = flat[j]
        order[fill[e]] = j
        inv[j] = fill[e]
        fill[e] += 1
    return {
        "counts": counts,
        "offsets": offsets,
        "order": order,
        "sorted_token": order // K,
        "sorted_slot": order % K,
        "inv": inv.reshape(T, K),
    }


# --------------------------------------------------------------------------
# Layer forward  [APEX-M3] section 13.2; [APEX-MoE] steps 4-5;
#                [MoE-FS] naive_forward; [K3-SLM] "Return to model width"
# --------------------------------------------------------------------------

class _WeightCache:
    """float64 copies of expert matrices, made on first use; at most
    max_entries are kept (least recently used dropped) so that large layers
    can be sampled token by token with bounded host memory."""

    def __init__(self, params, max_entries=48):
        self.p = params
        self.c = {}
        self.max_entries = max_entries

    def get(self, name, i=None):
        key = (name, i)
        if key in self.c:
            v = self.c.pop(key)
            self.c[key] = v
            return v
        a = self.p[name]
        a = a if i is None else a[i]
        if hasattr(a, "detach"):
            a = a.detach().float().cpu().numpy()
        v = f64(a)
        self.c[key] = v
        while len(self.c) > self.max_entries:
            self.c.pop(next(iter(self.c)))
        return v


def _to_np(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        return a.detach().float().cpu().numpy()
    return np.asarray(a)


def moe_forward_token(xt, idx_t, w_t, params, cache=None):
    """Output of one token x_t [d] given its selected experts and weights:

        MoE(x) = sum_s Shared_s(x) + sum_k g_k Expert_{e_k}(x)

    ([APEX-M3] section 13.2). In the latent variant the routed experts act on
    z = x W_down_latent and the routed sum is projected back by W_up_latent
    before it is added to the shared output ([K3-SLM] "Return to model width").
    """
    cache = cache or _WeightCache(params)
    xt = f64(xt)
    latent = params.get("W_down_latent") is not None
    zt = xt @ cache.get("W_down_latent") if latent else xt
    routed = np.zeros(zt.shape[0])
    for k in range(len(idx_t)):
        e = int(idx_t[k])
        routed = routed + w_t[k] * swiglu_ffn(zt, cache.get("W_gate", e), cache.get("W_up", e),
                                              cache.get("W_down", e))
    if latent:
        routed = routed @ cache.get("W_up_latent")
    shared = np.zeros(xt.shape[0])
    if params.get("Ws_gate") is not None:
        for s in range(params["Ws_gate"].shape[0]):
            shared = shared + swiglu_ffn(xt, cache.get("Ws_gate", s), cache.get("Ws_up", s),
                                         cache.get("Ws_down", s))
    return shared + routed


def moe_forward(x, params, gate, K, renormalize=False, routed_scale=1.0,
                tokens=None, routing=None):
    """Per-token forward of the whole layer (the naive reference shape).

    x [T, d]; params: dict with W_router, bias, W_gate, W_up, W_down, Ws_*,
    W_down_latent, W_up_latent (torch tensors or arrays). ``tokens`` restricts
    the computed rows (others are left NaN). ``routing`` = (idx [T, K], w [T, K])
    replaces the oracle's own routing (used for near-tie tokens only).
    Returns (out [T, d] float64, routing dict of the oracle's own route()).
    """
    xn = _to_np(x)
    T = xn.shape[0]
    rows = range(T) if tokens is None else tokens
    sub = np.asarray(list(rows), dtype=np.int64)
    rt = route(xn[sub], _to_np(params["W_router"]), _to_np(params.get("bias")), gate, K,
               renormalize, routed_scale)
    idx, w = rt["idx"], rt["w"]
    if routing is not None:
        idx = np.asarray(routing[0])[sub]
        w = np.asarray(routing[1])[sub]
    cache = _WeightCache(params)
    out = np.full((T, xn.shape[1]), np.nan)
    for i, t in enumerate(sub):
        out[t] = moe_forward_token(xn[t], idx[i], w[i], params, cache)
    return out, rt


def moe_forward_sorted(x, params, gate, K, renormalize=False, routed_scale=1.0,
                       tokens=None, routing=None):
    """Second formulation of the same layer: group the assignments with
    dispatch(), run each expert once on its contiguous block of rows, weight
    the rows, and scatter-add them back to their tokens ([MoE-FS]
    MoELayer.forward; [K3-SLM] grouped execution semantics). Pinned equal to
    the per-token form; it reads each expert's weights once, which makes
    whole large layers affordable on the CPU.

    ``tokens`` and ``routing`` work as in moe_forward: only the listed rows are
    computed (the others are NaN), and ``routing`` = (idx [T, K], w [T, K])
    replaces the oracle's own routing. Returns out [T, d] float64.
    """
    xn = f64(_to_np(x))
    T = xn.shape[0]
    sub = np.arange(T, dtype=np.int64) if tokens is None else np.asarray(list(tokens), np.int64)
    rt = route(xn[sub], _to_np(params["W_router"]), _to_np(params.get("bias")), gate, K,
               renormalize, routed_scale)
    idx, w = rt["idx"], rt["w"]
    if routing is not None:
        idx = np.asarray(routing[0])[sub]
        w = f64(np.asarray(routing[1])[sub])
    E = params["W_gate"].shape[0]
    dp = dispatch(idx, E)
    cache = _WeightCache(params)
    latent = params.get("W_down_latent") is not None
    xsub = xn[sub]
    z = xsub @ cache.get("W_down_latent") if latent else xsub
    xs = z[dp["sorted_token"]]
    ws = w.reshape(-1)[dp["order"]]
    ys = np.zeros_like(xs)
    for e in range(E):
        a, b = dp["offsets"][e], dp["offsets"][e + 1]
        if b > a:
            ys[a:b] = swiglu_ffn(xs[a:b], cache.get("W_gate", e), cache.get("W_up", e),
                                 cache.get("W_down", e))
    ys = ys * ws[:, None]
    routed = np.zeros_like(z)
    np.add.at(routed, dp["sorted_token"], ys)
    if latent:
        routed = routed @ cache.get("W_up_latent")
    shared = np.zeros_like(xsub)
    if params.get("Ws_gate") is not None:
        for s in range(params["Ws_gate"].shape[0]):
            shared = shared + swiglu_ffn(xsub, cache.get("Ws_gate", s), cache.get("Ws_up", s),
                                         cache.get("Ws_down", s))
    out = np.full((T, xn.shape[1]), np.nan)
    out[sub] = shared + routed
    return out


# --------------------------------------------------------------------------
# Balancers
# --------------------------------------------------------------------------

def quantile_rank(T, E, K):
    """0-based sorted index that the 'higher' quantile at p = K/E picks from
    T values: ceil(p * (T - 1)), with p and the product in FP32 as the FP32
    quantile computes them ([K3-SLM] QuantileBalancer.update)."""
    p = np.float32(K / E)
    return int(math.ceil(float(np.float32(p * np.float32(T - 1)))))


def quantile_bias_update(top_scores, scores, K):
    """New balance biases [E] FP32 ([K3-SLM] "QuantileBalancer: persistent
    biases, no gradient update"):

      thresh_t = top_scores[t, K]          the (K+1)-th corrected score
      rel[t, j] = thresh_t - s[t, j]       FP32 subtraction
      b_j = 'higher' quantile p = K/E of rel[:, j] over the T tokens
      b = b - mean(b)

    The quantile is the value at sorted index quantile_rank(T, E, K). The mean
    is a sequential float64 sum over j, divided by E and rounded once to FP32;
    the centring subtraction is FP32.
    """
    ts = np.asarray(top_scores, dtype=np.float32)
    s = np.asarray(scores, dtype=np.float32)
    T, E = s.shape
    thresh = ts[:, K]
    rel = (thresh[:, None] - s).astype(np.float32)
    q = quantile_rank(T, E, K)
    b = np.empty(E, dtype=np.float32)
    for j in range(E):
        b[j] = np.sort(rel[:, j], kind="stable")[q]
    acc = 0.0
    for j in range(E):
        acc += float(b[j])
    mean = np.float32(acc / E)
    return (b - mean).astype(np.float32)


def sign_bias_update(counts, N, K, bias, alpha):
    """Bias-based balancing ([APEX-M3] section 14.3): f_e = c_e / (N K),
    tau = 1/E, b_e <- clamp(b_e + alpha * sign(tau - f_e), -1, 1)."""
    c = f64(counts)
    E = c.shape[0]
    f = c / (N * K)
    tau = 1.0 / E
    b = f64(bias) + alpha * np.sign(tau - f)
    return np.clip(b, -1.0, 1.0)


# --------------------------------------------------------------------------
# Routing diagnostics  [MoE-FS] MoELayer.forward (Switch load-balancing loss);
#                      [BOOK-MoE] MoELoss.router_z_loss
# --------------------------------------------------------------------------

def routing_stats(r, idx, E):
    """Diagnostics of one batch's routing from the raw router logits r [T, E]
    (x W_router, no balance bias) and the selected experts idx [T, K]:

      P_e  = (1/T) sum_t softmax(r_t)_e         mean router probability
      f_e  = #{(t, k): idx[t, k] = e} / (T K)    share of the assignments
      aux  = E * sum_e f_e P_e                   Switch loss before its alpha
      z    = (1/T) sum_t (log sum_e exp r_te)^2  z-loss before its weight

    Returns dict(aux, z, P, f)."""
    r = f64(r)
    idx = np.asarray(idx)
    T = r.shape[0]
    K = idx.shape[1]
    m = r.max(axis=1, keepdims=True)
    ex = np.exp(r - m)
    p = ex / ex.sum(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(ex.sum(axis=1))
    P = p.mean(axis=0)
    f = np.bincount(idx.reshape(-1), minlength=E).astype(np.float64) / (T * K)
    return {"aux": float(E * np.sum(f * P)), "z": float(np.mean(lse ** 2)), "P": P, "f": f}


# --------------------------------------------------------------------------
# Backward pass  [K3-SLM] "The actual grouped GEMM, and the gradient path",
#                "Grouped expert execution and sparse gradients";
#                [APEX-M3] sections 12.2-12.3 and 13.2 (the forward it differentiates)
# --------------------------------------------------------------------------

def silu_grad(a):
    """d SiLU(a) / da = sigma(a) (1 + a (1 - sigma(a)))."""
    a = f64(a)
    s = sigmoid(a)
    return s * (1.0 + a * (1.0 - s))


def gate_logit_grad(r, bias, gate, idx, dw, renormalize=False, routed_scale=1.0):
    """dL/dr [E] of one token from dL/dg [K], the selection idx held fixed
    (top-K indices carry no gradient; [K3-SLM] "The actual grouped GEMM, and
    the gradient path"). The chain rule through each mode's own formula:

      softmax_topk        g = softmax over the selected c = r + b
      softmax_all_renorm  p = softmax over all E of r + b, g = p_sel / sum p_sel
      sigmoid             s = sigma(r), g = scale * s_sel (/ sum s_sel)
    The balance bias is a buffer without gradient."""
    r = f64(r)
    E = r.shape[0]
    b = np.zeros(E) if bias is None else f64(bias)
    idx = np.asarray(idx, dtype=np.int64)
    dw = f64(dw)
    dr = np.zeros(E)
    if gate == GATE_SOFTMAX_TOPK:
        sel = (r + b)[idx]
        ex = np.exp(sel - sel.max())
        g = ex / ex.sum()
        dr[idx] += g * (dw - np.dot(g, dw))
    elif gate == GATE_SOFTMAX_ALL_RENORM:
        z = r + b
        ez = np.exp(z - z.max())
        p = ez / ez.sum()
        P = p[idx].sum()
        g = p[idx] / P
        dp = np.zeros(E)
        dp[idx] = (dw - np.dot(dw, g)) / P
        dr = p * (dp - np.dot(p, dp))
    elif gate == GATE_SIGMOID:
        s = sigmoid(r)
        ds = np.zeros(E)
        if renormalize:
            S = s[idx].sum()
            ds[idx] = routed_scale * (dw - np.dot(dw, s[idx]) / S) / S
        else:
            ds[idx] = routed_scale * dw
        dr = ds * s * (1.0 - s)
    else:
        raise ValueError(gate)
    return dr


def round_bf16(a):
    """Rounds to FP32 (nearest-even), then to BF16 (nearest-even on the FP32
    bits: add 0x7FFF plus the kept lsb, drop the low 16 bits), returned as
    float64. Finite inputs."""
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def moe_backward(x, params, dout, gate, K, renormalize=False, routed_scale=1.0, routing=None,
                 latent_rows_bf16=False, tokens=None):
    """Gradients of L = sum(dout * out) for the layer of moe_forward, the
    routing (selection) held fixed. Per token and per selected expert, the
    chain rule of

        a = z W_gate[e], u = z W_up[e], h = SiLU(a) * u, y = h W_down[e]
        out = sum_k g_k y_k (latent: projected by W_up_latent) + shared(x)

    with z = x (latent: x W_down_latent) and g from the router logits
    x W_router (gate_logit_grad). ``routing`` = (idx [T, K]) replaces the
    oracle's own selection (near ties); the weights are recomputed from the
    logits either way.

    Experts that no token selects get no gradient ([K3-SLM] "Grouped expert
    execution and sparse gradients": inactive experts stay outside autograd):
    their entries of dW_gate / dW_up / dW_down are zero and ``active`` [E] is
    False for them. Returns a dict of float64 arrays: dx, dW_router, dW_gate,
    dW_up, dW_down, dWs_gate, dWs_up, dWs_down (or None), dW_down_latent,
    dW_up_latent (or None), active, dw [T, K] (dL/dg).

    latent_rows_bf16: the latent rows z are rounded to BF16 (round_bf16)
    before the experts use them, as a BF16 layer stores its activations; the
    derivative of that rounding is taken as 1.

    tokens: only these tokens are processed (large layers sampled token by
    token): their rows of dx and dw are complete, the other rows are zero,
    and the weight gradients hold only these tokens' terms."""
    xn = f64(_to_np(x))
    g_out = f64(_to_np(dout))
    T, d = xn.shape
    Wr = f64(_to_np(params["W_router"]))
    bias = _to_np(params.get("bias"))
    bias = None if bias is None else f64(bias)
    cache = _WeightCache(params, max_entries=10 ** 6 if tokens is None else 48)
    E = params["W_gate"].shape[0]
    rows = range(T) if tokens is None else [int(t) for t in tokens]
    r = np.zeros((T, Wr.shape[1]))
    for t in rows:
        r[t] = xn[t] @ Wr
    if routing is None:
        idx = np.zeros((T, K), dtype=np.int64)
        for t in rows:
            idx[t] = route_from_logits(r[t], bias, gate, K, renormalize, routed_scale)["idx"]
    else:
        idx = np.asarray(routing, dtype=np.int64)
    latent = params.get("W_down_latent") is not None
    Wdl = cache.get("W_down_latent") if latent else None
    Wul = cache.get("W_up_latent") if latent else None
    de = Wdl.shape[1] if latent else d
    F = params["W_gate"].shape[2]
    out = {
        "dx": np.zeros((T, d)), "dW_router": np.zeros_like(Wr),
        "dW_gate": np.zeros((E, de, F)), "dW_up": np.zeros((E, de, F)),
        "dW_down": np.zeros((E, F, de)), "active": np.zeros(E, dtype=bool),
        "dw": np.zeros((T, K)),
    }
    shared = params.get("Ws_gate") is not None
    if shared:
        S, _, Fs = params["Ws_gate"].shape
        out["dWs_gate"] = np.zeros((S, d, Fs))
        out["dWs_up"] = np.zeros((S, d, Fs))
        out["dWs_down"] = np.zeros((S, Fs, d))
    else:
        out["dWs_gate"] = out["dWs_up"] = out["dWs_down"] = None
    out["dW_down_latent"] = np.zeros_like(Wdl) if latent else None
    out["dW_up_latent"] = np.zeros_like(Wul) if latent else None

    def ffn_backward(zt, gy, Wg, Wu, Wd):
        """(y, dWg, dWu, dWd, dz) of one SwiGLU expert at one row, upstream gy."""
        a = zt @ Wg
        u = zt @ Wu
        h = silu(a) * u
        y = h @ Wd
        dh = gy @ Wd.T
        da = dh * u * silu_grad(a)
        du = dh * silu(a)
        return y, np.outer(zt, da), np.outer(zt, du), np.outer(h, gy), da @ Wg.T + du @ Wu.T

    for t in rows:
        xt = xn[t]
        zt = xt @ Wdl if latent else xt
        if latent and latent_rows_bf16:
            zt = round_bf16(zt)
        w_t = gates_for(r[t], bias, gate, idx[t], renormalize, routed_scale)
        gt = g_out[t]
        g_lat = gt @ Wul.T if latent else gt
        dz = np.zeros(de)
        routed = np.zeros(de)
        dw = np.zeros(K)
        for k in range(K):
            e = int(idx[t, k])
            out["active"][e] = True
            y, dWg, dWu, dWd, dzk = ffn_backward(zt, w_t[k] * g_lat, cache.get("W_gate", e),
                                                 cache.get("W_up", e), cache.get("W_down", e))
            # y here is the expert output for upstream w_k * g: the unweighted output
            # is the same y (it does not depend on the upstream gradient)
            routed = routed + w_t[k] * y
            dw[k] = np.dot(g_lat, y)
            out["dW_gate"][e] += dWg
            out["dW_up"][e] += dWu
            out["dW_down"][e] += dWd
            dz = dz + dzk
        out["dw"][t] = dw
        if latent:
            out["dW_up_latent"] += np.outer(routed, gt)
            out["dW_down_latent"] += np.outer(xt, dz)
            dxt = dz @ Wdl.T
        else:
            dxt = dz
        if shared:
            for s in range(S):
                _, dWg, dWu, dWd, dzs = ffn_backward(xt, gt, cache.get("Ws_gate", s),
                                                     cache.get("Ws_up", s), cache.get("Ws_down", s))
                out["dWs_gate"][s] += dWg
                out["dWs_up"][s] += dWu
                out["dWs_down"][s] += dWd
                dxt = dxt + dzs
        dr = gate_logit_grad(r[t], bias, gate, idx[t], dw, renormalize, routed_scale)
        out["dW_router"] += np.outer(xt, dr)
        out["dx"][t] = dxt + dr @ Wr.T
    return out
