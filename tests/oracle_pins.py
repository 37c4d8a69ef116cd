"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each pin takes the oracle module as an argument so that
test_oracle_pins.py can run it against the real oracle and against copies
with a planted mistake (which must make at least one pin fail).
"""
import json
import math
import os

import numpy as np
import scipy.special

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# -- SwiGLU -----------------------------------------------------------------

def pin_silu_table(o):
    """APEX-1 Math Ref Part 3, section 12.3 table."""
    g = golden("silu_table.json")
    for row in g["rows"]:
        x = row["x"]
        assert abs(float(o.sigmoid(x)) - row["sigma"]) <= g["tolerance"], row
        assert abs(float(o.silu(x)) - row["silu"]) <= g["tolerance"], row
    # SiLU is x * sigma(x): scipy's logistic function as an independent sigma
    xs = np.linspace(-30, 30, 61)
    np.testing.assert_allclose(o.silu(xs), xs * scipy.special.expit(xs), rtol=1e-14, atol=1e-300)


def pin_swiglu_example(o):
    """APEX-1 Math Ref Part 3, section 12.5, with the page's inconsistent
    steps handled as described in the fixture."""
    g = golden("swiglu_example_12_5.json")
    x = np.array(g["x"])
    Wg, Wu = np.array(g["W_gate"]), np.array(g["W_up"])
    # gate[0] is the one printed Step-1 value that follows from the matrices
    gate = x @ Wg
    assert abs(gate[0] - g["page_consistency"]["step1_gate0_exact"]) < 1e-12
    hd = g["hand_derived"]
    h = o.swiglu_hidden(x, Wg, Wu)
    np.testing.assert_allclose(h, hd["hidden"], atol=hd["tolerance"], rtol=0)
    np.testing.assert_allclose(o.silu(np.array(hd["gate"])), hd["silu_gate"],
                               atol=hd["tolerance"], rtol=0)
    # the page's Step 4 is the elementwise product of its Steps 2 and 3
    pr = g["printed"]
    np.testing.assert_allclose(np.array(pr["step2_silu"]) * np.array(pr["step3_up"]),
                               pr["step4_product"], atol=6e-4, rtol=0)


def _down_perm():
    # [d_ff=3, d=4]: out = [h1, 0, h0, 2*h2]
    return np.array([[0.0, 0.0, 1.0, 0.0], [1.0, 0.0, 0.0, 0.0], [0.0, 0.0, 0.0, 2.0]])


def _expected_perm_out():
    hd = golden("swiglu_example_12_5.json")["hand_derived"]["hidden"]
    return np.array([hd[1], 0.0, hd[0], 2.0 * hd[2]])


def pin_ffn_down_projection(o):
    """The down projection multiplies the hidden row vector by W_down [d_ff, d]:
    with a selection matrix the output is a known rearrangement of the
    hand-derived section 12.5 hidden vector."""
    g = golden("swiglu_example_12_5.json")
    x = np.array(g["x"])
    y = o.swiglu_ffn(x, np.array(g["W_gate"]), np.array(g["W_up"]), _down_perm())
    np.testing.assert_allclose(y, _expected_perm_out(), atol=4e-6, rtol=0)
    # a batch of rows is processed row by row
    yb = o.swiglu_ffn(np.stack([x, 2 * x]), np.array(g["W_gate"]), np.array(g["W_up"]),
                      _down_perm())
    np.testing.assert_allclose(yb[0], y, rtol=1e-15, atol=0)


# -- Router -------------------------------------------------------------------

def pin_router_example(o):
    """APEX-1 Math Ref Part 3, section 13.5."""
    g = golden("router_example_13_5.json")
    rt = o.route_from_logits(np.array(g["logits"]), np.array(g["bias"]), o.GATE_SOFTMAX_TOPK,
                             g["K"])
    assert list(rt["idx"]) == g["top_idx"]
    np.testing.assert_allclose(rt["w"], g["weights"], atol=g["tolerance"], rtol=0)
    assert abs(rt["margin"] - (0.8 - 0.1)) < 1e-12


def pin_tie_break(o):
    """Equal scores: the lower expert id ranks first; slot order is descending."""
    c = np.array([1.0, 3.0, 3.0, 0.0, 3.0])
    for gate in (o.GATE_SOFTMAX_TOPK, o.GATE_SOFTMAX_ALL_RENORM):
        assert list(o.route_from_logits(c, None, gate, 1)["idx"]) == [1]
        assert list(o.route_from_logits(c, None, gate, 2)["idx"]) == [1, 2]
        assert list(o.route_from_logits(c, None, gate, 4)["idx"]) == [1, 2, 4, 0]
        assert o.route_from_logits(c, None, gate, 2)["margin"] == 0.0
    assert list(o.rank_experts(np.array([2.0, 2.0, 2.0]))) == [0, 1, 2]


def pin_gate_formulas(o):
    """Gate weights against scipy's softmax / logistic on random logits."""
    rng = np.random.default_rng(1)
    for _ in range(20):
        E = int(rng.integers(3, 40))
        K = int(rng.integers(1, E - 1))
        r = rng.normal(size=E)
        b = rng.normal(scale=0.1, size=E)
        # softmax over the selected biased scores
        rt = o.route_from_logits(r, b, o.GATE_SOFTMAX_TOPK, K)
        c = r + b
        assert set(rt["idx"]) == set(np.argsort(-c)[:K])
        np.testing.assert_allclose(rt["w"], scipy.special.softmax(c[rt["idx"]]), rtol=1e-13)
        assert abs(rt["w"].sum() - 1) < 1e-13
        assert np.all(np.diff(c[rt["idx"]]) <= 0)
        # renormalised full softmax == softmax over the selected logits (identity)
        ra = o.route_from_logits(r, None, o.GATE_SOFTMAX_ALL_RENORM, K)
        assert set(ra["idx"]) == set(np.argsort(-r)[:K])
        np.testing.assert_allclose(ra["w"], scipy.special.softmax(r[ra["idx"]]), rtol=1e-12)
        assert abs(ra["w"].sum() - 1) < 1e-13
        # sigmoid: selection on s + b, weights the uncorrected s
        rs = o.route_from_logits(r, b, o.GATE_SIGMOID, K)
        s = scipy.special.expit(r)
        cs = s + b
        top = np.argsort(-cs)[:K + 1]
        assert list(rs["idx"]) == list(top[:K])
        np.testing.assert_allclose(rs["top_scores"], cs[top], rtol=1e-14)
        np.testing.assert_allclose(rs["w"], s[top[:K]], rtol=1e-14)
        assert np.all((rs["w"] > 0) & (rs["w"] < 1))
        rn = o.route_from_logits(r, b, o.GATE_SIGMOID, K, renormalize=True, routed_scale=2.5)
        np.testing.assert_allclose(rn["w"], 2.5 * s[top[:K]] / s[top[:K]].sum(), rtol=1e-13)
        # gates_for reproduces the router's own weights for its own selection
        for gate, rr, bb in ((o.GATE_SOFTMAX_TOPK, r, b), (o.GATE_SOFTMAX_ALL_RENORM, r, None),
                             (o.GATE_SIGMOID, r, b)):
            own = o.route_from_logits(rr, bb, gate, K)
            np.testing.assert_allclose(o.gates_for(rr, bb, gate, own["idx"]), own["w"],
                                       rtol=1e-13)


def pin_sigmoid_example(o):
    """Hand example of the sigmoid mode: s = sigma(r) = [1/2, 3/4, 1/4, 3/4];
    b = [0.3, 0, 0, -0.1] -> c = [0.8, 0.75, 0.25, 0.65]; K=1 keeps expert 0
    weighted by its uncorrected s = 0.5; the threshold candidate is expert 1."""
    r = np.array([0.0, math.log(3.0), -math.log(3.0), math.log(3.0)])
    b = np.array([0.3, 0.0, 0.0, -0.1])
    rt = o.route_from_logits(r, b, o.GATE_SIGMOID, 1)
    assert list(rt["idx"]) == [0]
    np.testing.assert_allclose(rt["w"], [0.5], rtol=1e-15)
    np.testing.assert_allclose(rt["top_scores"], [0.8, 0.75], rtol=1e-15)
    assert abs(rt["margin"] - 0.05) < 1e-15
    rt2 = o.route_from_logits(r, b, o.GATE_SIGMOID, 2)
    assert list(rt2["idx"]) == [0, 1]
    np.testing.assert_allclose(rt2["w"], [0.5, 0.75], rtol=1e-15)
    np.testing.assert_allclose(rt2["top_scores"], [0.8, 0.75, 0.65], rtol=1e-15)


# -- Dispatch -------------------------------------------------------------------

def pin_stable_dispatch_example(o):
    """kimi_k3 StableLatentMoE worked illustration."""
    g = golden("stable_dispatch_example.json")
    dp = o.dispatch(np.array(g["top_indices"]), g["E"])
    assert list(dp["order"]) == g["order"]
    assert list(dp["sorted_token"]) == g["sorted_token_ids"]
    assert list(dp["counts"]) == g["counts"]
    assert list(dp["offsets"][1:]) == g["ends"]
    # inverse: position of (t, k) in the sorted order
    inv = dp["inv"].reshape(-1)
    assert all(dp["order"][inv[j]] == j for j in range(len(g["flat"])))


def pin_dispatch_vs_library(o):
    """Dispatch equals NumPy's stable argsort / bincount / cumsum."""
    rng = np.random.default_rng(2)
    for _ in range(30):
        E = int(rng.integers(1, 20))
        K = int(rng.integers(1, min(E, 6) + 1))
        T = int(rng.integers(0, 50))
        idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]) if T else \
            np.zeros((0, K), np.int64)
        dp = o.dispatch(idx, E)
        flat = idx.reshape(-1)
        order = np.argsort(flat, kind="stable")
        assert np.array_equal(dp["order"], order)
        assert np.array_equal(dp["counts"], np.bincount(flat, minlength=E))
        assert np.array_equal(dp["offsets"][1:], np.cumsum(np.bincount(flat, minlength=E)))
        assert dp["counts"].sum() == T * K
        assert np.array_equal(dp["sorted_token"], order // K)
        assert np.array_equal(np.sort(dp["inv"].reshape(-1)), np.arange(T * K))


def pin_counts_sum(o):
    """'128 tokens x top-2 = 256 assignments' (MoE from scratch tutorial)."""
    rng = np.random.default_rng(3)
    x = rng.normal(size=(128, 64))
    Wr = rng.normal(size=(64, 8)) / 8
    rt = o.route(x, Wr, None, o.GATE_SOFTMAX_ALL_RENORM, 2)
    dp = o.dispatch(rt["idx"], 8)
    assert dp["counts"].sum() == 256
    np.testing.assert_allclose(rt["w"].sum(axis=1), 1.0, atol=1e-13)


# -- Layer ----------------------------------------------------------------------

def tiny_params(rng, d, F, E, S, Fs, latent=0):
    de = latent or d
    p = {
        "W_router": rng.normal(size=(d, E)) / math.sqrt(d),
        "bias": rng.normal(scale=0.01, size=E),
        "W_gate": rng.normal(size=(E, de, F)) / math.sqrt(de),
        "W_up": rng.normal(size=(E, de, F)) / math.sqrt(de),
        "W_down": rng.normal(size=(E, F, de)) / math.sqrt(F),
        "Ws_gate": rng.normal(size=(S, d, Fs)) / math.sqrt(d) if S else None,
        "Ws_up": rng.normal(size=(S, d, Fs)) / math.sqrt(d) if S else None,
        "Ws_down": rng.normal(size=(S, Fs, d)) / math.sqrt(Fs) if S else None,
        "W_down_latent": rng.normal(size=(d, latent)) / math.sqrt(d) if latent else None,
        "W_up_latent": rng.normal(size=(latent, d)) / math.sqrt(latent) if latent else None,
    }
    return p


def pin_output_composition(o):
    """MoE(x) = sum_s Shared_s(x) + sum_k g_k Expert_{e_k}(x) on section 12.5's
    matrices: expert 0 gives y (hand-derived), expert 1 gives 2y, the router
    logits are [ln 3, 0] so the K=2 softmax weights are [3/4, 1/4], and one
    shared expert equal to expert 0 adds y: total 2.25 y. With K=1 only
    expert 0 is used with weight 1: y + y."""
    g = golden("swiglu_example_12_5.json")
    x = np.array(g["x"])
    Wg, Wu, Wd = np.array(g["W_gate"]), np.array(g["W_up"]), _down_perm()
    Wr = np.zeros((4, 2))
    Wr[0, 0] = math.log(3.0)
    p = {"W_router": Wr, "bias": None,
         "W_gate": np.stack([Wg, Wg]), "W_up": np.stack([Wu, Wu]),
         "W_down": np.stack([Wd, 2 * Wd]),
         "Ws_gate": Wg[None], "Ws_up": Wu[None], "Ws_down": Wd[None]}
    y = _expected_perm_out()
    out, rt = o.moe_forward(x[None], p, o.GATE_SOFTMAX_TOPK, 2)
    assert list(rt["idx"][0]) == [0, 1]
    np.testing.assert_allclose(rt["w"][0], [0.75, 0.25], rtol=1e-14)
    np.testing.assert_allclose(out[0], 2.25 * y, atol=1e-5, rtol=0)
    out1, _ = o.moe_forward(x[None], p, o.GATE_SOFTMAX_TOPK, 1)
    np.testing.assert_allclose(out1[0], 2.0 * y, atol=1e-5, rtol=0)
    # without shared experts only the routed part remains
    p0 = dict(p, Ws_gate=None, Ws_up=None, Ws_down=None)
    out0, _ = o.moe_forward(x[None], p0, o.GATE_SOFTMAX_TOPK, 2)
    np.testing.assert_allclose(out0[0], 1.25 * y, atol=1e-5, rtol=0)


def pin_sorted_equals_naive(o):
    """The per-token forward equals the sorted-dispatch forward (MoE from
    scratch: 'sorted dispatch matches the reference')."""
    rng = np.random.default_rng(4)
    cases = [(o.GATE_SOFTMAX_ALL_RENORM, 0), (o.GATE_SOFTMAX_TOPK, 0), (o.GATE_SIGMOID, 0),
             (o.GATE_SIGMOID, 6)]
    for gate, L in cases:
        T, d, F, E, K, S, Fs = 37, 12, 10, 7, 3, 2, 9
        p = tiny_params(rng, d, F, E, S, Fs, latent=L)
        x = rng.normal(size=(T, d))
        a, _ = o.moe_forward(x, p, gate, K)
        b = o.moe_forward_sorted(x, p, gate, K)
        np.testing.assert_allclose(a, b, atol=1e-12, rtol=0)
        # a subset of rows, in any order, under an adopted selection: the same
        # rows, NaN elsewhere
        rows = [30, 2, 17, 5, 36]
        idx = np.stack([rng.permutation(E)[:K] for _ in range(T)])
        wts = rng.uniform(0.1, 1.0, size=(T, K))
        a, _ = o.moe_forward(x, p, gate, K, tokens=rows, routing=(idx, wts))
        b = o.moe_forward_sorted(x, p, gate, K, tokens=rows, routing=(idx, wts))
        assert np.isnan(b[[0, 1, 3]]).all()
        np.testing.assert_allclose(a[rows], b[rows], atol=1e-12, rtol=0)


def pin_shared_concat_identity(o):
    """S shared SwiGLU experts equal one SwiGLU of width S*Fs whose gate/up
    matrices are concatenated along d_ff and down matrices along the rows."""
    rng = np.random.default_rng(5)
    d, Fs, S = 9, 5, 3
    p = tiny_params(rng, d, 4, 3, S, Fs)
    x = rng.normal(size=(6, d))
    sep = sum(o.swiglu_ffn(x, p["Ws_gate"][s], p["Ws_up"][s], p["Ws_down"][s]) for s in range(S))
    cat = o.swiglu_ffn(x, np.concatenate(list(p["Ws_gate"]), axis=1),
                       np.concatenate(list(p["Ws_up"]), axis=1),
                       np.concatenate(list(p["Ws_down"]), axis=0))
    np.testing.assert_allclose(sep, cat, atol=1e-12, rtol=0)
    # and the layer's shared term is that sum
    p["W_gate"] = np.zeros_like(p["W_gate"])
    out, _ = o.moe_forward(x, p, o.GATE_SOFTMAX_TOPK, 2)
    np.testing.assert_allclose(out, sep, atol=1e-12, rtol=0)


def pin_latent_reduces_to_plain(o):
    """With W_down_latent = W_up_latent = identity (L = d) the latent layer is
    the plain layer with the same experts."""
    rng = np.random.default_rng(6)
    d = 8
    p = tiny_params(rng, d, 6, 5, 1, 7, latent=d)
    p["W_down_latent"] = np.eye(d)
    p["W_up_latent"] = np.eye(d)
    x = rng.normal(size=(11, d))
    a, _ = o.moe_forward(x, p, o.GATE_SIGMOID, 2)
    plain = dict(p, W_down_latent=None, W_up_latent=None)
    b, _ = o.moe_forward(x, plain, o.GATE_SIGMOID, 2)
    np.testing.assert_allclose(a, b, atol=1e-13, rtol=0)
    # and a scaled up-projection scales only the routed part
    p2 = dict(p, W_up_latent=3.0 * np.eye(d))
    c, _ = o.moe_forward(x, p2, o.GATE_SIGMOID, 2)
    sh = o.swiglu_ffn(x, p["Ws_gate"][0], p["Ws_up"][0], p["Ws_down"][0])
    np.testing.assert_allclose(c - sh, 3.0 * (b - sh), atol=1e-12, rtol=0)


# -- Balancers --------------------------------------------------------------------

def pin_quantile(o):
    """'higher' quantile = NumPy's method='higher'; centred biases sum to ~0;
    shifting every score by an exact constant leaves the biases unchanged."""
    rng = np.random.default_rng(7)
    for T, E, K in ((8193, 128, 8), (1025, 64, 8), (257, 16, 4), (65, 8, 2), (2, 4, 1)):
        s = (rng.integers(1, 1 << 20, size=(T, E)) / float(1 << 21)).astype(np.float32)
        top = np.sort(s, axis=1)[:, ::-1][:, :K + 1].astype(np.float32)
        b = o.quantile_bias_update(top, s, K)
        rel = (top[:, K][:, None] - s).astype(np.float32)
        q = np.quantile(rel.astype(np.float64), K / E, axis=0, method="higher")
        qrank = o.quantile_rank(T, E, K)
        assert qrank == math.ceil(K / E * (T - 1))
        mean = np.float32(sum(float(v) for v in q) / E)
        np.testing.assert_array_equal(b, (q.astype(np.float32) - mean).astype(np.float32))
        assert abs(float(np.sum(b.astype(np.float64)))) <= E * 2e-7
        # exact shift (all values on a 2^-21 grid below 1, shift 0.5: exact in FP32)
        b2 = o.quantile_bias_update(top + np.float32(0.5), s + np.float32(0.5), K)
        np.testing.assert_array_equal(b, b2)
    # tiny brute force: T=5, p=1/2 -> rank ceil(0.5*4)=2 (third smallest)
    s = np.array([[0.1], [0.5], [0.3], [0.9], [0.7]], dtype=np.float32)
    s2 = np.concatenate([s, np.float32(1.0) - s], axis=1)
    top = np.full((5, 2), 1.0, dtype=np.float32)
    b = o.quantile_bias_update(top, s2, 1)
    # column 0 rel = 1 - s: sorted [0.1,0.3,0.5,0.7,0.9] -> 0.5; column 1 rel = s -> 0.5
    np.testing.assert_allclose(b, [0.0, 0.0], atol=1e-7)


def pin_sign_bias_example(o):
    """APEX-1 Math Ref Part 3, section 14.5."""
    g = golden("sign_bias_example_14_5.json")
    nb = o.sign_bias_update(g["counts"], g["N"], g["K"], g["initial_bias"], g["alpha"])
    np.testing.assert_allclose(nb, g["new_bias"], atol=1e-15)
    f = np.array(g["counts"]) / (g["N"] * g["K"])
    np.testing.assert_allclose(f, g["observed_rates"], atol=5e-4)
    # clamp to [-1, 1]
    nb = o.sign_bias_update([16, 0, 0, 0], 8, 2, [-0.95, 0.95, 0.0, 0.0], 0.1)
    np.testing.assert_allclose(nb, [-1.0, 1.0, 0.1, 0.1], atol=1e-15)


def pin_routing_stats(o):
    """Switch loss and z-loss ([MoE-FS] MoELayer.forward, [BOOK-MoE]
    router_z_loss) on cases fixed by the definitions: a zero router gives
    P_e = 1/E, so aux = E * sum_e f_e / E = 1 for any routing and z = (ln E)^2;
    all assignments on one expert with one-hot-like logits give aux -> E;
    a 2-token, 2-expert hand example; shifting a token's logits by c leaves P
    unchanged and moves its log-sum-exp by c."""
    T, E, K = 6, 4, 2
    idx = np.array([[0, 1], [0, 2], [3, 0], [1, 0], [2, 3], [0, 1]])
    st = o.routing_stats(np.zeros((T, E)), idx, E)
    assert abs(st["aux"] - 1.0) < 1e-15
    assert abs(st["z"] - math.log(E) ** 2) < 1e-14
    assert np.allclose(st["P"], 1.0 / E) and abs(st["f"].sum() - 1.0) < 1e-15
    assert np.allclose(st["f"], np.array([5, 3, 2, 2]) / 12.0)
    # everything on expert 0, router certain of it: aux -> E * 1 * 1 = E
    big = np.zeros((5, E))
    big[:, 0] = 60.0
    st = o.routing_stats(big, np.zeros((5, 1), dtype=int), E)
    assert abs(st["aux"] - E) < 1e-12
    # hand example: r = [[ln 3, 0], [0, 0]], idx = [[0], [1]]
    # softmax rows [3/4, 1/4] and [1/2, 1/2] -> P = [5/8, 3/8]; f = [1/2, 1/2]
    # aux = 2 (5/16 + 3/16) = 1; lse = [ln 4, ln 2] -> z = ((ln 4)^2 + (ln 2)^2) / 2
    st = o.routing_stats(np.array([[math.log(3.0), 0.0], [0.0, 0.0]]), np.array([[0], [1]]), 2)
    assert np.allclose(st["P"], [5 / 8, 3 / 8], rtol=0, atol=1e-15)
    assert abs(st["aux"] - 1.0) < 1e-15
    assert abs(st["z"] - (math.log(4.0) ** 2 + math.log(2.0) ** 2) / 2) < 1e-14
    # second hand example, unequal shares: r = [[ln 3, 0], [ln 3, 0]], idx = [[0], [0]]
    # P = [3/4, 1/4], f = [1, 0] -> aux = 2 * 3/4 = 3/2
    st = o.routing_stats(np.array([[math.log(3.0), 0.0]] * 2), np.array([[0], [0]]), 2)
    assert abs(st["aux"] - 1.5) < 1e-15
    # shift invariance of P; lse moves by the shift
    rng = np.random.default_rng(9)
    r = rng.normal(size=(7, 5))
    a = o.routing_stats(r, np.zeros((7, 1), dtype=int), 5)
    b = o.routing_stats(r + 2.5, np.zeros((7, 1), dtype=int), 5)
    assert np.allclose(a["P"], b["P"], atol=1e-15)
    lse = np.log(np.exp(r).sum(axis=1))
    assert abs(a["z"] - np.mean(lse ** 2)) < 1e-12
    assert abs(b["z"] - np.mean((lse + 2.5) ** 2)) < 1e-12


# -- Backward -------------------------------------------------------------------

def _fd_loss(o, x, p, dout, gate, K, idx, renorm, scale):
    """L = sum(dout * out) of the layer with the selection idx held fixed and
    the gate weights recomputed from the (perturbed) router logits: built from
    the oracle's forward pieces only."""
    xn = np.asarray(x, float)
    r = o.router_logits(xn, p["W_router"])
    L = 0.0
    for t in range(xn.shape[0]):
        w_t = o.gates_for(r[t], p.get("bias"), gate, idx[t], renorm, scale)
        L += float(np.dot(dout[t], o.moe_forward_token(xn[t], idx[t], w_t, p, None)))
    return L


def pin_backward_finite_differences(o):
    """Every gradient of moe_backward against central differences of the
    forward (L = sum(dout * out), selection fixed), for each gate mode, with
    shared experts, renormalised and scaled sigmoid gates and the latent
    variant; experts nobody selects get no gradient (kimi_k3 StableLatentMoE,
    'Grouped expert execution and sparse gradients')."""
    rng = np.random.default_rng(11)
    eps = 1e-5
    cases = [(o.GATE_SOFTMAX_TOPK, 0, False, 1.0, 2), (o.GATE_SOFTMAX_ALL_RENORM, 0, False, 1.0, 1),
             (o.GATE_SIGMOID, 0, True, 2.5, 2), (o.GATE_SIGMOID, 5, False, 1.0, 0)]
    for gate, L, renorm, scale, S in cases:
        T, d, F, E, K, Fs = 5, 7, 6, 6, 2, 4
        p = tiny_params(rng, d, F, E, S, Fs, latent=L)
        p["bias"] = rng.normal(scale=0.01, size=E)
        p["bias"][E - 1] = -50.0  # expert E-1 is never selected
        x = rng.normal(size=(T, d))
        dout = rng.normal(size=(T, d))
        idx = o.route(x, p["W_router"], p["bias"], gate, K, renorm, scale)["idx"]
        assert not (idx == E - 1).any()
        g = o.moe_backward(x, p, dout, gate, K, renorm, scale)
        assert not g["active"][E - 1] and g["active"][np.unique(idx)].all()
        # a token subset gives those tokens' dx rows exactly and zero elsewhere
        gs = o.moe_backward(x, p, dout, gate, K, renorm, scale, tokens=[1, 3])
        assert np.array_equal(gs["dx"][[1, 3]], g["dx"][[1, 3]])
        assert not gs["dx"][[0, 2, 4]].any()
        for name in ("dW_gate", "dW_up", "dW_down"):
            assert not g[name][E - 1].any(), name

        def check(name, arr_key, grad, picks):
            for ii in picks:
                base = (p[arr_key] if arr_key != "x" else x)
                a = np.array(base, dtype=float, copy=True)
                q = dict(p)
                orig = a[ii]
                a[ii] = orig + eps
                if arr_key == "x":
                    lp = _fd_loss(o, a, q, dout, gate, K, idx, renorm, scale)
                else:
                    q[arr_key] = a
                    lp = _fd_loss(o, x, q, dout, gate, K, idx, renorm, scale)
                a[ii] = orig - eps
                if arr_key == "x":
                    lm = _fd_loss(o, a, q, dout, gate, K, idx, renorm, scale)
                else:
                    q[arr_key] = a
                    lm = _fd_loss(o, x, q, dout, gate, K, idx, renorm, scale)
                fd = (lp - lm) / (2 * eps)
                assert abs(grad[ii] - fd) <= 1e-7 * (1.0 + abs(fd)), (gate, name, ii, grad[ii], fd)

        def picks(shape, n):
            return [tuple(int(rng.integers(0, s)) for s in shape) for _ in range(n)]

        check("dx", "x", g["dx"], [(t, j) for t in range(T) for j in range(d)])
        check("dW_router", "W_router", g["dW_router"], [(i, j) for i in range(d) for j in range(E)])
        for name, key in (("dW_gate", "W_gate"), ("dW_up", "W_up"), ("dW_down", "W_down")):
            check(name, key, g[name], picks(p[key].shape, 10))
        if S:
            for name, key in (("dWs_gate", "Ws_gate"), ("dWs_up", "Ws_up"), ("dWs_down", "Ws_down")):
                check(name, key, g[name], picks(p[key].shape, 8))
        if L:
            for name, key in (("dW_down_latent", "W_down_latent"), ("dW_up_latent", "W_up_latent")):
                check(name, key, g[name], picks(p[key].shape, 8))


def pin_round_bf16(o):
    """round_bf16 equals PyTorch's FP32 -> BF16 conversion (nearest-even) on
    random values and on exact ties."""
    import torch
    rng = np.random.default_rng(12)
    v = np.concatenate([rng.normal(size=2000) * 10.0 ** rng.integers(-6, 6, size=2000),
                        [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 0.0]])
    ref = torch.tensor(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(o.round_bf16(v), ref)
    assert o.round_bf16(1.0 + 2.0 ** -8) == 1.0 and o.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6


ALL_PINS = [pin_silu_table, pin_swiglu_example, pin_ffn_down_projection, pin_router_example,
            pin_tie_break, pin_gate_formulas, pin_sigmoid_example, pin_stable_dispatch_example,
            pin_dispatch_vs_library, pin_counts_sum, pin_output_composition,
            pin_sorted_equals_naive, pin_shared_concat_identity, pin_latent_reduces_to_plain,
            pin_quantile, pin_sign_bias_example, pin_routing_stats,
            pin_backward_finite_differences, pin_round_bf16]
