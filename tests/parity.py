"""Glue for the GPU parity tests: run the CUDA path through the C ABI and the
oracle on the same seeded inputs, and compare.

Tolerances: routing ids, counts and permutations bit-exact wherever the
oracle's rank-K / rank-(K+1) score margin exceeds 1e-5. A token is a near tie
when any two consecutive scores among its top K+1 are within 1e-5 (that
covers the selection boundary and the slot order, both part of the bit-exact
arrays); near ties are counted, and for those tokens the oracle adopts the
GPU's expert selection, with gate weights by its own formulas. Layer outputs
within max-abs 1e-4 for FP32 layers and 2e-2 x RMS(oracle output) for BF16.
"""
import math

import numpy as np
import torch

from mixture_experts_ffn_fp32_gb300 import api
from mixture_experts_ffn_fp32_gb300 import workloads as W
from oracle import moe_oracle as O

NEAR_TIE = 1e-5
F32_ATOL = 1e-4
BF16_REL = 2e-2


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def npi(t):
    return t.detach().cpu().numpy().astype(np.int64)


def spec_of(w: W.Workload) -> api.LayerSpec:
    return api.LayerSpec.of(w)


def oracle_routing(w: W.Workload, inputs, rows=None):
    x = inputs["x"] if rows is None else inputs["x"][rows]
    return O.route(np64(x), np64(inputs["W_router"]),
                   None if inputs["bias"] is None else np64(inputs["bias"]),
                   w.gate, w.K, w.renormalize, w.routed_scale)


def merge_routing(w: W.Workload, inputs, ort, gpu_idx):
    """Oracle routing with the GPU's selection adopted for near-tie tokens."""
    near = ort["min_gap"] <= NEAR_TIE
    idx = ort["idx"].copy()
    wts = ort["w"].copy()
    bias = None if inputs["bias"] is None else np64(inputs["bias"])
    for t in np.where(near)[0]:
        idx[t] = gpu_idx[t]
        wts[t] = O.gates_for(ort["logits"][t], bias, w.gate, gpu_idx[t], w.renormalize,
                             w.routed_scale)
    return idx, wts, near


def check_routing(w, ort, gpu, near):
    """Bit-exact ids outside near ties; weights and margins close everywhere."""
    gi = npi(gpu["idx"])
    far = ~near
    mism = np.where((gi[far] != ort["idx"][far]).any(axis=1))[0]
    assert mism.size == 0, f"{mism.size} tokens routed differently outside near ties"
    # every GPU selection is K distinct valid ids
    assert gi.min() >= 0 and gi.max() < w.E
    srt = np.sort(gi, axis=1)
    assert w.K == 1 or (np.diff(srt, axis=1) > 0).all()
    gw = np64(gpu["w"])
    np.testing.assert_allclose(gw[far], ort["w"][far], atol=2e-6, rtol=1e-5)
    gm = np64(gpu["margin"])
    om = ort["margin"]
    fin = np.isfinite(om)
    np.testing.assert_allclose(gm[fin], om[fin], atol=2e-5, rtol=1e-4)
    assert np.all(np.isinf(gm[~fin]))
    if w.gate == "sigmoid":
        np.testing.assert_allclose(np64(gpu["top_scores"])[far], ort["top_scores"][far],
                                   atol=2e-6, rtol=0)
        np.testing.assert_allclose(np64(gpu["scores"]), ort["s"], atol=2e-6, rtol=0)
    else:
        np.testing.assert_allclose(gw.sum(axis=1), 1.0, atol=2e-6)


def check_dispatch(w, idx, wts_gpu_flat, gpu):
    """GPU dispatch results == oracle dispatch of the routing idx, bit for bit."""
    dp = O.dispatch(idx, w.E)
    assert np.array_equal(npi(gpu["counts"]), dp["counts"])
    assert np.array_equal(npi(gpu["offsets"]), dp["offsets"])
    assert np.array_equal(npi(gpu["sorted_token"]), dp["sorted_token"])
    assert np.array_equal(npi(gpu["inv"]).reshape(-1), dp["inv"].reshape(-1))
    sw = gpu["sorted_w"].detach().cpu().numpy()
    assert np.array_equal(sw, wts_gpu_flat[dp["order"]])
    assert int(dp["counts"].sum()) == w.T * w.K
    return dp


def check_output(w, out_gpu, ref, rows=None):
    g = np64(out_gpu)
    if rows is not None:
        g, ref = g[rows], ref[rows]
    assert np.isfinite(g).all(), "non-finite GPU output"
    err = float(np.abs(g - ref).max())
    if w.dtype == "f32":
        assert err <= F32_ATOL, f"max-abs error {err:.3e} > {F32_ATOL}"
        return err, None
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert err <= BF16_REL * rms, f"max-abs error {err:.3e} > {BF16_REL} x RMS {rms:.3e}"
    return err, rms


def run_forward(w: W.Workload, inputs, stream=None):
    spec = spec_of(w)
    ws = api.alloc_workspace(spec)
    out = api.forward(spec, inputs["x"], inputs, ws=ws)
    st = api.workspace_status(ws)
    assert st == api.MOE_OK, api.status_string(st)
    views = api.workspace_views(spec, ws)
    return out, views, ws


def sample_rows(w, gpu_idx, offsets=None, sorted_token=None, n_even=512, n_rare=8,
                n_tile_experts=4, seed=0, rare_cap=None):
    """Rows for a sampled comparison: n_even evenly spaced tokens (with the
    first and last), every token routed to the n_rare least-used experts that
    get any, and, for n_tile_experts experts (the most and least loaded of
    those with rows, and random others), the tokens at the first and last row
    of each of their 128-row and 256-row tiles in the expert-sorted order.
    rare_cap: at most that many tokens of each rare expert (all if None)."""
    rng = np.random.default_rng(seed)
    T = w.T
    rows = {0, T - 1}
    rows.update(int(v) for v in np.linspace(0, T - 1, num=min(T, n_even)).round())
    counts = np.bincount(gpu_idx.reshape(-1), minlength=w.E)
    used = np.where(counts > 0)[0]
    by_load = used[np.argsort(counts[used], kind="stable")]
    for e in by_load[:n_rare]:
        rows.update(int(t) for t in np.where((gpu_idx == e).any(axis=1))[0][:rare_cap])
    if offsets is not None and sorted_token is not None and used.size:
        pick = [int(by_load[-1]), int(by_load[0])]
        rest = [int(e) for e in used if e not in pick]
        if rest:
            pick += [int(e) for e in rng.choice(rest, size=min(len(rest), n_tile_experts - 2),
                                               replace=False)]
        for e in pick:
            a, b = int(offsets[e]), int(offsets[e + 1])
            for h in (128, 256):
                for s0 in range(a, b, h):
                    rows.add(int(sorted_token[s0]))
                    rows.add(int(sorted_token[min(s0 + h, b) - 1]))
    return sorted(rows)


def full_parity(w: W.Workload, device="cuda", sample=False, record=None):
    """Forward on the GPU, then: routing bit-exact on all tokens (outside near
    ties), dispatch bit-exact on all assignments, outputs against the oracle
    on every row (sample=False) or on sample_rows' set (sample=True). The
    oracle's expert-grouped form (pinned equal to its per-token form) keeps
    whole large layers affordable. ``record``: a path that gets one JSON line
    with the counts and errors."""
    inputs = W.make_inputs(w, device=device)
    out, views, ws = run_forward(w, inputs)
    torch.cuda.synchronize()
    ort = oracle_routing(w, inputs)
    gi = npi(views["idx"])
    idx, wts, near = merge_routing(w, inputs, ort, gi)
    check_routing(w, ort, views, near)
    # dispatch of the oracle's routing (GPU selection only at near ties), bit for bit
    dp = check_dispatch(w, idx, views["w"].detach().cpu().numpy().reshape(-1), views)
    rows = sample_rows(w, gi, dp["offsets"], dp["sorted_token"]) if sample else None
    ref = O.moe_forward_sorted(inputs["x"], inputs, w.gate, w.K, w.renormalize,
                               w.routed_scale, tokens=rows, routing=(idx, wts))
    err, rms = check_output(w, out, ref, rows)
    res = {"workload": w.name, "T": w.T, "near_ties": int(near.sum()),
           "near_ties_at_selection": int((ort["margin"] <= NEAR_TIE).sum()),
           "max_err": err, "rms": rms, "max_err_over_rms": None if rms is None else err / rms,
           "rows": w.T if rows is None else len(rows),
           "empty_experts": int((dp["counts"] == 0).sum())}
    if record:
        import json
        with open(record, "a") as f:
            f.write(json.dumps(res) + "\n")
    del inputs, out, views, ws
    torch.cuda.empty_cache()
    return res
