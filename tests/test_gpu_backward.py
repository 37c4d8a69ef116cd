"""Backward pass on the GPU (moe_backward through the C ABI) against the
oracle's float64 backward, on the GPU forward's own expert selection (the
selection carries no gradient, so both sides differentiate the same
piecewise-smooth function).

Tolerances. The CUDA-core form (layers whose widths are not all multiples of
64, and FP32 layers) computes in FP32 from the exact inputs, so its
gradients of non-latent layers stay within 1e-4 x RMS of the oracle's (FP32
sums of at most a few hundred terms of unit scale: ~1e-6 relative). The latent
variant's experts act on the forward's latent rows z, which a BF16 layer
stores in BF16; the oracle rounds its z the same way (latent_rows_bf16; with
exact z the rounding alone moves expert weight gradients by up to ~4% of
their RMS on this layer), and the remaining differences - an FP32 sum that
rounds to the other BF16 neighbour, and the forward's BF16 hidden rows inside
the routed sum dW_up_latent reads - stay within the forward's 2e-2 x RMS.
The tensor-core form rounds the upstream gradients and the activation
gradients (gy, da, du, g h) to BF16 before its products, as mixed-precision
backward passes do; emulating exactly that rounding on the oracle moves the
expert weight gradients by 0.24% in relative Frobenius norm and by at most
4.9% of their RMS on one element (on these layers), so the bound there is
1e-2 relative Frobenius and 1e-1 x RMS max-abs on every gradient.
"""
import math

import numpy as np
import pytest
import torch

from mixture_experts_ffn_fp32_gb300 import api as A
from mixture_experts_ffn_fp32_gb300 import workloads as W
from oracle import moe_oracle as O
from tests import parity as P

pytestmark = pytest.mark.gpu

LAYERS = {
    "f32_softmax_all": W.Workload("g_f1", T=60, d=64, d_ff=96, E=8, K=2, n_shared=1,
                                  shared_d_ff=64, dtype="f32", gate="softmax_all_renorm",
                                  has_bias=False),
    "bf16_topk_shared2": W.Workload("g_b1", T=70, d=128, d_ff=96, E=12, K=3, n_shared=2,
                                    shared_d_ff=64, dtype="bf16", gate="softmax_topk",
                                    bias_std=0.01, skew=1.2),
    "bf16_sigmoid_renorm": W.Workload("g_b2", T=50, d=96, d_ff=64, E=16, K=3, n_shared=1,
                                      shared_d_ff=32, dtype="bf16", gate="sigmoid",
                                      renormalize=True, routed_scale=2.5),
    "bf16_sparse_experts": W.Workload("g_b3", T=30, d=64, d_ff=48, E=40, K=2, n_shared=0,
                                      shared_d_ff=0, dtype="bf16", gate="softmax_topk",
                                      bias_std=0.01, skew=1.2),
    "bf16_latent_sigmoid": W.Workload("g_b4", T=40, d=128, d_ff=48, E=10, K=2, n_shared=1,
                                      shared_d_ff=64, dtype="bf16", gate="sigmoid",
                                      latent_dim=64),
}

# Widths that are multiples of 64: the tensor-core backward (several 128-row
# and 128-column tiles with ragged ends, experts padded to 64-column blocks,
# empty experts, one and two shared experts, latent rows).
TC_LAYERS = {
    "tc_topk_shared": W.Workload("g_t1", T=150, d=128, d_ff=192, E=6, K=2, n_shared=1,
                                 shared_d_ff=128, dtype="bf16", gate="softmax_topk",
                                 bias_std=0.01, skew=1.2),
    "tc_sigmoid_renorm_s2": W.Workload("g_t2", T=96, d=192, d_ff=128, E=12, K=3, n_shared=2,
                                       shared_d_ff=64, dtype="bf16", gate="sigmoid",
                                       renormalize=True, routed_scale=2.5),
    "tc_sparse": W.Workload("g_t3", T=40, d=128, d_ff=64, E=48, K=2, n_shared=0, shared_d_ff=0,
                            dtype="bf16", gate="softmax_topk", bias_std=0.01, skew=1.2),
    "tc_latent": W.Workload("g_t4", T=80, d=192, d_ff=128, E=8, K=2, n_shared=1,
                            shared_d_ff=128, dtype="bf16", gate="sigmoid", latent_dim=64),
    "tc_renorm_all": W.Workload("g_t5", T=64, d=64, d_ff=64, E=8, K=2, n_shared=1,
                                shared_d_ff=64, dtype="bf16", gate="softmax_all_renorm",
                                has_bias=False),
    # outputs 256 and more columns wide: the 128 x 256 tile form, ragged in N
    "tc_wide": W.Workload("g_t6", T=200, d=256, d_ff=320, E=5, K=2, n_shared=1,
                          shared_d_ff=256, dtype="bf16", gate="softmax_topk", bias_std=0.01),
    "tc_wide_latent": W.Workload("g_t7", T=120, d=320, d_ff=256, E=6, K=2, n_shared=1,
                                 shared_d_ff=64, dtype="bf16", gate="sigmoid", latent_dim=256),
}


def _dout(w, seed=7):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(w.T, w.d, generator=g, dtype=torch.float32).cuda()


def run(w, save_gate_up=False):
    spec = A.LayerSpec.of(w, save_gate_up=save_gate_up)
    inp = W.make_inputs(w, device="cuda")
    ws = A.alloc_workspace(spec)
    A.forward(spec, inp["x"], inp, ws=ws)
    views = A.workspace_views(spec, ws)
    gidx = P.npi(views["idx"])
    counts = P.npi(views["counts"])
    dout = _dout(w)
    # expert gradients pre-filled with NaN: slices of experts without rows must stay NaN
    shapes = A.grad_shapes(spec)
    grads = {n: torch.full(shapes[n], float("nan"), device="cuda")
             for n in ("dW_gate", "dW_up", "dW_down")}
    g = A.backward(spec, inp["x"], inp, dout, ws, grads=grads)
    torch.cuda.synchronize()
    assert A.workspace_status(ws) == A.MOE_OK
    return spec, inp, ws, gidx, counts, dout, g


def _tc(w):
    de = w.latent_dim or w.d
    return (w.dtype == "bf16" and w.d % 64 == 0 and w.d_ff % 64 == 0 and de % 64 == 0
            and (w.n_shared == 0 or w.shared_d_ff % 64 == 0))


CASES = [(n, False) for n in list(LAYERS) + list(TC_LAYERS)] + [(n, True) for n in TC_LAYERS]


@pytest.mark.parametrize("name,saved", CASES)
def test_backward_matches_oracle(name, saved):
    """saved: the forward kept its BF16 gate and up products (save_gate_up) and
    the SwiGLU backward runs in the epilogue of the dh products on them; the
    tensor-core form's bounds hold for it unchanged."""
    w = {**LAYERS, **TC_LAYERS}[name]
    assert _tc(w) == (name in TC_LAYERS)
    spec, inp, ws, gidx, counts, dout, g = run(w, save_gate_up=saved)
    ref = O.moe_backward(inp["x"], inp, dout, w.gate, w.K, w.renormalize, w.routed_scale,
                         routing=gidx, latent_rows_bf16=bool(w.latent_dim))
    assert np.array_equal(ref["active"], counts > 0)
    rel = 2e-2 if w.latent_dim else 1e-4
    frob = None
    if _tc(w):
        rel, frob = 1e-1, 1e-2
    for n, gt in g.items():
        r = ref[n]
        got = gt.detach().cpu().numpy().astype(np.float64)
        if n in ("dW_gate", "dW_up", "dW_down"):
            act = ref["active"]
            assert np.isnan(got[~act]).all(), f"{n}: an expert without rows got a gradient"
            got, r = got[act], r[act]
        assert np.isfinite(got).all(), n
        rms = float(np.sqrt(np.mean(r ** 2))) or 1.0
        err = float(np.abs(got - r).max())
        assert err <= rel * rms, f"{name} {n}: max-abs error {err:.3e} > {rel} x RMS {rms:.3e}"
        if frob is not None:
            fr = float(np.linalg.norm(got - r) / (np.linalg.norm(r) or 1.0))
            assert fr <= frob, f"{name} {n}: relative Frobenius error {fr:.3e} > {frob}"
    if w.latent_dim:
        check_against_exact_latent(name, w, inp, dout, gidx, g)


def check_against_exact_latent(name, w, inp, dout, gidx, g, tokens=None):
    """The latent gradients against the oracle's backward on the exact
    (unrounded) latent rows z, the definition: the BF16 storage of z alone
    moves the oracle's gradients by up to 3.6 % of their RMS on one element and
    0.35 % in relative Frobenius norm on these layers, so the bound is
    1e-1 x RMS max-abs and 1e-2 relative Frobenius on every gradient."""
    ref = O.moe_backward(inp["x"], inp, dout, w.gate, w.K, w.renormalize, w.routed_scale,
                         routing=gidx, latent_rows_bf16=False, tokens=tokens)
    for n, gt in g.items():
        r = ref[n]
        got = gt.detach().cpu().numpy().astype(np.float64)
        if tokens is not None:
            if n != "dx":
                continue
            got, r = got[tokens], r[tokens]
        if n in ("dW_gate", "dW_up", "dW_down"):
            got, r = got[ref["active"]], r[ref["active"]]
        rms = float(np.sqrt(np.mean(r ** 2))) or 1.0
        err = float(np.abs(got - r).max())
        fr = float(np.linalg.norm(got - r) / (np.linalg.norm(r) or 1.0))
        assert err <= 1e-1 * rms, f"{name} {n} (exact z): max-abs {err:.3e} > 0.1 x RMS {rms:.3e}"
        assert fr <= 1e-2, f"{name} {n} (exact z): relative Frobenius {fr:.3e} > 1e-2"


@pytest.mark.parametrize("name", ["tc_topk_shared", "tc_sigmoid_renorm_s2", "tc_latent", "tc_sparse"])
def test_saved_gate_up_forward_unchanged_and_gradients_agree(name):
    """Keeping the gate/up products changes no bit of the forward's output; the
    gradients from the saved BF16 products and from the recomputed FP32 ones
    agree to well within the bound either keeps against the oracle."""
    w = TC_LAYERS[name]
    inp = W.make_inputs(w, device="cuda")
    dout = _dout(w)
    outs, grads = [], []
    for saved in (False, True):
        spec = A.LayerSpec.of(w, save_gate_up=saved)
        ws = A.alloc_workspace(spec)
        outs.append(A.forward(spec, inp["x"], inp, ws=ws).clone())
        grads.append(A.backward(spec, inp["x"], inp, dout, ws))
        assert A.workspace_status(ws) == A.MOE_OK
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))
    for n in grads[0]:
        a = torch.nan_to_num(grads[0][n]).double()
        b = torch.nan_to_num(grads[1][n]).double()
        fr = float((a - b).norm() / (a.norm() + 1e-30))
        assert fr <= 5e-3, f"{name} {n}: saved vs recomputed relative Frobenius {fr:.3e}"


def test_backward_sparse_case_has_empty_experts():
    counts = run(LAYERS["bf16_sparse_experts"])[4]
    assert (counts == 0).any() and (counts > 0).any()


def test_backward_reproducible_and_optional_outputs():
    w = LAYERS["bf16_topk_shared2"]
    spec, inp, ws, gidx, counts, dout, g1 = run(w)
    g2 = A.backward(spec, inp["x"], inp, dout, ws,
                    grads={n: torch.full(A.grad_shapes(spec)[n], float("nan"), device="cuda")
                           for n in ("dW_gate", "dW_up", "dW_down")})
    for n in g1:
        assert torch.equal(torch.nan_to_num(g1[n], nan=7.0).view(torch.int32),
                           torch.nan_to_num(g2[n], nan=7.0).view(torch.int32)), n
    # only dx requested: the same dx
    g3 = A.backward(spec, inp["x"], inp, dout, ws,
                    grads={n: None for n in A.GRAD_NAMES if n != "dx"})
    assert set(g3) == {"dx"}
    assert torch.equal(g3["dx"].view(torch.int32), g1["dx"].view(torch.int32))


FULL = ["small", "medium_prefill", "medium_decode", "large_prefill", "large_prefill_zipf",
        "large_decode", "large_decode_zipf", "latent"]


@pytest.mark.parametrize("name,saved", [(n, False) for n in FULL] + [("small", True), ("latent", True)])
def test_full_size_backward_sampled_rows(name, saved):
    """The benchmark layers at full size: dx on sampled tokens (first, last,
    random, tokens of the rarest experts) against the oracle's backward of
    just those tokens, on the GPU's selection; expert slices of experts
    without rows stay as given; a second backward gives the same bits.
    saved: on the forward's kept gate/up products."""
    w = W.WORKLOADS[name]
    assert _tc(w)
    spec, inp, ws, gidx, counts, dout, g = run(w, save_gate_up=saved)
    rows = P.sample_rows(w, gidx, n_even=8, n_rare=2, rare_cap=4)
    ref = O.moe_backward(inp["x"], inp, dout, w.gate, w.K, w.renormalize, w.routed_scale,
                         routing=gidx, latent_rows_bf16=bool(w.latent_dim), tokens=rows)
    got = g["dx"][rows].detach().cpu().numpy().astype(np.float64)
    r = ref["dx"][rows]
    assert np.isfinite(got).all()
    rms = float(np.sqrt(np.mean(r ** 2)))
    err = float(np.abs(got - r).max())
    fr = float(np.linalg.norm(got - r) / np.linalg.norm(r))
    assert fr <= 1e-2, f"{name}: dx relative Frobenius error {fr:.3e} on sampled rows"
    assert err <= 1e-1 * rms, f"{name}: dx max-abs error {err:.3e} > 0.1 x RMS {rms:.3e}"
    empty = np.where(counts == 0)[0]
    for n in ("dW_gate", "dW_up", "dW_down"):
        if empty.size:
            assert torch.isnan(g[n][torch.as_tensor(empty, device=g[n].device)]).all(), n
        assert torch.isfinite(g[n][torch.as_tensor(np.where(counts > 0)[0], device=g[n].device)]).all(), n
    if w.latent_dim:
        check_against_exact_latent(name, w, inp, dout, gidx, g, tokens=rows)
    g2 = A.backward(spec, inp["x"], inp, dout, ws, grads={n: None for n in A.GRAD_NAMES if n != "dx"})
    assert torch.equal(g2["dx"].view(torch.int32), g["dx"].view(torch.int32))
    print(name, {"rows": len(rows), "frob": fr, "max_err_over_rms": err / rms, "empty_experts": int(empty.size)})
    del g, g2, ws, inp
    torch.cuda.empty_cache()
