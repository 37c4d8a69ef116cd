"""The token-column CTA-pair form of the grouped GEMMs (the expert's weights
as the MMA's A operand, the segment's tokens as its N columns), which the
forward takes when routed segments average 128 rows or more: oracle parity
on every row for layers whose shapes reach its edges, and agreement with the
row-tile forms (MOE_GEMM_FORM=rows) on the same inputs.

Edges covered: widths that are not multiples of 64 (per-strip copies instead
of the strip boxes) or of the 256/512-feature unit (a half-empty last unit,
an odd CTA without features), segments of 1..15 rows (N = 16), exactly 256
and 257 rows (one unit, then two of 128/129 rows), empty experts, several
shared experts (segments of the dense group), sigmoid and top-k gates.
"""
import os

import numpy as np
import pytest
import torch

from tests import parity as P
from mixture_experts_ffn_fp32_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from mixture_experts_ffn_fp32_gb300 import build
    build.build()
    from mixture_experts_ffn_fp32_gb300 import api
    return api


def _wl(name, **kw):
    base = dict(n_shared=1, shared_d_ff=256, dtype="bf16", gate="softmax_topk", bias_std=0.01)
    base.update(kw)
    return W.Workload(name, **base)


LAYERS = {
    # about 256 rows per expert: most segments take one unit, some two
    "e16_256rows": _wl("k_1", T=1024, d=512, d_ff=512, E=16, K=4),
    # ragged widths: d = 320 (plain units of 512 features: one half-empty, the
    # odd CTA of the pair has none), d_ff = 192 (SwiGLU unit half-empty, not a
    # multiple of 128), shared width 160 (per-strip copies)
    "ragged_widths": _wl("k_2", T=700, d=320, d_ff=192, E=8, K=3, shared_d_ff=160, skew=1.3),
    # strong skew: long segments (several units) beside segments of a few rows
    "skewed": _wl("k_3", T=2048, d=256, d_ff=384, E=32, K=2, n_shared=2, shared_d_ff=128,
                  skew=3.0),
    # sigmoid gate, no shared expert, 1024-wide d (two plain units per token tile)
    "sigmoid_noshared": _wl("k_4", T=600, d=1024, d_ff=256, E=4, K=2, n_shared=0,
                            shared_d_ff=0, gate="sigmoid", bias_std=0.0),
    # latent width 128 between the projections (the routed experts act on it)
    "latent": _wl("k_5", T=1024, d=256, d_ff=128, E=8, K=2, gate="sigmoid", latent_dim=128),
}


def _forward(A, w, inp, form=None):
    old = os.environ.get("MOE_GEMM_FORM")
    if form is None:
        os.environ.pop("MOE_GEMM_FORM", None)
    else:
        os.environ["MOE_GEMM_FORM"] = form
    try:
        spec = A.LayerSpec.of(w)
        ws = A.alloc_workspace(spec)
        out = A.forward(spec, inp["x"], inp, ws=ws).clone()
        st = A.workspace_status(ws)
        assert st == A.MOE_OK, A.status_string(st)
        return out
    finally:
        if old is None:
            os.environ.pop("MOE_GEMM_FORM", None)
        else:
            os.environ["MOE_GEMM_FORM"] = old


@pytest.mark.parametrize("name", list(LAYERS))
def test_token_form_matches_oracle_and_row_form(A, name):
    w = LAYERS[name]
    assert w.T * w.K >= 128 * w.E, "the layer must take the token-column form"
    inp = W.make_inputs(w, device="cuda")
    tok = _forward(A, w, inp)
    rows = _forward(A, w, inp, "rows")
    assert torch.isfinite(tok).all()
    # the two forms round the same products; any difference is the tensor
    # core's summation order inside one MMA, far below the BF16 bound
    diff = (tok - rows).abs().max().item()
    scale = rows.abs().max().item()
    assert diff <= 1e-4 * scale, (diff, scale)
    print(name, "bitwise" if torch.equal(tok.view(torch.int32), rows.view(torch.int32)) else diff)
    res = P.full_parity(w)
    print(name, res)


def _pairs_for(sizes):
    """Expert pairs (a, b, count) whose per-expert totals are `sizes`: the two
    experts with the most rows left are paired one token at a time."""
    left = list(sizes)
    out = {}
    while sum(left):
        order = sorted(range(len(left)), key=lambda e: -left[e])
        a, b = order[0], order[1]
        assert left[b] > 0, "no pairing"
        out[(a, b)] = out.get((a, b), 0) + 1
        left[a] -= 1
        left[b] -= 1
    return [(a, b, n) for (a, b), n in out.items()]


def test_segment_edges(A):
    """Segments of 0, 1, 15, 16, 255, 256, 257 and 600 rows, placed through the
    router: token class c has x = one-hot at dimension c (plus noise in the
    dimensions the router does not read) and W_router row c scores its two
    experts 5 and 4, every other expert 0."""
    from oracle import moe_oracle as O
    sizes = [0, 1, 15, 16, 255, 256, 257, 600]
    w = _wl("k_6", T=sum(sizes) // 2, d=256, d_ff=256, E=len(sizes), K=2, n_shared=1,
            shared_d_ff=128, bias_std=0.0, has_bias=False)
    pairs = _pairs_for(sizes)
    assert len(pairs) < 64
    inp = W.make_inputs(w, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(6)
    x = torch.randn(w.T, w.d, device="cuda", generator=gen)
    x[:, :64] = 0.0
    Wr = torch.zeros(w.d, w.E, device="cuda")
    t0 = 0
    for c, (a, b, n) in enumerate(pairs):
        x[t0:t0 + n, c] = 1.0
        Wr[c, a], Wr[c, b] = 5.0, 4.0
        t0 += n
    perm = torch.randperm(w.T, device="cuda", generator=gen)
    inp["x"] = x[perm].to(torch.bfloat16).contiguous()
    inp["W_router"] = Wr
    inp["bias"] = None
    tok = _forward(A, w, inp)
    rows = _forward(A, w, inp, "rows")
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    A.forward(spec, inp["x"], inp, ws=ws)
    counts = A.workspace_views(spec, ws)["counts"].cpu().numpy()
    assert list(counts) == sizes
    diff = (tok - rows).abs().max().item()
    assert diff <= 1e-4 * rows.abs().max().item(), diff
    ref = O.moe_forward_sorted(inp["x"], inp, w.gate, w.K, w.renormalize, w.routed_scale)
    P.check_output(w, tok, ref, None)
