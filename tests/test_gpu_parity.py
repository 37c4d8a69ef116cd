"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Small cases and the configurations at full size are compared element by
element on every output row, with routing and dispatch checked on every
token. Tolerances are in tests/parity.py.
"""
import os

import numpy as np
import pytest
import torch

from tests import parity as P
from mixture_experts_ffn_fp32_gb300 import workloads as W
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mixture_experts_ffn_fp32_gb300 import build
    build.build()
    yield
    torch.cuda.synchronize()


def api():
    from mixture_experts_ffn_fp32_gb300 import api as A
    return A


# Small layers that span several tiles and ragged tails in every dimension.
SMALL = {
    "f32_softmax_all": W.Workload("t_f32", T=300, d=96, d_ff=160, E=8, K=2, n_shared=1,
                                  shared_d_ff=112, dtype="f32", gate="softmax_all_renorm",
                                  has_bias=False),
    "f32_topk_noshared": W.Workload("t_f32b", T=77, d=64, d_ff=128, E=5, K=3, n_shared=0,
                                    shared_d_ff=0, dtype="f32", gate="softmax_topk",
                                    bias_std=0.01),
    "bf16_topk": W.Workload("t_b1", T=333, d=256, d_ff=384, E=16, K=4, n_shared=2,
                            shared_d_ff=256, dtype="bf16", gate="softmax_topk", bias_std=0.01),
    "bf16_topk_skew": W.Workload("t_b2", T=257, d=192, d_ff=176, E=40, K=6, n_shared=1,
                                 shared_d_ff=144, dtype="bf16", gate="softmax_topk",
                                 bias_std=0.01, skew=1.2),
    "bf16_renorm_all": W.Workload("t_b3", T=129, d=128, d_ff=256, E=8, K=2, n_shared=1,
                                  shared_d_ff=128, dtype="bf16", gate="softmax_all_renorm",
                                  has_bias=False),
    "bf16_noshared": W.Workload("t_b4", T=200, d=320, d_ff=208, E=12, K=3, n_shared=0,
                                shared_d_ff=0, dtype="bf16", gate="softmax_topk", bias_std=0.01),
    "bf16_sigmoid_latent": W.Workload("t_b5", T=190, d=256, d_ff=192, E=24, K=4, n_shared=1,
                                      shared_d_ff=320, dtype="bf16", gate="sigmoid",
                                      latent_dim=96),
    "bf16_sigmoid_renorm": W.Workload("t_b6", T=150, d=128, d_ff=128, E=16, K=3, n_shared=2,
                                      shared_d_ff=64, dtype="bf16", gate="sigmoid",
                                      renormalize=True, routed_scale=2.5),
    "bf16_sigmoid_latent_noshared": W.Workload("t_b7", T=64, d=128, d_ff=64, E=10, K=2,
                                               n_shared=0, shared_d_ff=0, dtype="bf16",
                                               gate="sigmoid", latent_dim=64),
    "bf16_one_token": W.Workload("t_b8", T=1, d=128, d_ff=128, E=6, K=2, n_shared=1,
                                 shared_d_ff=128, dtype="bf16", gate="softmax_topk",
                                 bias_std=0.01),
    "bf16_k_eq_e": W.Workload("t_b9", T=70, d=64, d_ff=64, E=4, K=4, n_shared=1,
                              shared_d_ff=64, dtype="bf16", gate="softmax_topk", bias_std=0.01),
    "bf16_e1": W.Workload("t_b10", T=140, d=64, d_ff=96, E=1, K=1, n_shared=0, shared_d_ff=0,
                          dtype="bf16", gate="softmax_topk", has_bias=False),
    "f32_one_token": W.Workload("t_f3", T=1, d=64, d_ff=64, E=4, K=2, n_shared=1,
                                shared_d_ff=64, dtype="f32", gate="softmax_all_renorm",
                                has_bias=False),
    "bf16_e256": W.Workload("t_b11", T=96, d=128, d_ff=128, E=256, K=8, n_shared=1,
                            shared_d_ff=128, dtype="bf16", gate="softmax_topk", bias_std=0.01,
                            skew=1.2),
    # Segments averaging >= 512 rows: the grouped GEMMs run as CTA pairs (256-row
    # tiles). Skew leaves some experts with fewer than 128 rows (the odd CTA of
    # a pair has no rows), widths that are not multiples of 64 take the per-strip
    # copies, and reduction lengths of 3.25 / 2.75 k-blocks end on a half-full
    # two-k-block stage.
    "pair_skew": W.Workload("t_p1", T=1200, d=256, d_ff=384, E=4, K=2, n_shared=1,
                            shared_d_ff=256, dtype="bf16", gate="softmax_topk", bias_std=0.01,
                            skew=1.5),
    "pair_ragged_widths": W.Workload("t_p2", T=1100, d=208, d_ff=176, E=2, K=1, n_shared=1,
                                     shared_d_ff=144, dtype="bf16", gate="softmax_topk",
                                     bias_std=0.01),
    "pair_latent_sigmoid": W.Workload("t_p3", T=1024, d=256, d_ff=192, E=4, K=2, n_shared=1,
                                      shared_d_ff=256, dtype="bf16", gate="sigmoid",
                                      latent_dim=128),
    # Decode batches (32 < E <= 128, T*K <= 1024): the cluster router and the
    # one-launch dispatch + gather. Ragged last token block and last slice of d,
    # both expert widths of the router (64 and 128 lanes), FP32 and BF16, the
    # sigmoid gate (top_scores/scores) on latent rows, exactly 1024 assignments.
    "decode_e64_ragged": W.Workload("t_d1", T=100, d=720, d_ff=128, E=64, K=8, n_shared=1,
                                   shared_d_ff=128, dtype="bf16", gate="softmax_topk",
                                   bias_std=0.01, skew=1.1),
    "decode_f32_e96": W.Workload("t_d2", T=37, d=208, d_ff=96, E=96, K=5, n_shared=1,
                                shared_d_ff=64, dtype="f32", gate="softmax_all_renorm",
                                has_bias=False),
    "decode_sigmoid_latent": W.Workload("t_d3", T=60, d=256, d_ff=64, E=48, K=4, n_shared=1,
                                       shared_d_ff=128, dtype="bf16", gate="sigmoid",
                                       latent_dim=64),
    "decode_max_assignments": W.Workload("t_d4", T=128, d=384, d_ff=64, E=128, K=8, n_shared=0,
                                        shared_d_ff=0, dtype="bf16", gate="softmax_topk",
                                        bias_std=0.01),
    # Batches of 1025..16384 assignments: dispatch and gather in one launch over
    # many CTAs (each counts every assignment itself). A flat-id count that is
    # not a multiple of four (the scalar tail of the id loads) with more than 64
    # experts (per-warp shared counters), and exactly 16384 assignments with
    # 16 experts.
    "wide_e96_tail": W.Workload("t_w1", T=701, d=192, d_ff=128, E=96, K=6, n_shared=1,
                                shared_d_ff=128, dtype="bf16", gate="softmax_topk",
                                bias_std=0.01, skew=1.2),
    "wide_max_assignments": W.Workload("t_w2", T=2048, d=128, d_ff=64, E=16, K=8, n_shared=0,
                                       shared_d_ff=0, dtype="bf16", gate="softmax_topk",
                                       bias_std=0.01),
    # 16800 assignments: the two-launch dispatch (chunk histograms, then the scatter)
    # and the separate row gather
    "two_launch_dispatch": W.Workload("t_w3", T=4200, d=64, d_ff=64, E=12, K=4, n_shared=1,
                                      shared_d_ff=64, dtype="bf16", gate="softmax_topk",
                                      bias_std=0.01, skew=0.8),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_layer_all_rows(name):
    res = P.full_parity(SMALL[name])
    print(name, res)


@pytest.mark.parametrize("name", ["tiny_f32"])
def test_tiny_f32_full_size_all_rows(name):
    res = P.full_parity(W.WORKLOADS[name])
    print(name, res)


FULL = ["small", "medium_prefill", "medium_decode", "large_prefill", "large_prefill_zipf",
        "large_decode", "large_decode_zipf", "latent"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_all_rows(name):
    """Every benchmark configuration at full size, every output row against the
    oracle (its expert-grouped form). MOE_PARITY_RECORD names a file that gets
    one JSON line per layer (near-tie count, max error, RMS, rows)."""
    res = P.full_parity(W.WORKLOADS[name], record=os.environ.get("MOE_PARITY_RECORD"))
    print(name, res)


def test_sampled_rows_cover_tiles_and_rare_experts():
    """The sampled row set used where every row would cost too much: evenly
    spaced tokens, every token of the rarest experts, tile boundaries."""
    w = W.WORKLOADS["large_prefill_zipf"]
    res = P.full_parity(w, sample=True)
    assert res["rows"] >= 512, res
    print(res)


# ---------------------------------------------------------------------------
# Router and dispatch on their own
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("gate,E,K", [("softmax_topk", 4, 2), ("softmax_topk", 64, 8),
                                      ("softmax_topk", 256, 8), ("softmax_all_renorm", 8, 2),
                                      ("softmax_all_renorm", 100, 7), ("sigmoid", 128, 8),
                                      ("sigmoid", 9, 8), ("softmax_topk", 33, 16),
                                      ("sigmoid", 20, 1), ("sigmoid", 8, 3), ("softmax_topk", 5, 5),
                                      ("softmax_all_renorm", 3, 1)])
@pytest.mark.parametrize("dtype,d,with_ws", [("bf16", 272, False), ("f32", 272, False),
                                             ("bf16", 256, True), ("bf16", 1024, True)])
def test_route(gate, E, K, dtype, d, with_ws):
    """Both router paths: the fused FP32 FMA kernel, and (BF16, E > 32, E % 8 == 0,
    d % 64 == 0, with a workspace) the tensor-core split-weight router."""
    A = api()
    w = W.Workload("r", T=517, d=d, d_ff=16, E=E, K=K, n_shared=0, shared_d_ff=0, dtype=dtype,
                   gate=gate, bias_std=0.02, skew=0.5 if gate != "sigmoid" else 0.0)
    inp = W.make_inputs(w, device="cuda")
    if gate == "sigmoid":
        inp["bias"] = (torch.randn(E, generator=torch.Generator().manual_seed(5)) * 0.05).cuda()
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec) if with_ws else None
    g = A.route(spec, inp["x"], inp["W_router"], inp["bias"], ws=ws)
    if ws is not None:
        assert A.workspace_status(ws) == A.MOE_OK
    ort = P.oracle_routing(w, inp)
    near = ort["min_gap"] <= P.NEAR_TIE
    P.check_routing(w, ort, g, near)


@pytest.mark.parametrize("gate,E,K", [("softmax_topk", 64, 8), ("softmax_topk", 256, 8),
                                      ("sigmoid", 128, 8), ("softmax_all_renorm", 100, 7),
                                      ("softmax_topk", 33, 16), ("sigmoid", 120, 4)])
@pytest.mark.parametrize("dtype,d,T", [("bf16", 272, 200), ("f32", 1024, 64), ("bf16", 4096, 1),
                                       ("bf16", 4096, 128), ("bf16", 2048, 64), ("f32", 112, 33)])
def test_route_few_tokens(gate, E, K, dtype, d, T):
    """Few tokens with 32 < E <= 256 and a workspace. Up to 128 tokens and more
    than 128 experts: the one-launch decode router (every CTA one slice of d for
    32 experts and all tokens, partials summed in slice order after a grid
    barrier), with ragged last slices, token counts that leave warps idle, a
    single token and the 128-token, 4096-wide, 256-expert batch; otherwise the
    FP32 cluster router (slices summed in slice order through distributed shared
    memory)."""
    A = api()
    w = W.Workload("r", T=T, d=d, d_ff=16, E=E, K=K, n_shared=0, shared_d_ff=0, dtype=dtype,
                   gate=gate, bias_std=0.02, skew=0.5 if gate != "sigmoid" else 0.0)
    inp = W.make_inputs(w, device="cuda")
    if gate == "sigmoid":
        inp["bias"] = (torch.randn(E, generator=torch.Generator().manual_seed(6)) * 0.05).cuda()
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    g = A.route(spec, inp["x"], inp["W_router"], inp["bias"], ws=ws)
    assert A.workspace_status(ws) == A.MOE_OK
    ort = P.oracle_routing(w, inp)
    near = ort["min_gap"] <= P.NEAR_TIE
    P.check_routing(w, ort, g, near)


@pytest.mark.parametrize("gate,E,K,T,d,dtype", [
    ("softmax_topk", 4, 2, 4096, 768, "bf16"),       # the 4096-token layer's router
    ("softmax_all_renorm", 8, 2, 300, 96, "f32"),
    ("softmax_topk", 64, 8, 200, 272, "bf16"),       # chunked router
    ("softmax_topk", 256, 8, 1030, 512, "bf16"),     # tensor-core router, ragged CTA tail
    ("sigmoid", 128, 8, 777, 256, "bf16"),
    ("softmax_topk", 16, 4, 1, 64, "f32")])
def test_routing_stats(gate, E, K, T, d, dtype):
    """Switch loss, z-loss and mean probabilities against the oracle's
    routing_stats on the GPU's own selection (f is a count of it), and
    reproducible bit for bit."""
    A = api()
    w = W.Workload("s", T=T, d=d, d_ff=16, E=E, K=K, n_shared=0, shared_d_ff=0, dtype=dtype,
                   gate=gate, bias_std=0.02, skew=0.5 if gate != "sigmoid" else 0.0)
    inp = W.make_inputs(w, device="cuda")
    spec = A.LayerSpec.of(w)
    g = A.routing_stats(spec, inp["x"], inp["W_router"], inp["bias"])
    assert A.workspace_status(g["ws"]) == A.MOE_OK
    gidx = P.npi(A.workspace_views(spec, g["ws"])["idx"])
    # the selection itself matches the oracle's outside near ties
    ort = P.oracle_routing(w, inp)
    near = ort["min_gap"] <= P.NEAR_TIE
    assert (gidx[~near] == ort["idx"][~near]).all()
    ref = O.routing_stats(ort["logits"], gidx, E)
    assert abs(g["aux"] - ref["aux"]) <= 2e-5 * max(1.0, abs(ref["aux"]))
    assert abs(g["z"] - ref["z"]) <= 2e-5 * max(1.0, abs(ref["z"]))
    np.testing.assert_allclose(P.np64(g["P"]), ref["P"], atol=2e-6, rtol=2e-5)
    g2 = A.routing_stats(spec, inp["x"], inp["W_router"], inp["bias"], ws=g["ws"])
    assert torch.equal(g["out"], g2["out"])


@pytest.mark.parametrize("T,E,K,skew", [(1, 1, 1, 0.0), (3, 3, 2, 0.0), (128, 256, 8, 0.0),
                                        (125, 64, 8, 1.1), (512, 5, 2, 0.8), (1000, 8, 2, 0.0),
                                        (1500, 64, 8, 1.1), (4096, 256, 8, 1.2),
                                        (777, 256, 16, 0.0), (20000, 7, 3, 0.5),
                                        (16384, 64, 8, 1.1)])
def test_dispatch_bit_exact(T, E, K, skew):
    A = api()
    idx, wts = W.random_routing(T, E, K, device="cuda", seed=T + E, skew=skew)
    spec = A.LayerSpec(T=T, d=16, d_ff=16, E=E, K=K)
    g = A.dispatch(spec, idx, wts)
    w = W.Workload("d", T=T, d=16, d_ff=16, E=E, K=K, n_shared=0, shared_d_ff=0, dtype="bf16",
                   gate="softmax_topk")
    P.check_dispatch(w, P.npi(idx), wts.cpu().numpy().reshape(-1), g)
    assert A.workspace_status(g["ws"]) == A.MOE_OK


@pytest.mark.parametrize("name", ["wide_e96_tail", "wide_max_assignments", "bf16_topk",
                                  "pair_skew", "decode_e64_ragged", "bf16_e256",
                                  "two_launch_dispatch"])
def test_forward_dispatch_bit_exact(name):
    """The dispatch a forward leaves in its workspace (one-launch single-CTA,
    one-launch many-CTA or two-launch form) is the oracle's stable dispatch of
    the forward's own routing, bit for bit."""
    A = api()
    w = SMALL[name]
    inp = W.make_inputs(w, device="cuda")
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    A.forward(spec, inp["x"], inp, ws=ws)
    v = A.workspace_views(spec, ws)
    P.check_dispatch(w, P.npi(v["idx"]), v["w"].cpu().numpy().reshape(-1), v)
    assert A.workspace_status(ws) == A.MOE_OK


def test_dispatch_worked_example():
    """kimi_k3 StableLatentMoE illustration: [[2,0],[0,2],[2,1]]."""
    A = api()
    idx = torch.tensor([[2, 0], [0, 2], [2, 1]], dtype=torch.int32, device="cuda")
    wts = torch.arange(6, dtype=torch.float32, device="cuda").view(3, 2)
    g = A.dispatch(A.LayerSpec(T=3, d=16, d_ff=16, E=3, K=2), idx, wts)
    assert g["sorted_token"].tolist() == [0, 1, 2, 0, 1, 2]
    assert g["counts"].tolist() == [2, 1, 3]
    assert g["offsets"].tolist() == [0, 2, 3, 6]
    assert g["sorted_w"].tolist() == [1.0, 2.0, 5.0, 0.0, 3.0, 4.0]


def test_dispatch_flags_out_of_range_ids():
    A = api()
    idx = torch.tensor([[0, 1], [5, 1], [1, -1]], dtype=torch.int32, device="cuda")
    wts = torch.ones(3, 2, device="cuda")
    g = A.dispatch(A.LayerSpec(T=3, d=16, d_ff=16, E=3, K=2), idx, wts)
    assert A.workspace_status(g["ws"]) == A.MOE_ERR_DEVICE_INDEX
    assert g["counts"].tolist() == [1, 3, 0]
    assert A.workspace_status(g["ws"]) == A.MOE_OK  # cleared by the read


# ---------------------------------------------------------------------------
# Balancers
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,K", [(8192, 128, 8), (1000, 16, 4), (7, 4, 2), (4096, 256, 8)])
def test_quantile_bias_update_bit_exact(T, E, K):
    A = api()
    g = torch.Generator(device="cuda").manual_seed(T * 7 + E)
    s = torch.sigmoid(torch.randn(T, E, device="cuda", generator=g))
    b = torch.randn(E, device="cuda", generator=g) * 0.1
    top = torch.topk(s + b, K + 1, dim=1).values.contiguous()
    bias = torch.zeros(E, device="cuda")
    A.quantile_bias_update(top, s, K, bias)
    ref = O.quantile_bias_update(top.cpu().numpy(), s.cpu().numpy(), K)
    assert np.array_equal(bias.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_quantile_update_after_latent_forward():
    """The latent layer's forward leaves top_scores / scores in its workspace;
    the update on them equals the oracle's bit for bit, and a second forward
    with the new bias still matches the oracle."""
    A = api()
    w = W.WORKLOADS["latent"].resized(T=1024)
    inp = W.make_inputs(w, device="cuda")
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    A.forward(spec, inp["x"], inp, ws=ws)
    v = A.workspace_views(spec, ws)
    bias = inp["bias"].clone()
    A.quantile_bias_update(v["top_scores"], v["scores"], w.K, bias)
    ref = O.quantile_bias_update(v["top_scores"].cpu().numpy(), v["scores"].cpu().numpy(), w.K)
    assert np.array_equal(bias.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert abs(float(bias.double().sum())) < 1e-4
    inp["bias"] = bias
    out, views, ws2 = P.run_forward(w, inp)
    ort = P.oracle_routing(w, inp)
    idx, wts, near = P.merge_routing(w, inp, ort, P.npi(views["idx"]))
    P.check_routing(w, ort, views, near)
    rows = list(range(0, w.T, 97))
    ref_out, _ = O.moe_forward(inp["x"], inp, w.gate, w.K, tokens=rows, routing=(idx, wts))
    P.check_output(w, out, ref_out, rows)


def test_sign_bias_update():
    A = api()
    counts = torch.tensor([5, 4, 3, 4], dtype=torch.int32, device="cuda")
    bias = torch.zeros(4, device="cuda")
    A.sign_bias_update(counts, 8, 2, bias, 0.1)
    np.testing.assert_allclose(bias.cpu().numpy(), [-0.1, 0.0, 0.1, 0.0], atol=1e-7)
    g = torch.Generator().manual_seed(3)
    c = torch.randint(0, 50, (64,), generator=g, dtype=torch.int32)
    b0 = (torch.rand(64, generator=g) * 2 - 1)
    bias = b0.clone().cuda()
    A.sign_bias_update(c.cuda(), 400, 8, bias, 0.05)
    ref = O.sign_bias_update(c.numpy(), 400, 8, b0.numpy(), 0.05)
    np.testing.assert_allclose(bias.cpu().numpy(), ref, atol=1e-7)


# ---------------------------------------------------------------------------
# API behaviour
# ---------------------------------------------------------------------------

def test_forward_deterministic_and_host_variant():
    A = api()
    w = W.WORKLOADS["small"].resized(T=1000)
    inp = W.make_inputs(w, device="cuda")
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    o1 = A.forward(spec, inp["x"], inp, ws=ws).clone()
    o2 = A.forward(spec, inp["x"], inp, ws=ws).clone()
    assert torch.equal(o1.view(torch.int32), o2.view(torch.int32))
    xh = inp["x"].cpu().pin_memory()
    oh = torch.empty((w.T, w.d), dtype=torch.float32).pin_memory()
    A.forward_host(spec, xh, inp, oh, ws)
    assert torch.equal(oh.view(torch.int32), o1.cpu().view(torch.int32))
    assert A.workspace_status(ws) == A.MOE_OK
    # BF16 output: the same FP32 result rounded once to nearest-even
    sb = A.LayerSpec.of(w, out_dtype="bf16")
    ob = A.forward(sb, inp["x"], inp, ws=ws)
    assert ob.dtype == torch.bfloat16
    assert torch.equal(ob.view(torch.int16), o1.to(torch.bfloat16).view(torch.int16))


def test_launch_count_grows():
    A = api()
    w = W.WORKLOADS["tiny_f32"]
    inp = W.make_inputs(w, device="cuda")
    n0 = A.launch_count()
    A.forward(A.LayerSpec.of(w), inp["x"], inp)
    torch.cuda.synchronize()
    # router, single-CTA dispatch (T*K = 256 assignments), gate/up, routed down,
    # shared down fused with the combine
    assert A.launch_count() - n0 == 5


def test_decode_launches_and_dirty_workspace():
    """A decode batch routes in one cluster launch and runs everything else in
    one more (the fused decode back end); nothing in the workspace carries over
    between forwards, so a workspace full of garbage gives the same result, bit
    for bit."""
    A = api()
    w = W.WORKLOADS["medium_decode"].resized(T=64, d=512, d_ff=128)
    inp = W.make_inputs(w, device="cuda")
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    torch.cuda.synchronize()
    n0 = A.launch_count()
    o1 = A.forward(spec, inp["x"], inp, ws=ws).clone()
    torch.cuda.synchronize()
    # router, fused back end
    assert A.launch_count() - n0 == 2
    ws.fill_(0xFF)
    o2 = A.forward(spec, inp["x"], inp, ws=ws).clone()
    assert A.workspace_status(ws) == A.MOE_OK
    assert torch.equal(o1.view(torch.int32), o2.view(torch.int32))
    o3 = A.forward(spec, inp["x"], inp, ws=ws)
    assert torch.equal(o1.view(torch.int32), o3.view(torch.int32))


def test_bounded_wait_gives_up_and_context_survives():
    A = api()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    st = A.selftest_wait_timeout(20, ws)
    assert st == A.MOE_ERR_TIMEOUT
    # the context is still usable and the error word was cleared
    assert A.workspace_status(ws) == A.MOE_OK
    P.full_parity(SMALL["bf16_one_token"])
