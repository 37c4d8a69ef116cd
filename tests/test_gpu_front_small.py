"""The one-launch front end of prefill batches with few experts (router,
dispatch and row gather in one cooperative launch: BF16, E <= 8,
1024 < T*K <= 16384, no latent projection). Its routing equals the standalone
router's (moe_route) bit for bit, its dispatch the standalone dispatch's
(moe_dispatch), and the layer output the oracle's on every row; a dirty
workspace changes nothing (the grid barrier keeps no state between launches),
and the forward is one launch shorter than with the separate kernels.
"""
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
    base = dict(n_shared=1, shared_d_ff=128, dtype="bf16", gate="softmax_topk", bias_std=0.01)
    base.update(kw)
    return W.Workload(name, **base)


LAYERS = {
    # E = 4 with the vector W_router reads, tokens not a multiple of the CTA count
    "e4_k2": _wl("s_1", T=1500, d=256, d_ff=256, E=4, K=2),
    # E = 3 (scalar reads, EP = 4), K = 1, the smallest batch that takes the path
    "e3_k1": _wl("s_2", T=1025, d=64, d_ff=128, E=3, K=1, n_shared=0, shared_d_ff=0),
    # E = 8, K = 4, sigmoid with renormalisation and a routed scale
    "e8_sigmoid": _wl("s_3", T=700, d=512, d_ff=128, E=8, K=4, gate="sigmoid", bias_std=0.0,
                      renormalize=True, routed_scale=2.5),
    # E = 6 (EP = 8, scalar reads), softmax over all experts renormalised
    "e6_renorm_all": _wl("s_4", T=3000, d=192, d_ff=64, E=6, K=3,
                         gate="softmax_all_renorm", has_bias=False),
    # the largest batch (T*K = 16384) and a wide row (d = 2048)
    "e8_max": _wl("s_5", T=2048, d=2048, d_ff=128, E=8, K=8, n_shared=0, shared_d_ff=0),
    # E = 1: every token on the one expert
    "e1": _wl("s_6", T=2000, d=128, d_ff=64, E=1, K=1, has_bias=False),
}


@pytest.mark.parametrize("name", list(LAYERS))
def test_front_small_equals_separate_kernels_and_oracle(A, name):
    w = LAYERS[name]
    assert 1024 < w.T * w.K <= 16384 and w.E <= 8
    inp = W.make_inputs(w, device="cuda")
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    ws.fill_(0x5A)  # no initial state is needed
    n0 = A.launch_count()
    A.forward(spec, inp["x"], inp, ws=ws)
    n_fwd = A.launch_count() - n0
    assert A.workspace_status(ws) == A.MOE_OK
    v = A.workspace_views(spec, ws)
    r = A.route(spec, inp["x"], inp["W_router"], inp["bias"])
    for k in ("idx", "w", "margin") + (("top_scores", "scores") if w.gate == "sigmoid" else ()):
        assert torch.equal(v[k].view(torch.int32), r[k].view(torch.int32)), k
    dsp = A.dispatch(spec, r["idx"], r["w"])
    for k in ("counts", "offsets", "sorted_token", "inv"):
        assert torch.equal(v[k].reshape(-1), dsp[k].reshape(-1)), k
    assert torch.equal(v["sorted_w"].view(torch.int32), dsp["sorted_w"].view(torch.int32))
    # router, gate/up, down, combine: four launches
    assert n_fwd == 4, n_fwd
    res = P.full_parity(w)
    print(name, res)


def test_front_small_replays_in_a_graph(A):
    w = LAYERS["e4_k2"]
    inp = W.make_inputs(w, device="cuda")
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    out = torch.empty((w.T, w.d), dtype=spec.torch_out_dtype, device="cuda")
    A.forward(spec, inp["x"], inp, out=out, ws=ws)
    ref = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        A.forward(spec, inp["x"], inp, out=out, ws=ws, stream=s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
    assert A.workspace_status(ws) == A.MOE_OK
    # new tokens in place: every replay routes and counts them anew (a replay
    # must not pass the grid barrier on the previous replay's tags)
    for seed in (3, 4, 5):
        gen = torch.Generator(device="cuda").manual_seed(seed)
        inp["x"].copy_(torch.randn(w.T, w.d, device="cuda", generator=gen).to(inp["x"].dtype))
        g.replay()
        torch.cuda.synchronize()
        ref2 = A.forward(spec, inp["x"], inp, ws=A.alloc_workspace(spec))
        assert torch.equal(out.view(torch.int32), ref2.view(torch.int32)), seed
    assert A.workspace_status(ws) == A.MOE_OK


# Larger prefill batches (16384 < T*K <= 1024 per SM): the dispatch and the row
# gather in one cooperative launch with the same launch-id grid barrier.
ONEPASS = {
    "e64_k8": _wl("s_7", T=2500, d=256, d_ff=128, E=64, K=8, skew=1.2),
    "e256_k6_ragged": _wl("s_8", T=3001, d=320, d_ff=64, E=256, K=6, n_shared=0, shared_d_ff=0),
    "e8_k4_latent": _wl("s_9", T=4500, d=256, d_ff=128, E=8, K=4, gate="sigmoid", latent_dim=128),
}


@pytest.mark.parametrize("name", list(ONEPASS))
def test_onepass_dispatch_equals_two_launch_dispatch(A, name):
    w = ONEPASS[name]
    assert 16384 < w.T * w.K <= 1024 * torch.cuda.get_device_properties(0).multi_processor_count
    inp = W.make_inputs(w, device="cuda")
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    ws.fill_(0x3C)  # no initial state is needed
    out = A.forward(spec, inp["x"], inp, ws=ws).clone()
    assert A.workspace_status(ws) == A.MOE_OK
    v = A.workspace_views(spec, ws)
    dsp = A.dispatch(spec, v["idx"].clone(), v["w"].clone())
    for k in ("counts", "offsets", "sorted_token", "inv"):
        assert torch.equal(v[k].reshape(-1), dsp[k].reshape(-1)), k
    assert torch.equal(v["sorted_w"].view(torch.int32), dsp["sorted_w"].view(torch.int32))
    # replayed in a graph: the same bits
    o2 = torch.empty_like(out)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        A.forward(spec, inp["x"], inp, out=o2, ws=ws, stream=s)
    for _ in range(2):
        o2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o2.view(torch.int32), out.view(torch.int32))
    # new tokens in place: the replay follows them
    for seed in (3, 4):
        gen = torch.Generator(device="cuda").manual_seed(seed)
        src = inp["x"]
        src.copy_(torch.randn(src.shape, device="cuda", generator=gen).to(src.dtype))
        g.replay()
        torch.cuda.synchronize()
        ref2 = A.forward(spec, inp["x"], inp, ws=A.alloc_workspace(spec))
        assert torch.equal(o2.view(torch.int32), ref2.view(torch.int32)), seed
    assert A.workspace_status(ws) == A.MOE_OK
    res = P.full_parity(w)
    print(name, res)
