"""The one-launch decode router (at most 128 tokens, 128 < E <= 256, with a
workspace): its grid barrier keeps no state between launches, so a workspace
full of garbage, repeated calls and graph replays give the same routing bit
for bit, and the routing equals the oracle's outside near ties. Batches of
fewer than 128 tokens leave part of the CTA's warps on further parts of each
slice (their sums are added in part order)."""
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


CASES = {
    "large_decode_router": dict(T=128, d=4096, E=256, K=8, gate="softmax_topk"),
    "e192_t64": dict(T=64, d=2048, E=192, K=8, gate="softmax_topk"),
    # a partial last expert block (200 = 6 * 32 + 8)
    "t24_sigmoid_e200": dict(T=24, d=1008, E=200, K=6, gate="sigmoid"),
    # E not a multiple of 4: W_router columns copied one by one
    "e129_t100": dict(T=100, d=512, E=129, K=4, gate="softmax_all_renorm"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_decode_router_dirty_workspace_and_graph(A, name):
    c = CASES[name]
    w = W.Workload("rd", T=c["T"], d=c["d"], d_ff=16, E=c["E"], K=c["K"], n_shared=0, shared_d_ff=0,
                   dtype="bf16", gate=c["gate"], bias_std=0.02 if c["gate"] != "sigmoid" else 0.0,
                   skew=0.5 if c["gate"] != "sigmoid" else 0.0)
    inp = W.make_inputs(w, device="cuda")
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    ws.zero_()
    g0 = {k: v.clone() for k, v in A.route(spec, inp["x"], inp["W_router"], inp["bias"], ws=ws).items()
          if isinstance(v, torch.Tensor)}
    assert A.workspace_status(ws) == A.MOE_OK
    ws.fill_(0xA7)
    g1 = A.route(spec, inp["x"], inp["W_router"], inp["bias"], ws=ws)
    assert A.workspace_status(ws) == A.MOE_OK
    for k in ("idx", "w", "margin"):
        assert torch.equal(g0[k].view(torch.int32), g1[k].view(torch.int32)), k
    # replayed in a graph on the same (now used) workspace
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        gr = A.route(spec, inp["x"], inp["W_router"], inp["bias"], ws=ws, stream=s)
    for _ in range(3):
        gr["idx"].fill_(-1)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(gr["idx"], g0["idx"])
        assert torch.equal(gr["w"].view(torch.int32), g0["w"].view(torch.int32))
    assert A.workspace_status(ws) == A.MOE_OK
    # new tokens in place: each replay routes them anew (a replay must not pass
    # the grid barrier on the previous replay's tags and partials)
    x0 = inp["x"].clone()
    for seed in (3, 4, 5):
        gen = torch.Generator(device="cuda").manual_seed(seed)
        inp["x"].copy_(torch.randn(inp["x"].shape, device="cuda", generator=gen).to(inp["x"].dtype))
        graph.replay()
        torch.cuda.synchronize()
        e = A.route(spec, inp["x"], inp["W_router"], inp["bias"], ws=A.alloc_workspace(spec))
        assert torch.equal(gr["idx"], e["idx"]), seed
        assert torch.equal(gr["w"].view(torch.int32), e["w"].view(torch.int32)), seed
    assert A.workspace_status(ws) == A.MOE_OK
    inp["x"].copy_(x0)
    ort = P.oracle_routing(w, inp)
    near = ort["min_gap"] <= P.NEAR_TIE
    P.check_routing(w, ort, g0, near)
