"""The fused decode path: a decode batch of a BF16 layer without latent
projection (at most 128 tokens, T*K <= 1024, widths multiples of 64) runs in
two launches, the router and one persistent kernel for everything after it
(dispatch, row gather, grouped gate/up, grouped down, shared experts,
combine). Its output equals that of the separate launches bit for bit (a
forward with save_gate_up set takes the separate launches, and keeping the
gate/up products changes no bit of the output), and the oracle within the
BF16 bound on every row.
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
    # ragged rows and columns: d not a multiple of 256 (a half-empty last down
    # tile), F not a multiple of 128, the cluster router
    "e64_ragged": _wl("f_1", T=100, d=320, d_ff=192, E=64, K=6, skew=1.1),
    # 256 experts (the cluster router reading W_router from global memory), two
    # shared experts narrower than a 128-column tile
    "e256_two_shared": _wl("f_2", T=128, d=512, d_ff=128, E=256, K=8, n_shared=2,
                           shared_d_ff=64, skew=1.2),
    # few experts (the warp-per-token router), no shared expert
    "e16_no_shared": _wl("f_3", T=40, d=256, d_ff=256, E=16, K=4, n_shared=0, shared_d_ff=0),
    # strong skew: one expert takes nearly every token (a full 128-row unit)
    "one_hot_expert": _wl("f_4", T=128, d=256, d_ff=128, E=33, K=2, skew=4.0),
    "one_token": _wl("f_5", T=1, d=128, d_ff=64, E=48, K=3, shared_d_ff=64),
    "k_eq_e": _wl("f_6", T=16, d=128, d_ff=128, E=8, K=8),
    "sigmoid": _wl("f_7", T=60, d=256, d_ff=128, E=64, K=6, gate="sigmoid", bias_std=0.0),
    "renorm_all": _wl("f_8", T=96, d=192, d_ff=64, E=40, K=2, gate="softmax_all_renorm",
                      has_bias=False),
    "max_assignments": _wl("f_9", T=128, d=384, d_ff=64, E=128, K=8, n_shared=0,
                           shared_d_ff=0),
}


def _forward(A, spec, inp, ws):
    out = A.forward(spec, inp["x"], inp, ws=ws).clone()
    st = A.workspace_status(ws)
    assert st == A.MOE_OK, A.status_string(st)
    return out


@pytest.mark.parametrize("name", list(LAYERS))
def test_fused_equals_separate_launches_and_oracle(A, name):
    w = LAYERS[name]
    inp = W.make_inputs(w, device="cuda")
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    n0 = A.launch_count()
    fused = _forward(A, spec, inp, ws)
    assert A.launch_count() - n0 == 2, "router + the fused back end"
    sep_spec = A.LayerSpec.of(w, save_gate_up=True)
    sws = A.alloc_workspace(sep_spec)
    n0 = A.launch_count()
    sep = _forward(A, sep_spec, inp, sws)
    assert A.launch_count() - n0 > 2
    assert torch.equal(fused.view(torch.int32), sep.view(torch.int32))
    # the dispatch the fused kernel wrote out equals the separate dispatch's
    fv, sv = A.workspace_views(spec, ws), A.workspace_views(sep_spec, sws)
    for k in ("counts", "offsets", "sorted_token", "inv"):
        assert torch.equal(fv[k], sv[k]), k
    assert torch.equal(fv["sorted_w"].view(torch.int32), sv["sorted_w"].view(torch.int32))
    res = P.full_parity(w)
    print(name, res)


def test_fused_bf16_output_and_dirty_workspace(A):
    w = LAYERS["e64_ragged"]
    inp = W.make_inputs(w, device="cuda")
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    o1 = _forward(A, spec, inp, ws)
    ws.fill_(0xFF)  # garbage counters and buffers: the router zeroes what must start at zero
    o2 = _forward(A, spec, inp, ws)
    assert torch.equal(o1.view(torch.int32), o2.view(torch.int32))
    sb = A.LayerSpec.of(w, out_dtype="bf16")
    ob = A.forward(sb, inp["x"], inp, ws=ws)
    assert A.workspace_status(ws) == A.MOE_OK
    assert torch.equal(ob.view(torch.int16), o1.to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("name", ["medium_decode", "large_decode", "large_decode_zipf"])
def test_full_size_decode_two_launches_bit_exact(A, name):
    """The decode configurations: two launches, and the same bits as the
    separate launches (oracle parity on every row: test_full_size_all_rows)."""
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w, device="cuda")
    spec = A.LayerSpec.of(w)
    ws = A.alloc_workspace(spec)
    _forward(A, spec, inp, ws)
    torch.cuda.synchronize()
    n0 = A.launch_count()
    fused = _forward(A, spec, inp, ws)
    assert A.launch_count() - n0 == 2
    sep_spec = A.LayerSpec.of(w, save_gate_up=True)
    sep = _forward(A, sep_spec, inp, A.alloc_workspace(sep_spec))
    assert torch.equal(fused.view(torch.int32), sep.view(torch.int32))
    del inp, ws
    torch.cuda.empty_cache()
