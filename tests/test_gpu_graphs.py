"""moe_forward and moe_backward captured into a CUDA graph and replayed.

Neither call synchronises, allocates or reads device memory on the host, so
both can be captured: a replay must give the same bits as an eager call, and
a replay after the inputs were overwritten in place must follow the new
inputs (nothing of the captured call's data is baked into the graph).
Layers: the many-CTA dispatch (a ragged 1332-assignment batch), the CTA-pair
GEMMs, a decode batch (cluster router, one-launch dispatch + gather) and the
two-launch dispatch whose last histogram CTA re-arms its ticket.
"""
import pytest
import torch

from mixture_experts_ffn_fp32_gb300 import api as A
from mixture_experts_ffn_fp32_gb300 import workloads as W
from tests.test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int32) if t.dtype == torch.float32 else t.contiguous().view(torch.int16)


@pytest.mark.parametrize("name", ["bf16_topk", "pair_skew", "decode_e64_ragged", "two_launch_dispatch"])
def test_forward_captured_in_graph(name):
    w = SMALL[name]
    spec = A.LayerSpec.of(w)
    inp = W.make_inputs(w, device="cuda")
    ws = A.alloc_workspace(spec)
    out = torch.empty((w.T, w.d), dtype=spec.torch_out_dtype, device="cuda")
    ref = A.forward(spec, inp["x"], inp, ws=ws).clone()  # eager (also first-use setup)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        A.forward(spec, inp["x"], inp, out=out, ws=ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(ref))
    # new token values in place: the replay follows them
    gen = torch.Generator(device="cuda").manual_seed(11)
    inp["x"].copy_(torch.randn(w.T, w.d, device="cuda", generator=gen).to(inp["x"].dtype))
    g.replay()
    torch.cuda.synchronize()
    ref2 = A.forward(spec, inp["x"], inp, ws=A.alloc_workspace(spec))
    assert torch.equal(_bits(out), _bits(ref2))
    assert not torch.equal(_bits(ref2), _bits(ref))
    assert A.workspace_status(ws) == A.MOE_OK


@pytest.mark.parametrize("saved", [False, True])
def test_forward_and_backward_captured_in_graph(saved):
    w = W.Workload("t_g1", T=150, d=128, d_ff=192, E=6, K=2, n_shared=1, shared_d_ff=128,
                   dtype="bf16", gate="softmax_topk", bias_std=0.01, skew=1.2)
    spec = A.LayerSpec.of(w, save_gate_up=saved)
    inp = W.make_inputs(w, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(5)
    dout = torch.randn(w.T, w.d, device="cuda", generator=gen)
    ws = A.alloc_workspace(spec)
    bws = torch.empty(A.backward_workspace_size(spec), dtype=torch.uint8, device="cuda")
    shapes = A.grad_shapes(spec)
    grads = {n: torch.zeros(shp, device="cuda") for n, shp in shapes.items()}
    out = torch.empty((w.T, w.d), dtype=spec.torch_out_dtype, device="cuda")
    # eager reference (also the first-use setup of every kernel)
    A.forward(spec, inp["x"], inp, out=out, ws=ws)
    ref = A.backward(spec, inp["x"], inp, dout, ws, grads={n: torch.zeros_like(v) for n, v in grads.items()},
                     bws=bws)
    ref = {n: v.clone() for n, v in ref.items()}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        A.forward(spec, inp["x"], inp, out=out, ws=ws, stream=s)
        A.backward(spec, inp["x"], inp, dout, ws, grads=grads, bws=bws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    for n in ref:
        assert torch.equal(_bits(grads[n]), _bits(ref[n])), n
    assert A.workspace_status(ws) == A.MOE_OK
