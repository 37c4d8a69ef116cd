"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (for example a runtime that owns all device memory,
or code that must not call cudaMalloc after start-up). It keeps its scratch
in a fixed array inside the library instead of a caller workspace; its
results must equal moe_dispatch's bit for bit, call after call.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from mixture_experts_ffn_fp32_gb300 import build
    build.build()
    from mixture_experts_ffn_fp32_gb300 import api
    return api


def _routing(T, E, K, seed):
    from mixture_experts_ffn_fp32_gb300 import workloads as W
    return W.random_routing(T, E, K, device="cuda", seed=seed, skew=0.8)


@pytest.mark.parametrize("T,E,K", [(4096, 4, 2), (3000, 64, 8), (8192, 256, 8), (1, 3, 2)])
def test_noalloc_dispatch_matches_workspace_dispatch(A, T, E, K):
    spec = A.LayerSpec(T=T, d=16, d_ff=16, E=E, K=K)
    for call in range(2):  # two calls in a row reuse the library's scratch array
        idx, w = _routing(T, E, K, seed=1000 * call + T + E)
        ref = A.dispatch(spec, idx, w)
        got = A.dispatch_noalloc(spec, idx, w)
        torch.cuda.synchronize()
        for key in ("counts", "offsets", "sorted_token", "inv"):
            assert torch.equal(got[key], ref[key]), (call, key)
        assert torch.equal(got["sorted_w"].view(torch.int32), ref["sorted_w"].view(torch.int32))
        assert A.workspace_status(ref["ws"]) == A.MOE_OK


def test_noalloc_dispatch_rejects_sizes_beyond_its_array(A):
    spec = A.LayerSpec(T=16384, d=16, d_ff=16, E=64, K=8)  # T*K = 131072 > 65536
    idx, w = _routing(16384, 64, 8, seed=7)
    with pytest.raises(A.MoeError) as ei:
        A.dispatch_noalloc(spec, idx, w)
    assert ei.value.status == A.MOE_ERR_UNSUPPORTED
