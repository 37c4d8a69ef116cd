"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (for example a runtime that owns all device memory,
or code that must not call cudaMalloc after start-up). It keeps its scratch
in a fixed array inside the library instead of a caller workspace; its
results must equal moe_dispatch's bit for bit, and the oracle's stable
dispatch, call after call.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
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
    from oracle import moe_oracle as O
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
        # and the oracle's stable counting sort of the same ids
        dp = O.dispatch(idx.cpu().numpy(), E)
        assert np.array_equal(got["counts"].cpu().numpy(), dp["counts"])
        assert np.array_equal(got["offsets"].cpu().numpy(), dp["offsets"])
        assert np.array_equal(got["sorted_token"].cpu().numpy(), dp["sorted_token"])
        assert np.array_equal(got["inv"].cpu().numpy().reshape(-1), dp["inv"].reshape(-1))
        assert np.array_equal(got["sorted_w"].cpu().numpy(),
                              w.cpu().numpy().reshape(-1)[dp["order"]])


def test_noalloc_dispatch_skips_an_out_of_range_id(A):
    """One id equal to E: it is skipped, offsets[E] = T*K - 1 tells the caller,
    and every other assignment lands where the dispatch of the valid ones puts
    it (the same as moe_dispatch)."""
    T, E, K = 500, 16, 4
    spec = A.LayerSpec(T=T, d=16, d_ff=16, E=E, K=K)
    idx, w = _routing(T, E, K, seed=11)
    bad = (123, 2)
    idx[bad] = E
    got = A.dispatch_noalloc(spec, idx, w)
    ref = A.dispatch(spec, idx, w)
    torch.cuda.synchronize()
    assert A.workspace_status(ref["ws"]) == A.MOE_ERR_DEVICE_INDEX
    off = got["offsets"].cpu().numpy()
    assert off[E] == T * K - 1
    for key in ("counts", "offsets"):
        assert torch.equal(got[key], ref[key]), key
    n = int(off[E])
    assert torch.equal(got["sorted_token"][:n], ref["sorted_token"][:n])
    valid = torch.ones(T, K, dtype=torch.bool, device="cuda")
    valid[bad] = False
    assert torch.equal(got["inv"][valid], ref["inv"][valid])
    # the valid assignments against the oracle's stable order of them
    ids = idx.cpu().numpy().reshape(-1)
    keep = np.flatnonzero(ids < E)
    order = keep[np.argsort(ids[keep], kind="stable")]
    assert np.array_equal(got["sorted_token"][:n].cpu().numpy(), order // K)
    assert np.array_equal(np.bincount(ids[keep], minlength=E), got["counts"].cpu().numpy())
    # a following call with valid ids gives the moe_dispatch results again
    idx2, w2 = _routing(T, E, K, seed=12)
    got2 = A.dispatch_noalloc(spec, idx2, w2)
    ref2 = A.dispatch(spec, idx2, w2)
    torch.cuda.synchronize()
    for key in ("counts", "offsets", "sorted_token", "inv"):
        assert torch.equal(got2[key], ref2[key]), key


def test_noalloc_dispatch_rejects_sizes_beyond_its_array(A):
    spec = A.LayerSpec(T=16384, d=16, d_ff=16, E=64, K=8)  # T*K = 131072 > 65536
    idx, w = _routing(16384, 64, 8, seed=7)
    with pytest.raises(A.MoeError) as ei:
        A.dispatch_noalloc(spec, idx, w)
    assert ei.value.status == A.MOE_ERR_UNSUPPORTED
