"""The C-ABI library builds, loads without a GPU, exports every function
include/moe.h declares, and rejects invalid calls on the host before any
CUDA work (no compute call is made here)."""
import ctypes
import os
import subprocess

import pytest

from mixture_experts_ffn_fp32_gb300 import build as B

pytestmark = pytest.mark.skipif(not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="CUDA toolkit (nvcc) not available")


@pytest.fixture(scope="module")
def api():
    B.build()
    from mixture_experts_ffn_fp32_gb300 import api as A
    return A


def test_every_declared_symbol_is_exported(api):
    names = api.header_functions()
    assert len(names) >= 18, names
    for n in ["moe_route", "moe_dispatch", "moe_forward", "moe_quantile_bias_update"]:
        assert n in names
    L = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(L, n), f"{n} declared in moe.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    moe_syms = {s for s in exported if s.startswith("moe_")}
    assert moe_syms == set(names), (moe_syms ^ set(names))


def _spec(api, **kw):
    base = dict(T=64, d=64, d_ff=128, E=8, K=2, n_shared=1, shared_d_ff=128, dtype="bf16",
                gate="softmax_topk")
    base.update(kw)
    return api.LayerSpec(**base)


def test_workspace_size_and_validation(api):
    assert api.workspace_size(_spec(api)) > 0
    bigger = api.workspace_size(_spec(api, T=4096))
    assert bigger > api.workspace_size(_spec(api))
    bad = [dict(K=9), dict(K=0), dict(T=0), dict(gate="sigmoid", K=8), dict(d=60),
           dict(E=300, K=2), dict(K=17, E=64), dict(latent_dim=512, dtype="f32")]
    for kw in bad:
        with pytest.raises(api.MoeError) as ei:
            api.workspace_size(_spec(api, **kw))
        assert ei.value.status in (api.MOE_ERR_INVALID_ARG, api.MOE_ERR_UNSUPPORTED), kw


def test_saved_gate_up_workspace(api):
    """save_gate_up grows the workspace by the BF16 gate and up products of every
    routed row and shared expert (4 (T K d_ff + T S Fs) bytes, plus at most the
    four regions' 256-byte alignment) on a layer whose backward runs on the
    tensor cores, and nowhere else; a value other than 0 or 1 is rejected."""
    T, K, F, S, Fs = 64, 2, 128, 1, 128
    base = api.workspace_size(_spec(api))
    saved = api.workspace_size(_spec(api, save_gate_up=True))
    grow = 4 * (T * K * F + T * S * Fs)
    assert grow <= saved - base <= grow + 4 * 256
    for kw in (dict(dtype="f32"), dict(d_ff=96)):  # CUDA-core backward: nothing kept
        assert api.workspace_size(_spec(api, save_gate_up=True, **kw)) == api.workspace_size(_spec(api, **kw))
    cfg = _spec(api).config()
    cfg.save_gate_up = 2
    n = ctypes.c_size_t(0)
    assert api.lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == api.MOE_ERR_INVALID_ARG


def test_status_strings_and_metadata(api):
    L = api.lib()
    assert L.moe_version().decode().count(".") == 2
    for s in range(7):
        assert len(L.moe_status_string(s)) >= 2
    assert L.moe_stage_name(0) == b"router"
    assert L.moe_stage_name(99) is None
    assert api.launch_count() == 0
    assert L.moe_set_wait_timeout_ms(0) == api.MOE_ERR_INVALID_ARG
    assert L.moe_set_wait_timeout_ms(1000) == api.MOE_OK


def test_host_side_rejections_do_not_touch_the_gpu(api):
    L = api.lib()
    spec = _spec(api)
    cfg = spec.config()
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced on the host
    w = api.Weights()
    for f in api.Weights._fields_:
        setattr(w, f[0], 1 << 20)
    w.bias = None
    # null input
    assert L.moe_forward(ctypes.byref(cfg), None, ctypes.byref(w), fake, fake, 1 << 30, None) == \
        api.MOE_ERR_INVALID_ARG
    # workspace too small
    assert L.moe_forward(ctypes.byref(cfg), fake, ctypes.byref(w), fake, fake, 16, None) == \
        api.MOE_ERR_WORKSPACE
    # misaligned x
    assert L.moe_forward(ctypes.byref(cfg), ctypes.c_void_p((1 << 20) + 2), ctypes.byref(w), fake,
                         fake, 1 << 30, None) == api.MOE_ERR_INVALID_ARG
    # missing shared weights
    w2 = api.Weights()
    w2.W_router = w2.W_gate = w2.W_up = w2.W_down = 1 << 20
    assert L.moe_forward(ctypes.byref(cfg), fake, ctypes.byref(w2), fake, fake, 1 << 30, None) == \
        api.MOE_ERR_INVALID_ARG
    # invalid config through every entry point
    bad = _spec(api, K=9).config()
    assert L.moe_route(ctypes.byref(bad), fake, fake, None, fake, fake, None, None, None, None, 0,
                       None) == api.MOE_ERR_INVALID_ARG
    assert L.moe_route(ctypes.byref(cfg), fake, fake, None, fake, fake, None, None, None, fake, 8,
                       None) == api.MOE_ERR_WORKSPACE
    assert L.moe_dispatch(ctypes.byref(bad), fake, fake, fake, fake, fake, fake, fake, fake, 1 << 30,
                          None) == api.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake, fake, fake, 8,
                          None) == api.MOE_ERR_WORKSPACE
    assert L.moe_quantile_bias_update(8, 4, 4, fake, fake, fake, fake, 1 << 20, None) == \
        api.MOE_ERR_INVALID_ARG  # K + 1 > E
    assert L.moe_quantile_bias_update(8, 16, 2, fake, fake, fake, fake, 4, None) == \
        api.MOE_ERR_WORKSPACE
    assert L.moe_sign_bias_update(0, 8, 2, fake, fake, 0.1, None) == api.MOE_ERR_INVALID_ARG
    # routing diagnostics: workspace and output are required, sizes checked
    assert L.moe_routing_stats(ctypes.byref(cfg), fake, fake, None, None, fake, 1 << 30, None) == \
        api.MOE_ERR_INVALID_ARG
    assert L.moe_routing_stats(ctypes.byref(cfg), fake, fake, None, fake, None, 0, None) == \
        api.MOE_ERR_INVALID_ARG
    assert L.moe_routing_stats(ctypes.byref(cfg), fake, fake, None, fake, fake, 8, None) == \
        api.MOE_ERR_WORKSPACE
    assert L.moe_routing_stats(ctypes.byref(bad), fake, fake, None, fake, fake, 1 << 30, None) == \
        api.MOE_ERR_INVALID_ARG
    assert L.moe_timing_end(None, 0, None, None) == api.MOE_ERR_INVALID_ARG
    # backward: dout and dx required, gradients only for parts the layer has,
    # both workspaces checked
    g = api.Grads()
    g.dx = 1 << 20
    big = 1 << 40
    assert L.moe_backward(ctypes.byref(cfg), fake, ctypes.byref(w), None, ctypes.byref(g), fake,
                          big, fake, big, None) == api.MOE_ERR_INVALID_ARG
    g0 = api.Grads()
    assert L.moe_backward(ctypes.byref(cfg), fake, ctypes.byref(w), fake, ctypes.byref(g0), fake,
                          big, fake, big, None) == api.MOE_ERR_INVALID_ARG
    gl = api.Grads()
    gl.dx = gl.dW_up_latent = 1 << 20
    assert L.moe_backward(ctypes.byref(cfg), fake, ctypes.byref(w), fake, ctypes.byref(gl), fake,
                          big, fake, big, None) == api.MOE_ERR_INVALID_ARG
    assert L.moe_backward(ctypes.byref(cfg), fake, ctypes.byref(w), fake, ctypes.byref(g), fake,
                          big, fake, 16, None) == api.MOE_ERR_WORKSPACE
    assert L.moe_backward(ctypes.byref(cfg), fake, ctypes.byref(w), ctypes.c_void_p((1 << 20) + 4),
                          ctypes.byref(g), fake, big, fake, big, None) == api.MOE_ERR_INVALID_ARG
    assert L.moe_backward(ctypes.byref(bad), fake, ctypes.byref(w), fake, ctypes.byref(g), fake,
                          big, fake, big, None) == api.MOE_ERR_INVALID_ARG
    n = ctypes.c_size_t(0)
    assert L.moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == api.MOE_OK
    assert n.value > 0
    assert api.launch_count() == 0


def test_workspace_views_are_disjoint_and_inside(api):
    for kw in (dict(), dict(gate="sigmoid", K=2, E=8), dict(dtype="f32", gate="softmax_all_renorm")):
        spec = _spec(api, **kw)
        total = api.workspace_size(spec)
        v = api.Views()
        base = 1 << 24
        assert api.lib().moe_get_workspace_views(ctypes.byref(spec.config()), ctypes.c_void_p(base),
                                                 ctypes.byref(v)) == api.MOE_OK
        T, K, E = spec.T, spec.K, spec.E
        sizes = {"topk_idx": T * K * 4, "topk_w": T * K * 4, "margin": T * 4,
                 "top_scores": T * (K + 1) * 4, "scores": T * E * 4, "counts": E * 4,
                 "offsets": (E + 1) * 4, "sorted_token": T * K * 4, "sorted_w": T * K * 4,
                 "inv": T * K * 4}
        spans = []
        for name, n in sizes.items():
            p = getattr(v, name)
            if p is None:
                assert spec.gate != "sigmoid" and name in ("top_scores", "scores")
                continue
            assert p % 256 == 0 and base <= p and p + n <= base + total, name
            spans.append((p, p + n))
        spans.sort()
        assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
