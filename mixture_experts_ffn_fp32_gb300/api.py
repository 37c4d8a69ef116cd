"""Thin Python binding of libmoe (include/moe.h).

Argument marshalling only: torch CUDA tensors are checked for device, dtype
and contiguity and passed as plain pointers together with the current CUDA
stream. Every step of the layer runs in the library's kernels; there is no
fallback path. The library is loaded on first use and must exist (build it
with ``mixture_experts_ffn_fp32_gb300.build.build()``).
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass

import torch

from . import build as _build

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, \
    MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_INDEX = range(7)
MOE_F32, MOE_BF16 = 0, 1
GATES = {"softmax_topk": 0, "softmax_all_renorm": 1, "sigmoid": 2}

HEADER = os.path.join(_build.ROOT, "include", "moe.h")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class Config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("E", ctypes.c_int32), ("K", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("shared_d_ff", ctypes.c_int32), ("latent_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("gate", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("routed_scale", ctypes.c_float),
                ("out_dtype", ctypes.c_int32), ("save_gate_up", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("W_router", "bias", "W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down",
                 "W_down_latent", "W_up_latent")]


GRAD_NAMES = ("dx", "dW_router", "dW_gate", "dW_up", "dW_down", "dWs_gate", "dWs_up",
              "dWs_down", "dW_down_latent", "dW_up_latent")


class Grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in GRAD_NAMES]


class Views(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("topk_idx", "topk_w", "margin", "top_scores", "scores", "counts", "offsets",
                 "sorted_token", "sorted_w", "inv")]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmoe. Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"libmoe.so is not built ({path}); run "
                               "mixture_experts_ffn_fp32_gb300.build.build() first")
        L = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        cfgp = ctypes.POINTER(Config)
        sigs = {
            "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "moe_version": (ctypes.c_char_p, []),
            "moe_workspace_size": (ctypes.c_int, [cfgp, ctypes.POINTER(sz)]),
            "moe_get_workspace_views": (ctypes.c_int, [cfgp, vp, ctypes.POINTER(Views)]),
            "moe_route": (ctypes.c_int, [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "moe_dispatch": (ctypes.c_int, [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "moe_dispatch_noalloc": (ctypes.c_int, [cfgp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "moe_forward": (ctypes.c_int, [cfgp, vp, ctypes.POINTER(Weights), vp, vp, sz, vp]),
            "moe_forward_host": (ctypes.c_int, [cfgp, vp, ctypes.POINTER(Weights), vp, vp, sz, vp]),
            "moe_quantile_bias_update": (ctypes.c_int, [i32, i32, i32, vp, vp, vp, vp, sz, vp]),
            "moe_quantile_workspace_size": (sz, [i32, i32]),
            "moe_sign_bias_update": (ctypes.c_int, [i32, i32, i32, vp, vp, ctypes.c_float, vp]),
            "moe_routing_stats": (ctypes.c_int, [cfgp, vp, vp, vp, vp, vp, sz, vp]),
            "moe_workspace_status": (ctypes.c_int, [vp, vp]),
            "moe_backward_workspace_size": (ctypes.c_int, [cfgp, ctypes.POINTER(sz)]),
            "moe_backward": (ctypes.c_int, [cfgp, vp, ctypes.POINTER(Weights), vp,
                                            ctypes.POINTER(Grads), vp, sz, vp, sz, vp]),
            "moe_timing_begin": (ctypes.c_int, [i32, ctypes.c_uint32]),
            "moe_timing_end": (ctypes.c_int, [ctypes.POINTER(ctypes.c_float), i32,
                                              ctypes.POINTER(i32), ctypes.POINTER(i32)]),
            "moe_stage_name": (ctypes.c_char_p, [i32]),
            "moe_launch_count": (ctypes.c_uint64, []),
            "moe_set_wait_timeout_ms": (ctypes.c_int, [i32]),
            "moe_selftest_wait_timeout": (ctypes.c_int, [i32, vp, vp]),
        }
        for name, (res, args) in sigs.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/moe.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(moe_[a-z0-9_]+)\s*\(",
                                 src, flags=re.M)))


def status_string(s: int) -> str:
    return lib().moe_status_string(int(s)).decode()


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


@dataclass(frozen=True)
class LayerSpec:
    T: int
    d: int
    d_ff: int
    E: int
    K: int
    n_shared: int = 0
    shared_d_ff: int = 0
    latent_dim: int = 0
    dtype: str = "bf16"
    gate: str = "softmax_topk"
    renormalize: bool = False
    routed_scale: float = 1.0
    out_dtype: str = "f32"
    save_gate_up: bool = False  # forward keeps the gate/up products for the backward

    @staticmethod
    def of(w, out_dtype: str = "f32", save_gate_up: bool = False) -> "LayerSpec":
        """From any object with the Workload attribute names."""
        return LayerSpec(w.T, w.d, w.d_ff, w.E, w.K, w.n_shared, w.shared_d_ff, w.latent_dim,
                         w.dtype, w.gate, bool(w.renormalize), float(w.routed_scale), out_dtype,
                         bool(save_gate_up))

    def config(self) -> Config:
        return Config(self.T, self.d, self.d_ff, self.E, self.K, self.n_shared,
                      self.shared_d_ff if self.n_shared else 0, self.latent_dim,
                      MOE_F32 if self.dtype == "f32" else MOE_BF16, GATES[self.gate],
                      int(self.renormalize), float(self.routed_scale),
                      MOE_F32 if self.out_dtype == "f32" else MOE_BF16, int(self.save_gate_up))

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def torch_out_dtype(self):
        return torch.float32 if self.out_dtype == "f32" else torch.bfloat16


def workspace_size(spec: LayerSpec) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(spec.config()), ctypes.byref(n)),
           "moe_workspace_size")
    return n.value


def alloc_workspace(spec: LayerSpec, device="cuda") -> torch.Tensor:
    return torch.empty(workspace_size(spec), dtype=torch.uint8, device=device)


def _dev(t, dtype, name, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def weights_struct(spec: LayerSpec, p: dict) -> Weights:
    dt = spec.torch_dtype
    de = spec.latent_dim or spec.d
    S, Fs = spec.n_shared, spec.shared_d_ff
    w = Weights()
    w.W_router = _dev(p["W_router"], torch.float32, "W_router", (spec.d, spec.E)).data_ptr()
    b = p.get("bias")
    w.bias = None if b is None else _dev(b, torch.float32, "bias", (spec.E,)).data_ptr()
    w.W_gate = _dev(p["W_gate"], dt, "W_gate", (spec.E, de, spec.d_ff)).data_ptr()
    w.W_up = _dev(p["W_up"], dt, "W_up", (spec.E, de, spec.d_ff)).data_ptr()
    w.W_down = _dev(p["W_down"], dt, "W_down", (spec.E, spec.d_ff, de)).data_ptr()
    if S:
        w.Ws_gate = _dev(p["Ws_gate"], dt, "Ws_gate", (S, spec.d, Fs)).data_ptr()
        w.Ws_up = _dev(p["Ws_up"], dt, "Ws_up", (S, spec.d, Fs)).data_ptr()
        w.Ws_down = _dev(p["Ws_down"], dt, "Ws_down", (S, Fs, spec.d)).data_ptr()
    if spec.latent_dim:
        w.W_down_latent = _dev(p["W_down_latent"], dt, "W_down_latent",
                               (spec.d, spec.latent_dim)).data_ptr()
        w.W_up_latent = _dev(p["W_up_latent"], dt, "W_up_latent",
                             (spec.latent_dim, spec.d)).data_ptr()
    return w


def route(spec: LayerSpec, x: torch.Tensor, W_router: torch.Tensor, bias=None, stream=None,
          ws: torch.Tensor | None = None):
    """moe_route: returns dict idx [T,K] int32, w [T,K], margin [T] (+ top_scores
    [T,K+1] and scores [T,E] in sigmoid mode). With a workspace the tensor-core
    router is used where the layer allows it (as in forward)."""
    dev = x.device
    _dev(x, spec.torch_dtype, "x", (spec.T, spec.d))
    _dev(W_router, torch.float32, "W_router", (spec.d, spec.E))
    if bias is not None:
        _dev(bias, torch.float32, "bias", (spec.E,))
    out = {
        "idx": torch.empty((spec.T, spec.K), dtype=torch.int32, device=dev),
        "w": torch.empty((spec.T, spec.K), dtype=torch.float32, device=dev),
        "margin": torch.empty((spec.T,), dtype=torch.float32, device=dev),
    }
    sig = spec.gate == "sigmoid"
    if sig:
        out["top_scores"] = torch.empty((spec.T, spec.K + 1), dtype=torch.float32, device=dev)
        out["scores"] = torch.empty((spec.T, spec.E), dtype=torch.float32, device=dev)
    _check(lib().moe_route(ctypes.byref(spec.config()), x.data_ptr(), W_router.data_ptr(),
                           _ptr(bias), out["idx"].data_ptr(), out["w"].data_ptr(),
                           out["margin"].data_ptr(), _ptr(out.get("top_scores")),
                           _ptr(out.get("scores")), _ptr(ws), 0 if ws is None else ws.numel(),
                           _stream(stream)), "moe_route")
    return out


def dispatch(spec: LayerSpec, idx: torch.Tensor, w: torch.Tensor, ws: torch.Tensor | None = None,
             stream=None):
    """moe_dispatch: returns dict counts, offsets, sorted_token, sorted_w, inv."""
    dev = idx.device
    _dev(idx, torch.int32, "topk_idx", (spec.T, spec.K))
    _dev(w, torch.float32, "topk_w", (spec.T, spec.K))
    ws = alloc_workspace(spec, dev) if ws is None else ws
    TK = spec.T * spec.K
    out = {
        "counts": torch.empty((spec.E,), dtype=torch.int32, device=dev),
        "offsets": torch.empty((spec.E + 1,), dtype=torch.int32, device=dev),
        "sorted_token": torch.empty((TK,), dtype=torch.int32, device=dev),
        "sorted_w": torch.empty((TK,), dtype=torch.float32, device=dev),
        "inv": torch.empty((spec.T, spec.K), dtype=torch.int32, device=dev),
    }
    _check(lib().moe_dispatch(ctypes.byref(spec.config()), idx.data_ptr(), w.data_ptr(),
                              out["counts"].data_ptr(), out["offsets"].data_ptr(),
                              out["sorted_token"].data_ptr(), out["sorted_w"].data_ptr(),
                              out["inv"].data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)),
           "moe_dispatch")
    out["ws"] = ws
    return out


def dispatch_noalloc(spec: LayerSpec, idx: torch.Tensor, w: torch.Tensor, out: dict | None = None,
                     stream=None):
    """moe_dispatch_noalloc: moe_dispatch without a workspace, for callers that
    cannot allocate device memory (the library keeps the scratch in a fixed
    device array; T*K <= 65536, E <= 256). ``out`` may hold preallocated
    counts, offsets, sorted_token, sorted_w and inv tensors."""
    dev = idx.device
    _dev(idx, torch.int32, "topk_idx", (spec.T, spec.K))
    _dev(w, torch.float32, "topk_w", (spec.T, spec.K))
    TK = spec.T * spec.K
    if out is None:
        out = {
            "counts": torch.empty((spec.E,), dtype=torch.int32, device=dev),
            "offsets": torch.empty((spec.E + 1,), dtype=torch.int32, device=dev),
            "sorted_token": torch.empty((TK,), dtype=torch.int32, device=dev),
            "sorted_w": torch.empty((TK,), dtype=torch.float32, device=dev),
            "inv": torch.empty((spec.T, spec.K), dtype=torch.int32, device=dev),
        }
    _check(lib().moe_dispatch_noalloc(ctypes.byref(spec.config()), idx.data_ptr(), w.data_ptr(),
                                      out["counts"].data_ptr(), out["offsets"].data_ptr(),
                                      out["sorted_token"].data_ptr(), out["sorted_w"].data_ptr(),
                                      out["inv"].data_ptr(), _stream(stream)),
           "moe_dispatch_noalloc")
    return out


def forward(spec: LayerSpec, x: torch.Tensor, params: dict, out: torch.Tensor | None = None,
            ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """moe_forward: the whole layer on device tensors."""
    _dev(x, spec.torch_dtype, "x", (spec.T, spec.d))
    ws = alloc_workspace(spec, x.device) if ws is None else ws
    if out is None:
        out = torch.empty((spec.T, spec.d), dtype=spec.torch_out_dtype, device=x.device)
    _dev(out, spec.torch_out_dtype, "out", (spec.T, spec.d))
    w = weights_struct(spec, params)
    _check(lib().moe_forward(ctypes.byref(spec.config()), x.data_ptr(), ctypes.byref(w),
                             out.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)),
           "moe_forward")
    return out


def backward_workspace_size(spec: LayerSpec) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_backward_workspace_size(ctypes.byref(spec.config()), ctypes.byref(n)),
           "moe_backward_workspace_size")
    return int(n.value)


def grad_shapes(spec: LayerSpec) -> dict:
    de = spec.latent_dim or spec.d
    S, Fs, L = spec.n_shared, spec.shared_d_ff, spec.latent_dim
    sh = {"dx": (spec.T, spec.d), "dW_router": (spec.d, spec.E),
          "dW_gate": (spec.E, de, spec.d_ff), "dW_up": (spec.E, de, spec.d_ff),
          "dW_down": (spec.E, spec.d_ff, de)}
    if S:
        sh.update(dWs_gate=(S, spec.d, Fs), dWs_up=(S, spec.d, Fs), dWs_down=(S, Fs, spec.d))
    if L:
        sh.update(dW_down_latent=(spec.d, L), dW_up_latent=(L, spec.d))
    return sh


def backward(spec: LayerSpec, x: torch.Tensor, params: dict, dout: torch.Tensor, ws: torch.Tensor,
             grads: dict | None = None, bws: torch.Tensor | None = None, stream=None) -> dict:
    """moe_backward after a moe_forward on ws: FP32 gradients of sum(dout * out).
    ``grads`` maps names of GRAD_NAMES to preallocated FP32 tensors (absent
    names are allocated, zero-filled: an expert slice that gets no gradient
    stays as given); a name mapped to None is not computed."""
    _dev(x, spec.torch_dtype, "x", (spec.T, spec.d))
    _dev(dout, torch.float32, "dout", (spec.T, spec.d))
    shapes = grad_shapes(spec)
    out = {}
    given = grads or {}
    for n, shp in shapes.items():
        if n in given:
            if given[n] is not None:
                out[n] = _dev(given[n], torch.float32, n, shp)
        else:
            out[n] = torch.zeros(shp, dtype=torch.float32, device=x.device)
    if "dx" not in out:
        raise ValueError("dx is required")
    g = Grads()
    for n in GRAD_NAMES:
        setattr(g, n, out[n].data_ptr() if n in out else None)
    if bws is None:
        bws = torch.empty(backward_workspace_size(spec), dtype=torch.uint8, device=x.device)
    w = weights_struct(spec, params)
    _check(lib().moe_backward(ctypes.byref(spec.config()), x.data_ptr(), ctypes.byref(w),
                              dout.data_ptr(), ctypes.byref(g), ws.data_ptr(), ws.numel(),
                              bws.data_ptr(), bws.numel(), _stream(stream)),
           "moe_backward")
    return out


def forward_host(spec: LayerSpec, x_host: torch.Tensor, params: dict, out_host: torch.Tensor,
                 ws: torch.Tensor, stream=None) -> torch.Tensor:
    """moe_forward_host: host x / out (pinned for asynchronous DMA); synchronises."""
    for n, t, dt in (("x_host", x_host, spec.torch_dtype), ("out_host", out_host, spec.torch_out_dtype)):
        if t.is_cuda or not t.is_contiguous() or t.dtype != dt or t.numel() != spec.T * spec.d:
            raise ValueError(f"{n} must be a contiguous host tensor of {dt} with T*d elements")
    w = weights_struct(spec, params)
    _check(lib().moe_forward_host(ctypes.byref(spec.config()), x_host.data_ptr(), ctypes.byref(w),
                                  out_host.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)),
           "moe_forward_host")
    return out_host


def workspace_views(spec: LayerSpec, ws: torch.Tensor) -> dict:
    """Torch views of the routing/dispatch results a forward left in ws."""
    v = Views()
    _check(lib().moe_get_workspace_views(ctypes.byref(spec.config()), ws.data_ptr(), ctypes.byref(v)),
           "moe_get_workspace_views")
    base = ws.data_ptr()
    T, K, E = spec.T, spec.K, spec.E

    def view(ptr, n, dtype, shape):
        if ptr is None:
            return None
        off = ptr - base
        esz = torch.tensor([], dtype=dtype).element_size()
        return ws[off: off + n * esz].view(dtype).view(*shape)

    i32, f32 = torch.int32, torch.float32
    return {
        "idx": view(v.topk_idx, T * K, i32, (T, K)),
        "w": view(v.topk_w, T * K, f32, (T, K)),
        "margin": view(v.margin, T, f32, (T,)),
        "top_scores": view(v.top_scores, T * (K + 1), f32, (T, K + 1)),
        "scores": view(v.scores, T * E, f32, (T, E)),
        "counts": view(v.counts, E, i32, (E,)),
        "offsets": view(v.offsets, E + 1, i32, (E + 1,)),
        "sorted_token": view(v.sorted_token, T * K, i32, (T * K,)),
        "sorted_w": view(v.sorted_w, T * K, f32, (T * K,)),
        "inv": view(v.inv, T * K, i32, (T, K)),
    }


def quantile_bias_update(top_scores: torch.Tensor, scores: torch.Tensor, K: int, bias: torch.Tensor,
                         ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """moe_quantile_bias_update: replaces bias [E] in place and returns it."""
    T, E = scores.shape
    _dev(top_scores, torch.float32, "top_scores", (T, K + 1))
    _dev(scores, torch.float32, "scores", (T, E))
    _dev(bias, torch.float32, "bias", (E,))
    n = lib().moe_quantile_workspace_size(T, E)
    ws = torch.empty(n, dtype=torch.uint8, device=scores.device) if ws is None else ws
    _check(lib().moe_quantile_bias_update(T, E, K, top_scores.data_ptr(), scores.data_ptr(),
                                          bias.data_ptr(), ws.data_ptr(), ws.numel(),
                                          _stream(stream)), "moe_quantile_bias_update")
    return bias


def routing_stats(spec: LayerSpec, x: torch.Tensor, W_router: torch.Tensor, bias=None,
                  ws: torch.Tensor | None = None, stream=None, read: bool = True) -> dict:
    """Switch load-balancing loss (before alpha), router z-loss (before its
    weight) and mean router probabilities of one batch (moe_routing_stats).
    Returns dict(out [2+E] device tensor, ws) and, with read=True (waits for
    the stream), aux, z and P [E] on the host."""
    ws = alloc_workspace(spec, x.device) if ws is None else ws
    out = torch.empty(2 + spec.E, dtype=torch.float32, device=x.device)
    _check(lib().moe_routing_stats(ctypes.byref(spec.config()), _ptr(x), _ptr(W_router),
                                   _ptr(bias), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_routing_stats")
    res = {"out": out, "ws": ws}
    if read:
        (stream if stream is not None else torch.cuda.current_stream()).synchronize()
        vals = out.cpu()
        res.update(aux=float(vals[0]), z=float(vals[1]), P=vals[2:])
    return res


def sign_bias_update(counts: torch.Tensor, N: int, K: int, bias: torch.Tensor, alpha: float,
                     stream=None) -> torch.Tensor:
    E = counts.shape[0]
    _dev(counts, torch.int32, "counts", (E,))
    _dev(bias, torch.float32, "bias", (E,))
    _check(lib().moe_sign_bias_update(E, N, K, counts.data_ptr(), bias.data_ptr(), float(alpha),
                                      _stream(stream)), "moe_sign_bias_update")
    return bias


def workspace_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronises and returns (and clears) the workspace's device error status."""
    return lib().moe_workspace_status(ws.data_ptr(), _stream(stream))


def launch_count() -> int:
    return int(lib().moe_launch_count())


def set_wait_timeout_ms(ms: int):
    _check(lib().moe_set_wait_timeout_ms(int(ms)), "moe_set_wait_timeout_ms")


def selftest_wait_timeout(ms: int, ws: torch.Tensor, stream=None) -> int:
    return lib().moe_selftest_wait_timeout(int(ms), ws.data_ptr(), _stream(stream))


STAGES = ["router", "latent_down", "dispatch", "gather", "gate_up", "down", "combine", "latent_up",
          "decode_fused", "route_dispatch_gather"]


class StageTimer:
    """Per-stage CUDA-event timing of moe_forward calls (library-owned events).
    stages: names to time (None = all)."""

    def __init__(self, max_calls: int, stages=None):
        mask = 0xFFFFFFFF if stages is None else sum(1 << STAGES.index(n) for n in stages)
        _check(lib().moe_timing_begin(int(max_calls), mask), "moe_timing_begin")

    def finish(self) -> tuple[dict, int]:
        arr = (ctypes.c_float * 32)()
        ns, nc = ctypes.c_int32(0), ctypes.c_int32(0)
        _check(lib().moe_timing_end(arr, 32, ctypes.byref(ns), ctypes.byref(nc)), "moe_timing_end")
        names = [lib().moe_stage_name(i).decode() for i in range(ns.value)]
        return {n: arr[i] for i, n in enumerate(names)}, nc.value
