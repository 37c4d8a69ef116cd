"""Seeded synthetic workloads for the routed MoE SwiGLU FFN forward.

This module holds shapes and random tensors only: it contains no routing,
FFN, dispatch or combine arithmetic. The CUDA path's callers and the
oracle's callers both draw their inputs here, so the two implementations
see identical tensors while sharing no code.

Shapes follow the configurations the pages describe:

* ``tiny_f32`` - the "MoE from scratch" tutorial's MoELayer demo: batch 4 x 32
  tokens of width 64, d_ff 128, 8 experts, top-2, one shared expert, router
  softmax over all experts then renormalised over the two selected, FP32.
* ``small``, ``medium_*``, ``large_*`` - APEX-1 Mathematical Reference Part 3,
  section 13.3 (Small 4/2/1, Medium 64/8/2, Large 256/8/2 experts/active/shared),
  with d and d_ff as fixed by the benchmark configurations; router
  r = x W_router + b, top-K of r, softmax over the K selected scores.
* ``latent`` - kimi_k3 "StableLatentMoE and QuantileBalancer": FP32 sigmoid
  router, top-(K+1) of s + bias, experts on a latent z = x W_down_latent.

Value recipe: x ~ N(0, 1); every weight matrix ~ N(0, 1/fan_in) (fan_in = the
contraction length it multiplies); balance bias ~ N(0, bias_std^2) plus a
per-expert skew offset -skew * ln(rank) with rank a random permutation of
1..E. Tensors are drawn in FP32 by torch's generator on the requested device
(a separate deterministic seed per tensor, and per expert for expert weights)
and rounded to nearest-even BF16 for the BF16 workloads.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass, replace

import torch

GATE_SOFTMAX_TOPK = "softmax_topk"
GATE_SOFTMAX_ALL_RENORM = "softmax_all_renorm"
GATE_SIGMOID = "sigmoid"


@dataclass(frozen=True)
class Workload:
    """Problem sizes and routing options of one MoE layer forward."""

    name: str
    T: int                 # tokens (batch x sequence, flattened)
    d: int                 # model width (M in the latent variant)
    d_ff: int              # routed expert hidden width (I in the latent variant)
    E: int                 # routed experts
    K: int                 # active routed experts per token
    n_shared: int          # always-on shared experts
    shared_d_ff: int       # hidden width of each shared expert
    dtype: str             # "f32" | "bf16": activations and expert weights
    gate: str              # GATE_* constant
    latent_dim: int = 0    # 0 = experts act on x; L = experts act on z = x W_down_latent
    bias_std: float = 0.0  # std of the balance bias draw (0 and skew 0 -> no bias)
    skew: float = 0.0      # per-expert logit offset -skew*ln(rank)
    renormalize: bool = False
    routed_scale: float = 1.0
    has_bias: bool = True

    @property
    def d_expert(self) -> int:
        """Input/output width of the routed experts (d, or L when latent)."""
        return self.latent_dim if self.latent_dim else self.d

    def resized(self, **kw) -> "Workload":
        return replace(self, **kw)

    def flops(self) -> float:
        """Algorithmic FLOPs of one forward (multiply-add = 2)."""
        T, d, E, K = self.T, self.d, self.E, self.K
        router = 2.0 * T * d * E
        shared = 6.0 * T * d * self.shared_d_ff * self.n_shared
        if self.latent_dim:
            L = self.latent_dim
            routed = 6.0 * T * L * self.d_ff * K + 2.0 * T * d * L * 2
        else:
            routed = 6.0 * T * d * self.d_ff * K
        return router + shared + routed


WORKLOADS: dict[str, Workload] = {
    "tiny_f32": Workload("tiny_f32", T=128, d=64, d_ff=128, E=8, K=2, n_shared=1,
                         shared_d_ff=128, dtype="f32", gate=GATE_SOFTMAX_ALL_RENORM,
                         has_bias=False),
    "small": Workload("small", T=4096, d=768, d_ff=2048, E=4, K=2, n_shared=1,
                      shared_d_ff=2048, dtype="bf16", gate=GATE_SOFTMAX_TOPK,
                      bias_std=0.01),
    "medium_prefill": Workload("medium_prefill", T=16384, d=2048, d_ff=1408, E=64, K=8,
                               n_shared=2, shared_d_ff=1408, dtype="bf16",
                               gate=GATE_SOFTMAX_TOPK, bias_std=0.01, skew=1.1),
    "medium_decode": Workload("medium_decode", T=64, d=2048, d_ff=1408, E=64, K=8,
                              n_shared=2, shared_d_ff=1408, dtype="bf16",
                              gate=GATE_SOFTMAX_TOPK, bias_std=0.01, skew=1.1),
    "large_prefill": Workload("large_prefill", T=8192, d=4096, d_ff=2048, E=256, K=8,
                              n_shared=2, shared_d_ff=2048, dtype="bf16",
                              gate=GATE_SOFTMAX_TOPK, bias_std=0.01),
    "large_prefill_zipf": Workload("large_prefill_zipf", T=8192, d=4096, d_ff=2048, E=256,
                                   K=8, n_shared=2, shared_d_ff=2048, dtype="bf16",
                                   gate=GATE_SOFTMAX_TOPK, bias_std=0.01, skew=1.2),
    "large_decode": Workload("large_decode", T=128, d=4096, d_ff=2048, E=256, K=8,
                             n_shared=2, shared_d_ff=2048, dtype="bf16",
                             gate=GATE_SOFTMAX_TOPK, bias_std=0.01),
    "large_decode_zipf": Workload("large_decode_zipf", T=128, d=4096, d_ff=2048, E=256,
                                  K=8, n_shared=2, shared_d_ff=2048, dtype="bf16",
                                  gate=GATE_SOFTMAX_TOPK, bias_std=0.01, skew=1.2),
    # one shared DenseFFN of width 2*1024, as the latent page builds it
    "latent": Workload("latent", T=8192, d=2048, d_ff=1024, E=128, K=8, n_shared=1,
                       shared_d_ff=2048, dtype="bf16", gate=GATE_SIGMOID, latent_dim=512),
}

# Reduced copies of the large layers for profiler captures that must stay at a
# few GB of device memory: the same widths and the same rows per expert
# (T*K/E = 256), an eighth of the experts and tokens.
PROFILE_CASES: dict[str, Workload] = {
    "large_prefill_e32": replace(WORKLOADS["large_prefill"], name="large_prefill_e32", T=1024,
                                 E=32),
    "large_decode_e32": replace(WORKLOADS["large_decode"], name="large_decode_e32", E=32),
    # the 128-token, 256-expert router of the large decode batch, with narrow experts
    "decode_e256_router": replace(WORKLOADS["large_decode"], name="decode_e256_router", d_ff=128,
                                  shared_d_ff=128),
}
WORKLOADS.update(PROFILE_CASES)

# The single-GPU throughput workload: the largest configuration, the
# APEX-large-like prefill batch (T=8192, d=4096, d_ff=2048, 256 experts, top-8,
# two shared experts).
BENCH_WORKLOAD = "large_prefill"

# Every configuration, in the order the bench reports them.
ALL_BENCH = ["tiny_f32", "small", "medium_prefill", "medium_decode", "large_prefill",
             "large_prefill_zipf", "large_decode", "large_decode_zipf", "latent"]


def _seed(base: int, *parts) -> int:
    h = hashlib.sha256(repr((int(base),) + tuple(parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, base, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(base, *parts))
    return g


def torch_dtype(w: Workload) -> torch.dtype:
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def _normal(shape, std, device, dtype, base, *parts) -> torch.Tensor:
    g = _gen(device, base, *parts)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _expert_stack(n, shape, std, device, dtype, base, name) -> torch.Tensor:
    out = torch.empty((n,) + tuple(shape), device=device, dtype=dtype)
    for e in range(n):
        out[e].copy_(_normal(shape, std, device, dtype, base, name, e))
    return out


def _stack_geometry(w: Workload, which: str):
    """(shape of one matrix, std, seed name) of an expert stack of make_inputs."""
    de = w.d_expert
    S, Fs = w.n_shared, w.shared_d_ff
    geo = {
        "W_gate": ((de, w.d_ff), 1.0 / math.sqrt(de)),
        "W_up": ((de, w.d_ff), 1.0 / math.sqrt(de)),
        "W_down": ((w.d_ff, de), 1.0 / math.sqrt(w.d_ff)),
        "Ws_gate": ((w.d, Fs), 1.0 / math.sqrt(w.d) if S else 1.0),
        "Ws_up": ((w.d, Fs), 1.0 / math.sqrt(w.d) if S else 1.0),
        "Ws_down": ((Fs, w.d), 1.0 / math.sqrt(Fs) if S else 1.0),
    }
    shape, std = geo[which]
    return shape, std, w.name + "/" + which


def expert_matrix(w: Workload, which: str, e: int, device="cpu", seed: int = 0) -> torch.Tensor:
    """Matrix e of the expert stack `which` (W_gate, W_up, W_down, Ws_*) alone:
    the same values as make_inputs(w, device, seed)[which][e]."""
    shape, std, name = _stack_geometry(w, which)
    return _normal(shape, std, device, torch_dtype(w), seed, name, e)


def make_bias(w: Workload, seed: int = 0) -> torch.Tensor | None:
    """Balance bias [E] FP32 on the CPU (None when the workload has none)."""
    if not w.has_bias:
        return None
    if w.gate == GATE_SIGMOID:
        # the quantile balancer's persistent buffer starts at zeros
        return torch.zeros(w.E, dtype=torch.float32)
    b = torch.zeros(w.E, dtype=torch.float32)
    if w.bias_std:
        b += _normal((w.E,), w.bias_std, "cpu", torch.float32, seed, w.name, "bias")
    if w.skew:
        g = _gen("cpu", seed, w.name, "rank")
        rank = torch.randperm(w.E, generator=g).to(torch.float64) + 1.0
        b += (-w.skew * torch.log(rank)).to(torch.float32)
    return b


def make_inputs(w: Workload, device="cpu", seed: int = 0, with_x: bool = True,
                routed_experts: bool = True) -> dict:
    """All tensors of one forward, row-major and contiguous.

    x [T, d]; W_router [d, E] FP32; bias [E] FP32 or None;
    W_gate, W_up [E, d_e, d_ff]; W_down [E, d_ff, d_e] (d_e = d, or L when latent);
    Ws_gate, Ws_up [S, d, Fs]; Ws_down [S, Fs, d];
    W_down_latent [d, L], W_up_latent [L, d] when latent.
    routed_experts=False leaves W_gate, W_up, W_down out (expert_matrix makes
    any one of them on its own).
    """
    dt = torch_dtype(w)
    de = w.d_expert
    t: dict = {}
    if with_x:
        t["x"] = _normal((w.T, w.d), 1.0, device, dt, seed, w.name, "x", w.T)
    t["W_router"] = _normal((w.d, w.E), 1.0 / math.sqrt(w.d), device, torch.float32,
                            seed, w.name, "W_router")
    b = make_bias(w, seed)
    t["bias"] = None if b is None else b.to(device)
    names = (("W_gate", "W_up", "W_down") if routed_experts else ())
    for which in names:
        shape, std, name = _stack_geometry(w, which)
        t[which] = _expert_stack(w.E, shape, std, device, dt, seed, name)
    S = w.n_shared
    if S:
        for which in ("Ws_gate", "Ws_up", "Ws_down"):
            shape, std, name = _stack_geometry(w, which)
            t[which] = _expert_stack(S, shape, std, device, dt, seed, name)
    else:
        t["Ws_gate"] = t["Ws_up"] = t["Ws_down"] = None
    if w.latent_dim:
        L = w.latent_dim
        t["W_down_latent"] = _normal((w.d, L), 1.0 / math.sqrt(w.d), device, dt, seed,
                                     w.name, "W_down_latent")
        t["W_up_latent"] = _normal((L, w.d), 1.0 / math.sqrt(L), device, dt, seed,
                                   w.name, "W_up_latent")
    else:
        t["W_down_latent"] = t["W_up_latent"] = None
    return t


def make_x(w: Workload, device="cpu", seed: int = 0) -> torch.Tensor:
    return _normal((w.T, w.d), 1.0, device, torch_dtype(w), seed, w.name, "x", w.T)


def random_routing(T: int, E: int, K: int, device="cpu", seed: int = 0,
                   skew: float = 0.0) -> tuple[torch.Tensor, torch.Tensor]:
    """Random top-K expert ids [T, K] (distinct per token) and weights [T, K] FP32.

    With skew > 0 experts are drawn with probability proportional to
    rank^-skew (rank a random permutation of 1..E), so some receive no token.
    """
    g = _gen("cpu", seed, "routing", T, E, K, skew)
    if skew:
        rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
        p = rank ** (-skew)
    else:
        p = torch.ones(E, dtype=torch.float64)
    idx = torch.multinomial(p.expand(T, E), K, replacement=False, generator=g)
    wts = torch.rand((T, K), generator=g, dtype=torch.float32)
    return idx.to(torch.int32).to(device), wts.to(device)
