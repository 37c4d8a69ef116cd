"""Throughput of the routed MoE SwiGLU FFN layer forward on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--no-cpu-baseline] [--no-workloads]

One step = one whole layer forward (router, dispatch, grouped gate/up,
grouped down, shared experts, combine) over one batch of T synthetic tokens
with inputs resident in HBM. The headline workload is the largest
configuration, the APEX-large-like prefill batch (T=8192, d=4096, d_ff=2048,
256 experts, top-8, two shared experts). Each timed step is bracketed by CUDA
events on the launching stream; L2 is flushed (a 256 MB write, larger than the
129 MB L2) between timed steps, outside the events. The JSON line reports
whole-job tokens/s (all ranks), the layer's TFLOP/s and roofline fraction, the
dominant kernel's roofline fraction (measured by the library's own stage
events), the end-to-end number through moe_forward_host (host buffers, copies
inside the timed region), SM clocks sampled during the timed region, the CPU
oracle on a bounded sample of the same workload, and a `workloads` block that
times every configuration the same way (its tokens/s, TFLOP/s, roofline
fraction, per-stage times and the router's near-tie count). With N > 1
(torchrun) every rank runs an independent replica of the layer on its own GPU
(the layer has no exchange step on one GPU); the step time is the max over
ranks.

--impl reference times the CPU oracle (float64 NumPy, per-token loop) on the
host cores, on a bounded sample of tokens of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s and TFLOP/s (fraction of tensor/HBM roofline) on 1 GB300"
L2_FLUSH_BYTES = 256 << 20
L2_NOTE = ("flushed between timed steps, outside the events: a 256 MB write, then a read of "
           "the same buffer so that L2 holds clean lines")
NEAR_TIE = 1e-5


def l2_flush(flush, i):
    """Evict the layer's data from L2: write a buffer larger than L2, then read
    it back, so that the next step does not pay for writing back the flush's
    dirty lines."""
    import torch
    flush.fill_(i & 0xFF)
    flush.view(torch.int64).sum()


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=None)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-backward", action="store_true", help="skip the timed backward pass")
    p.add_argument("--no-diag", action="store_true", help="skip the routing diagnostics pass")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the per-configuration block")
    p.add_argument("--workload-steps", type=int, default=10)
    p.add_argument("--out-dtype", choices=["f32", "bf16"], default="f32")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, device="cpu") -> float:
    """Slowest rank's value (replicas run independently; the job takes as long
    as its slowest rank). Identity without an initialised process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, step_ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's step."""
    return world * tokens_per_rank / (step_ms / 1e3)


# FP32 FFMA peak of the CUDA cores: 152 SMs x 128 FP32 lanes x 2 FLOP x the
# maximum SM clock (2070 MHz, or MEASURED_PEAKS.json's sm_max_mhz).
def fp32_alu_tflops(sm_mhz: float = 2070.0) -> float:
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured",
                "fp32_tflops": fp32_alu_tflops(d.get("sm_max_mhz", 2070.0))}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback", "fp32_tflops": fp32_alu_tflops()}


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------

def gate_up_flops(w) -> float:
    """FLOPs of the grouped gate/up launch: the routed rows against the gate
    and up matrices of their experts, plus every token against the shared
    experts' (the shared experts run in the same launch in every BF16 layer,
    the latent one included)."""
    de = w.latent_dim or w.d
    f = 4.0 * w.T * w.K * de * w.d_ff
    f += 4.0 * w.T * w.d * w.shared_d_ff * w.n_shared
    return f


def gate_up_bytes(w, counts=None) -> float:
    """Algorithmic HBM bytes of the grouped gate/up launch: gate and up weights
    of the experts that get tokens and of the shared experts, the operand rows
    read once (routed rows and the token rows of the shared experts), the
    hidden rows written once."""
    es = 4 if w.dtype == "f32" else 2
    de = w.latent_dim or w.d
    used = w.E if counts is None else int(sum(1 for c in counts if c > 0))
    b = used * 2 * de * w.d_ff * es + w.T * w.K * de * es + w.T * w.K * w.d_ff * es
    b += w.n_shared * 2 * w.d * w.shared_d_ff * es
    if w.n_shared:
        b += w.T * w.d * es + w.T * w.n_shared * w.shared_d_ff * es
    return float(b)


def backward_flops(w) -> float:
    """Algorithmic FLOPs of the backward: twice the forward's expert GEMMs
    (input and weight gradients), the router's two, the latent projections'
    four; the recomputation of the gate/up products is not counted."""
    de = w.latent_dim or w.d
    f = 12.0 * w.T * w.K * de * w.d_ff
    f += 12.0 * w.T * w.d * w.shared_d_ff * w.n_shared
    f += 4.0 * w.T * w.d * w.E
    if w.latent_dim:
        f += 8.0 * w.T * w.d * w.latent_dim
    return f


def backward_bytes(w, counts=None) -> float:
    """Algorithmic HBM bytes of the backward: x, the upstream gradient (FP32)
    and the weights of the experts that got tokens (+ shared, router, latent
    projections) read once; dx and every weight gradient written once in FP32
    (the gradients of experts without tokens are not written)."""
    es = 4 if w.dtype == "f32" else 2
    de = w.latent_dim or w.d
    used = w.E if counts is None else int(sum(1 for c in counts if c > 0))
    wts = used * 3 * de * w.d_ff + w.n_shared * 3 * w.d * w.shared_d_ff
    lat = 2 * w.d * w.latent_dim if w.latent_dim else 0
    b = (wts + lat) * (es + 4)          # weights read, their gradients written
    b += w.d * w.E * (4 + 4)            # router weights read, gradient written
    b += w.T * w.d * (es + 4 + 4)       # x and the upstream gradient read, dx written
    return float(b)


def layer_bytes(w, counts=None) -> float:
    """Algorithmic HBM bytes of one forward: weights of the experts that get
    tokens + shared + router weights + x read + out written (FP32 out)."""
    es = 4 if w.dtype == "f32" else 2
    de = w.latent_dim or w.d
    used = w.E if counts is None else int(sum(1 for c in counts if c > 0))
    b = used * 3 * de * w.d_ff * es
    b += w.n_shared * 3 * w.d * w.shared_d_ff * es
    b += w.d * w.E * 4
    if w.latent_dim:
        b += 2 * w.d * w.latent_dim * es
    b += w.T * w.d * es + w.T * w.d * 4
    return float(b)


def layer_roofline(w, ms, counts, pk) -> dict:
    """max(FLOP / tensor peak, bytes / HBM peak) over the measured step time."""
    f32 = w.dtype == "f32"
    fpk = pk["fp32_tflops"] if f32 else pk["bf16_tflops"]
    t_flop = w.flops() / (fpk * 1e12)
    t_hbm = layer_bytes(w, counts) / (pk["hbm_gbs"] * 1e9)
    bound = ("alu" if f32 else "tensor") if t_flop >= t_hbm else "hbm"
    r = {"t_flop_ms": t_flop * 1e3, "t_hbm_ms": t_hbm * 1e3, "bound": bound,
         "frac": max(t_flop, t_hbm) * 1e3 / ms, "peak_source": pk["source"],
         "flop_peak": "FP32 FFMA" if f32 else "BF16 burst"}
    sus = pk.get("bf16_tflops_sustained")
    if not f32 and sus:
        # against the BF16 rate sustained for seconds under the power cap
        r["frac_of_sustained"] = max(w.flops() / (sus * 1e12), t_hbm) * 1e3 / ms
    return r


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "common.cuh", "warp_stage.cuh"):
        with open(os.path.join(ROOT, "mixture_experts_ffn_fp32_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the gate/up kernel from the committed ncu
    summary (profiles/gate_up_traffic.txt), if it was taken on the current
    kernel source; else None. Returns (bytes, note)."""
    path = os.path.join(ROOT, "profiles", "gate_up_traffic.txt")
    if not os.path.exists(path):
        return None, None
    src = kernel_source_hash()
    with open(path) as f:
        for ln in f:
            if ln.startswith("#") or "=" not in ln:
                continue
            kv = dict(p.split("=", 1) for p in ln.split())
            if kv.get("workload") == workload and kv.get("kernel_source") == src:
                return int(kv["dram_bytes_per_launch"]), kv.get("note")
    return None, None


# ---------------------------------------------------------------------------
# clocks sampler
# ---------------------------------------------------------------------------

class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.idx)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline leg and the reference arm)
#
# Worker processes are spawned (never forked after CUDA is up) and run
# single-threaded. Each makes the workload's inputs on the CPU once, except the
# routed experts' matrices, which it makes one at a time when the oracle first
# reads them (the large layers hold 13 GB of expert weights; a token reads
# K of them): making them is not counted in the oracle's time.
# ---------------------------------------------------------------------------

_WORKER_STATE = {}


class _LazyExperts:
    """An expert stack that makes matrix e on first use (the same values the
    workload generator gives), keeping the last `keep` of them; time spent
    making matrices accumulates in clock[0]."""

    def __init__(self, w, which, seed, keep, clock):
        from mixture_experts_ffn_fp32_gb300 import workloads as W
        self.W, self.w, self.which, self.seed = W, w, which, seed
        self.keep, self.clock = keep, clock
        self.cache = {}
        one = (w.d_ff, w.d_expert) if which == "W_down" else (w.d_expert, w.d_ff)
        self.shape = (w.E,) + one

    def __getitem__(self, e):
        e = int(e)
        if e in self.cache:
            v = self.cache.pop(e)
            self.cache[e] = v
            return v
        t0 = time.perf_counter()
        v = self.W.expert_matrix(self.w, self.which, e, "cpu", self.seed)
        self.clock[0] += time.perf_counter() - t0
        self.cache[e] = v
        while len(self.cache) > self.keep:
            self.cache.pop(next(iter(self.cache)))
        return v


def _oracle_worker(args):
    """Oracle forward of the listed tokens; returns (oracle seconds, tokens)."""
    name, tokens, seed = args
    from mixture_experts_ffn_fp32_gb300 import workloads as W
    from oracle import moe_oracle as O
    w = W.WORKLOADS[name]
    st = _WORKER_STATE.get((name, seed))
    if st is None:
        _WORKER_STATE.clear()
        clock = [0.0]
        inp = W.make_inputs(w, device="cpu", seed=seed, routed_experts=False)
        for which in ("W_gate", "W_up", "W_down"):
            inp[which] = _LazyExperts(w, which, seed, 2 * w.K, clock)
        st = (w, inp, clock)
        _WORKER_STATE[(name, seed)] = st
    w, inp, clock = st
    g0 = clock[0]
    t0 = time.perf_counter()
    O.moe_forward(inp["x"], inp, w.gate, w.K, w.renormalize, w.routed_scale, tokens=tokens)
    return time.perf_counter() - t0 - (clock[0] - g0), len(tokens)


def _mem_available_gb() -> float:
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    return int(ln.split()[1]) / 1e6
    except OSError:
        pass
    return 16.0


def oracle_workers(name: str) -> int:
    """Worker count: every host core, fewer if the per-worker memory (the
    oracle's float64 weight cache of 48 matrices, the inputs and the made
    expert matrices) would take more than a third of the available memory."""
    from mixture_experts_ffn_fp32_gb300 import workloads as W
    w = W.WORKLOADS[name]
    cores = os.cpu_count() or 1
    mat = max(w.d_expert, w.d) * max(w.d_ff, w.shared_d_ff)
    per = (48 * mat * 8 + 6 * w.K * mat * 2 + 3 * w.T * w.d * 4) / 1e9
    return max(1, min(cores, int(_mem_available_gb() / 3 / max(per, 1e-3))))


def _pool(n):
    ctx = mp.get_context("spawn")
    os.environ.update({"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1",
                       "MKL_NUM_THREADS": "1"})
    return ctx.Pool(n)


def sample_tokens(T: int, n: int, offset: int = 0) -> list:
    """n evenly spaced tokens of T, shifted by offset (wrapping)."""
    n = max(1, min(n, T))
    step = T / n
    return sorted({(int(i * step) + offset) % T for i in range(n)})


def oracle_sample_size(name: str) -> int:
    """Tokens for about 10-30 s of oracle work on the machine's cores."""
    from mixture_experts_ffn_fp32_gb300 import workloads as W
    w = W.WORKLOADS[name]
    per_tok = (w.K + w.n_shared) * 3 * (w.latent_dim or w.d) * max(w.d_ff, w.shared_d_ff)
    return int(max(16, min(w.T, 2e10 // max(per_tok, 1))))


def time_oracle(name: str, tokens: list, pool, workers: int, seed: int = 0) -> dict:
    """The oracle on `tokens`, split over the workers. All-core throughput =
    tokens / the slowest worker's oracle time; single-thread = tokens / the
    summed oracle time of all workers."""
    chunks = [tokens[i::workers] for i in range(workers)]
    chunks = [c for c in chunks if c]
    t0 = time.perf_counter()
    res = pool.map(_oracle_worker, [(name, c, seed) for c in chunks])
    wall = time.perf_counter() - t0
    busy = [r[0] for r in res]
    return {"tokens": len(tokens), "slowest_s": max(busy), "cpu_s": sum(busy), "wall_s": wall,
            "value": len(tokens) / max(busy), "single_thread_value": len(tokens) / sum(busy),
            "workers": len(chunks)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def gemm_kernel_name(w) -> str:
    """The grouped GEMM kernel the forward's gate/up launch takes: the
    token-column CTA pair where routed segments average 128 to 511 rows (the
    library's rule, MOE_GEMM_FORM overriding it), else the row-tile kernel."""
    form = os.environ.get("MOE_GEMM_FORM", "")
    rows, E = w.T * w.K, w.E
    token = form.startswith("t") or (not form.startswith("r") and 128 * E <= rows < 512 * E)
    return "tc_token_pair_kernel<SwiGLU>" if token else "tc_grouped_gemm_kernel<SwiGLU>"


def gate_up_roofline(w, gu_ms, counts, pk, name):
    """The grouped gate/up launch against the roof that bounds it: tensor on
    prefill batches, HBM (weight streaming) on decode batches, FP32 FFMA for
    the FP32 layer."""
    gu_flops = gate_up_flops(w)
    gu_bytes = gate_up_bytes(w, counts)
    f32 = w.dtype == "f32"
    flop_peak = pk["fp32_tflops"] if f32 else pk["bf16_tflops"]
    hbm = gu_bytes / (pk["hbm_gbs"] * 1e9) > gu_flops / (flop_peak * 1e12)
    ok = gu_ms and gu_ms > 0
    if f32:
        roof = {"kernel": "simt_grouped_gemm_kernel (gate_up)", "bound": "alu",
                "achieved": gu_flops / (gu_ms / 1e3) / 1e12 if ok else None, "peak": flop_peak,
                "unit": "TFLOP/s",
                "peak_source": "FP32 FFMA: 152 SMs x 128 lanes x 2 FLOP x max SM clock",
                "flops_per_launch": gu_flops}
    elif hbm:
        roof = {"kernel": gemm_kernel_name(w) + " (gate_up)", "bound": "hbm",
                "achieved": gu_bytes / (gu_ms / 1e3) / 1e9 if ok else None,
                "peak": pk["hbm_gbs"], "unit": "GB/s",
                "peak_source": f"{pk['source']} HBM copy", "bytes_per_launch": gu_bytes}
    else:
        roof = {"kernel": gemm_kernel_name(w) + " (gate_up)", "bound": "tensor",
                "achieved": gu_flops / (gu_ms / 1e3) / 1e12 if ok else None,
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "peak_source": f"{pk['source']} bf16 burst", "flops_per_launch": gu_flops}
    roof["frac"] = roof["achieved"] / roof["peak"] if roof["achieved"] else None
    sus = pk.get("bf16_tflops_sustained")
    if roof["bound"] == "tensor" and sus and roof["achieved"]:
        # the same launch against the cuBLAS rate sustained for seconds under the power cap
        roof["peak_sustained"] = sus
        roof["frac_of_sustained"] = roof["achieved"] / sus
    traffic, note = profiled_traffic(name)
    roof["traffic"] = traffic
    if note:
        roof["traffic_note"] = note.replace("_", " ")
    roof["algorithmic_bytes_per_launch"] = gu_bytes
    roof["avg_launch_ms"] = gu_ms
    return roof


def fused_bytes(w, counts=None) -> float:
    """Algorithmic HBM bytes of the fused decode back end: the weights of the
    experts that get tokens and of the shared experts, x read, out written."""
    return layer_bytes(w, counts) - w.d * w.E * 4


def dominant_roofline(w, stages, ncalls, counts, pk, name):
    """The dominant kernel of the forward against its roof: the fused decode
    back end where it ran (HBM-bound weight streaming), else the grouped
    gate/up launch."""
    fz = stages.get("decode_fused", 0.0) / max(1, ncalls)
    if fz > 0:
        b = fused_bytes(w, counts)
        ach = b / (fz / 1e3) / 1e9
        return {"kernel": "decode_fused_kernel (dispatch + gate/up + down + combine)",
                "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "peak_source": f"{pk['source']} HBM copy", "bytes_per_launch": b,
                "frac": ach / pk["hbm_gbs"], "traffic": None, "algorithmic_bytes_per_launch": b,
                "avg_launch_ms": fz}
    return gate_up_roofline(w, stages.get("gate_up", 0.0) / max(1, ncalls), counts, pk, name)


class Layer:
    """One workload's inputs, workspace and output on the device."""

    def __init__(self, api, W, name, dev, seed, out_dtype):
        self.w = W.WORKLOADS[name]
        self.name = name
        self.api = api
        self.spec = api.LayerSpec.of(self.w, out_dtype=out_dtype)
        self.inp = W.make_inputs(self.w, device=dev, seed=seed)
        self.ws = api.alloc_workspace(self.spec, dev)
        import torch
        self.out = torch.empty((self.w.T, self.w.d), dtype=self.spec.torch_out_dtype, device=dev)

    def step(self, stream):
        self.api.forward(self.spec, self.inp["x"], self.inp, out=self.out, ws=self.ws,
                         stream=stream)

    def check(self, stream, when):
        st = self.api.workspace_status(self.ws, stream)
        if st != self.api.MOE_OK:
            raise RuntimeError(f"{self.name}: device status {when}: {self.api.status_string(st)}")

    def routing_summary(self):
        v = self.api.workspace_views(self.spec, self.ws)
        counts = v["counts"].cpu().tolist()
        margin = v["margin"].float().cpu()
        return counts, int((margin <= NEAR_TIE).sum())


def time_steps(layer, stream, flush, steps, stage_timer=None):
    """Mean CUDA-event time of `steps` forwards, L2 flushed before each (outside
    the events)."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        l2_flush(flush, i)
        starts[i].record(stream)
        layer.step(stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return sum(per) / len(per)


def stage_breakdown(api, layer, stream, flush, n):
    """Per-stage times from an instrumented pass (an event between stages)."""
    timer = api.StageTimer(n)
    for i in range(n):
        l2_flush(flush, i)
        layer.step(stream)
    br, nb = timer.finish()
    return {k: v / max(1, nb) for k, v in br.items() if v > 0}


def measure_workload(api, W, name, dev, stream, flush, steps, warmup, out_dtype, pk):
    """One configuration: warm-up, timed forwards, gate/up launch time, stage
    breakdown, roofline fractions and the router's near-tie count."""
    import torch
    layer = Layer(api, W, name, dev, 0, out_dtype)
    for _ in range(warmup):
        layer.step(stream)
    layer.check(stream, "after warm-up")
    timer = api.StageTimer(steps, stages=["gate_up", "decode_fused"])
    ms = time_steps(layer, stream, flush, steps)
    st, nc = timer.finish()
    layer.check(stream, "after the timed steps")
    counts, near = layer.routing_summary()
    w = layer.w
    res = {"T": w.T, "ms_per_step": ms, "tokens_per_s": w.T / (ms / 1e3),
           "tflops": w.flops() / (ms / 1e3) / 1e12,
           "layer_roofline": layer_roofline(w, ms, counts, pk),
           "dominant": dominant_roofline(w, st, nc, counts, pk, name),
           "stage_ms": stage_breakdown(api, layer, stream, flush, min(steps, 5)),
           "near_ties_at_selection": near, "experts_used": sum(1 for c in counts if c > 0)}
    del layer
    torch.cuda.empty_cache()
    return res


def time_backward(api, W, layer, dev, stream, flush, n_bw, pk):
    """Forward then moe_backward on one workspace, each timed with CUDA events
    (L2 flushed before each forward); the forward keeps its gate/up products
    (save_gate_up) for a tensor-core layer, and the recomputing form is timed
    too."""
    import torch
    w = layer.w
    torch.manual_seed(1)
    dout = torch.randn(w.T, w.d, device=dev, dtype=torch.float32)
    de = w.latent_dim or w.d
    tc = (w.dtype == "bf16" and w.d % 64 == 0 and w.d_ff % 64 == 0 and de % 64 == 0
          and (w.n_shared == 0 or w.shared_d_ff % 64 == 0))

    def run(bspec):
        bws = torch.empty(api.backward_workspace_size(bspec), dtype=torch.uint8, device=dev)
        fws = layer.ws if bspec is layer.spec else torch.empty(api.workspace_size(bspec),
                                                               dtype=torch.uint8, device=dev)
        grads = {n: torch.empty(s_, dtype=torch.float32, device=dev)
                 for n, s_ in api.grad_shapes(bspec).items()}
        f_ms, b_ms = [], []
        for i in range(n_bw + 2):
            l2_flush(flush, i)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            api.forward(bspec, layer.inp["x"], layer.inp, out=layer.out, ws=fws, stream=stream)
            ev[1].record(stream)
            api.backward(bspec, layer.inp["x"], layer.inp, dout, fws, grads=grads, bws=bws,
                         stream=stream)
            ev[2].record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                f_ms.append(ev[0].elapsed_time(ev[1]))
                b_ms.append(ev[1].elapsed_time(ev[2]))
        st = api.workspace_status(fws, stream)
        if st != api.MOE_OK:
            raise RuntimeError(f"device status after the backward: {api.status_string(st)}")
        del bws, grads, fws
        torch.cuda.empty_cache()
        return sum(f_ms) / len(f_ms), sum(b_ms) / len(b_ms)

    f_re, b_re = run(layer.spec)
    bfl = backward_flops(w)
    bpk = pk["bf16_tflops"] if tc else pk["fp32_tflops"]
    counts, _ = layer.routing_summary()
    t_flop = bfl / (bpk * 1e12) * 1e3
    t_hbm = backward_bytes(w, counts) / (pk["hbm_gbs"] * 1e9) * 1e3
    if tc:
        f_sv, bms = run(api.LayerSpec.of(w, save_gate_up=True))
    else:
        f_sv, bms = f_re, b_re
    return {"ms": bms, "tflops": bfl / (bms / 1e3) / 1e12, "flops_per_step": bfl,
            "bound": "tensor" if tc else "alu", "peak": bpk, "unit": "TFLOP/s",
            "frac": bfl / (bms / 1e3) / 1e12 / bpk,
            "layer_roofline": {"t_flop_ms": t_flop, "t_hbm_ms": t_hbm,
                               "bound": ("tensor" if tc else "alu") if t_flop >= t_hbm else "hbm",
                               "frac": max(t_flop, t_hbm) / bms,
                               "bytes_per_step": backward_bytes(w, counts),
                               "note": "max(FLOPs / peak, algorithmic bytes / HBM copy rate) over the "
                                       "backward's time; the bytes read x, the upstream gradient and "
                                       "the used experts' weights once and write dx and every weight "
                                       "gradient (FP32) once"},
            "forward_ms": f_sv, "training_step_ms": f_sv + bms,
            "recompute": {"ms": b_re, "forward_ms": f_re, "training_step_ms": f_re + b_re},
            "note": ("moe_backward (all gradients) after a forward on the same workspace; "
                     + ("the forward keeps its BF16 gate/up products (save_gate_up) and the "
                        "backward reads them ('recompute': the backward recomputes them "
                        "instead); expert contractions on tcgen05 (BF16 operands, FP32 sums), "
                        "peak = measured BF16 burst; " if tc else
                        "FP32 FFMA grouped GEMMs, peak = FP32 FFMA; ")
                     + "L2 flushed before each forward; CUDA events around the forward and "
                       "the backward separately; FLOPs exclude recomputed products")}


def gpu_index_of(local):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            return int(vis.split(",")[local])
        except (ValueError, IndexError):
            return local
    return local


def run_ours(args, name):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from mixture_experts_ffn_fp32_gb300 import build
    build.build()
    from mixture_experts_ffn_fp32_gb300 import api
    from mixture_experts_ffn_fp32_gb300 import workloads as W

    pk = peaks()
    layer = Layer(api, W, name, dev, rank, args.out_dtype)
    w = layer.w
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        layer.step(stream)
    layer.check(stream, "after warm-up")
    counts, near = layer.routing_summary()

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = Clocks(gpu_index_of(local))
    clocks.start()
    barrier()
    n0 = api.launch_count()
    timer = api.StageTimer(args.steps, stages=["gate_up", "decode_fused"])
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        l2_flush(flush, i)
        starts[i].record(stream)
        layer.step(stream)
        ends[i].record(stream)
    barrier()
    t_wall = time.perf_counter() - t_wall0
    stages, ncalls = timer.finish()
    launches = api.launch_count() - n0
    clk = clocks.stop()
    layer.check(stream, "after the timed steps")
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(sum(per) / len(per), dev)
    breakdown = stage_breakdown(api, layer, stream, flush, min(args.steps, 20))

    # end to end through the host-buffer entry point (copies inside the timed region)
    e2e = None
    if not args.no_e2e:
        xh = layer.inp["x"].cpu().pin_memory()
        oh = torch.empty((w.T, w.d), dtype=layer.spec.torch_out_dtype).pin_memory()
        for _ in range(max(1, args.warmup)):
            api.forward_host(layer.spec, xh, layer.inp, oh, layer.ws, stream=stream)
        e_ms = []
        for i in range(args.steps):
            l2_flush(flush, i)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            api.forward_host(layer.spec, xh, layer.inp, oh, layer.ws, stream=stream)
            b.record(stream)
            b.synchronize()
            e_ms.append(a.elapsed_time(b))
        em = max_over_ranks(sum(e_ms) / len(e_ms), dev)
        e2e = {"value": job_tokens_per_s(w.T, world, em), "unit": "tokens/s",
               "h2d_bytes_per_step": xh.numel() * xh.element_size(),
               "d2h_bytes_per_step": oh.numel() * oh.element_size(), "ms_per_step": em}
        del xh, oh

    if rank != 0:
        del layer
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    # routing diagnostics (Switch loss, z-loss; moe_routing_stats): their own
    # pass, outside the timed forward region
    diag = None
    bwd = None
    if world == 1 and not args.no_diag:
        dws = api.alloc_workspace(layer.spec)
        x, Wr, b = layer.inp["x"], layer.inp["W_router"], layer.inp["bias"]
        api.routing_stats(layer.spec, x, Wr, b, ws=dws, stream=stream)
        d_ms = []
        for i in range(min(args.steps, 10)):
            l2_flush(flush, i)
            ea = torch.cuda.Event(enable_timing=True)
            eb = torch.cuda.Event(enable_timing=True)
            ea.record(stream)
            api.routing_stats(layer.spec, x, Wr, b, ws=dws, stream=stream, read=False)
            eb.record(stream)
            torch.cuda.synchronize()
            d_ms.append(ea.elapsed_time(eb))
        g = api.routing_stats(layer.spec, x, Wr, b, ws=dws, stream=stream)
        diag = {"ms": sum(d_ms) / len(d_ms), "aux": g["aux"], "z": g["z"],
                "note": "moe_routing_stats (router + diagnostics reduction) timed alone with "
                        "CUDA events, L2 flushed before each call"}
        del dws
    if world == 1:
        if not args.no_backward:
            bwd = time_backward(api, W, layer, dev, stream, flush, max(1, min(args.steps, 5)), pk)

    line = {
        "metric": METRIC, "value": job_tokens_per_s(w.T, world, ms), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": config_of(w, name, args.out_dtype, world),
        "tflops": w.flops() / (ms / 1e3) / 1e12 * world,
        "tflops_per_gpu": w.flops() / (ms / 1e3) / 1e12,
        "layer_roofline": layer_roofline(w, ms, counts, pk),
        "roofline": dominant_roofline(w, stages, ncalls, counts, pk, name),
        "stage_ms": breakdown,
        "stage_ms_note": "separate instrumented pass (an event between every stage)",
        "near_ties_at_selection": near,
        "near_ties_note": ("tokens whose router margin (selection score at rank K minus rank "
                           "K+1, the router's own output) is at most 1e-5"),
        "routing_diagnostics": diag,
        "backward": bwd,
        "gpu_launches": int(launches),
        "wall_s_timed": t_wall,
        "clocks": clk,
        "e2e": e2e,
    }
    del layer
    torch.cuda.empty_cache()

    if world == 1 and not args.no_workloads:
        blk = {}
        bclk = Clocks(gpu_index_of(local))
        bclk.start()
        for other in W.ALL_BENCH:
            blk[other] = measure_workload(api, W, other, dev, stream, flush, args.workload_steps,
                                          3, args.out_dtype, pk)
        line["workloads"] = blk
        line["workloads_note"] = (f"every configuration, {args.workload_steps} timed forwards "
                                  "after 3 warm-ups, L2 flushed between them, CUDA events; "
                                  "dominant = the dominant kernel against its roof: the grouped "
                                  "gate/up launch, or the fused decode back end")
        line["workloads_clocks"] = bclk.stop()

    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(name)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def config_of(w, name, out_dtype, world):
    return {"workload": name, "T": w.T, "d": w.d, "d_ff": w.d_ff, "E": w.E, "K": w.K,
            "n_shared": w.n_shared, "shared_d_ff": w.shared_d_ff, "latent_dim": w.latent_dim,
            "gate": w.gate, "out_dtype": out_dtype,
            "parallelism": "replicas" if world > 1 else "single", "l2": L2_NOTE}


def cpu_baseline(name):
    """The oracle as it stands on a bounded, evenly spaced sample of the
    workload's tokens, all host cores (spawned single-threaded workers)."""
    from mixture_experts_ffn_fp32_gb300 import workloads as W
    w = W.WORKLOADS[name]
    workers = oracle_workers(name)
    toks = sample_tokens(w.T, oracle_sample_size(name))
    pool = _pool(workers)
    try:
        r = time_oracle(name, toks, pool, workers)
    finally:
        pool.close()
    return {"value": r["value"], "unit": "tokens/s", "cores": r["workers"], "kind": "oracle",
            "single_thread_value": r["single_thread_value"],
            "sample": (f"{r['tokens']} of {w.T} tokens (evenly spaced), full layer per token, "
                       f"float64 NumPy oracle (per-token loop), {r['workers']} spawned "
                       f"single-threaded workers, {r['cpu_s']:.1f} CPU-s of oracle time; "
                       "value = tokens / the slowest worker's oracle time, single_thread_value "
                       "= tokens / the summed oracle time; making the random expert matrices "
                       "is not counted")}


def run_reference(args, name):
    """The CPU oracle as the reference arm: each step runs it on a bounded,
    evenly spaced sample of the workload's tokens (shifted every step) on all
    host cores; ms_per_step is the measured oracle time of that work."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from mixture_experts_ffn_fp32_gb300 import workloads as W
    w = W.WORKLOADS[name]
    workers = oracle_workers(name)
    n = max(workers, oracle_sample_size(name) // max(1, args.steps + args.warmup))
    pool = _pool(workers)
    try:
        for i in range(args.warmup):
            time_oracle(name, sample_tokens(w.T, n, offset=i), pool, workers)
        runs = []
        t0 = time.perf_counter()
        for i in range(args.steps):
            runs.append(time_oracle(name, sample_tokens(w.T, n, offset=args.warmup + i), pool,
                                    workers))
        wall = time.perf_counter() - t0
    finally:
        pool.close()
    step_s = [r["slowest_s"] for r in runs]
    toks = sum(r["tokens"] for r in runs)
    value = toks / sum(step_s)
    single = toks / sum(r["cpu_s"] for r in runs)
    ms = 1e3 * sum(step_s) / len(step_s)
    sample = (f"{n} of {w.T} tokens per step (evenly spaced, shifted by one token each step), "
              f"full layer per token, float64 NumPy oracle (per-token loop), {workers} spawned "
              "single-threaded workers; a step's time is its slowest worker's oracle time")
    line = {"metric": METRIC, "impl": "reference", "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, name, args.out_dtype, world),
            "tokens_per_step": n,
            "ms_per_layer_extrapolated": 1e3 * w.T / value,
            "wall_s_timed": wall,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": workers,
                             "kind": "oracle", "single_thread_value": single, "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    from mixture_experts_ffn_fp32_gb300 import workloads as W
    name = args.workload or W.BENCH_WORKLOAD
    if name not in W.WORKLOADS:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(W.WORKLOADS)}")
    if args.impl == "reference":
        run_reference(args, name)
    else:
        run_ours(args, name)


if __name__ == "__main__":
    main()
