"""Throughput of the routed MoE SwiGLU FFN layer forward on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--no-cpu-baseline]

One step = one whole layer forward (router, dispatch, grouped gate/up,
grouped down, shared experts, combine) over one batch of T synthetic tokens
with inputs resident in HBM. Each timed step is bracketed by CUDA events on
the launching stream; L2 is flushed (a 256 MB write, larger than the 129 MB
L2) between timed steps, outside the events. The JSON line reports whole-job
tokens/s (all ranks), the layer's TFLOP/s, the dominant kernel's roofline
fraction (measured by the library's own stage events), the end-to-end number
through moe_forward_host (host buffers, copies inside the timed region), SM
clocks sampled during the timed region, and the CPU oracle on a bounded
sample of the same workload. With N > 1 (torchrun) every rank runs an
independent replica of the layer on its own GPU (the layer has no exchange
step on one GPU); the step time is the max over ranks.

--impl reference times the CPU oracle (float64 NumPy, per-token loop) on the
host cores, on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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
    """FLOPs of the grouped gate/up launch: routed rows x 2 matrices + shared."""
    de = w.latent_dim or w.d
    f = 4.0 * w.T * w.K * de * w.d_ff
    if not w.latent_dim:
        f += 4.0 * w.T * w.d * w.shared_d_ff * w.n_shared
    return f


def gate_up_bytes(w, counts=None) -> float:
    """Algorithmic HBM bytes of the grouped gate/up launch: gate and up weights
    of the experts that get tokens and of the shared experts, the BF16 operand
    rows read once, the BF16 hidden rows written once."""
    es = 4 if w.dtype == "f32" else 2
    de = w.latent_dim or w.d
    used = w.E if counts is None else int(sum(1 for c in counts if c > 0))
    b = used * 2 * de * w.d_ff * es + w.T * w.K * de * es + w.T * w.K * w.d_ff * es
    if not w.latent_dim:
        b += w.n_shared * 2 * w.d * w.shared_d_ff * es
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


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "common.cuh", "warp_stage.cuh"):
        with open(os.path.join(ROOT, "mixture_experts_ffn_fp32_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the gate/up kernel from the committed ncu
    summary (profiles/gate_up_traffic.txt), if it was taken on the current
    kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "gate_up_traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    with open(path) as f:
        for ln in f:
            if ln.startswith("#") or "=" not in ln:
                continue
            kv = dict(p.split("=", 1) for p in ln.split())
            if kv.get("workload") == workload and kv.get("kernel_source") == src:
                return int(kv["dram_bytes_per_launch"])
    return None


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
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def _oracle_worker(args):
    name, T, tokens, seed = args
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    import numpy as np  # noqa: F401
    from mixture_experts_ffn_fp32_gb300 import workloads as W
    from oracle import moe_oracle as O
    w = W.WORKLOADS[name].resized(T=T)
    inp = W.make_inputs(w, device="cpu", seed=seed)
    t0 = time.perf_counter()
    O.moe_forward(inp["x"], inp, w.gate, w.K, w.renormalize, w.routed_scale, tokens=tokens)
    return time.perf_counter() - t0


def _pool(n):
    ctx = mp.get_context("spawn")
    env_threads = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}
    os.environ.update(env_threads)
    return ctx.Pool(n)


def cpu_oracle_tokens_per_s(name: str, n_tokens: int, pool, cores: int, seed: int = 0):
    """Time the oracle on n_tokens tokens of the workload, split over the pool."""
    from mixture_experts_ffn_fp32_gb300 import workloads as W
    w = W.WORKLOADS[name]
    step = max(1, w.T // n_tokens)
    toks = list(range(0, w.T, step))[:n_tokens]
    chunks = [toks[i::cores] for i in range(cores)]
    chunks = [c for c in chunks if c]
    t0 = time.perf_counter()
    busy = pool.map(_oracle_worker, [(name, w.T, c, seed) for c in chunks])
    wall = time.perf_counter() - t0
    # throughput over the oracle's own compute (slowest worker), not input generation
    return len(toks) / max(busy), {"tokens": len(toks), "cpu_seconds": sum(busy), "wall_s": wall}


def oracle_sample_tokens(name: str) -> int:
    from mixture_experts_ffn_fp32_gb300 import workloads as W
    w = W.WORKLOADS[name]
    per_tok = (w.K + w.n_shared) * 3 * (w.latent_dim or w.d) * max(w.d_ff, w.shared_d_ff)
    # about 2e10 multiply-adds in total (~10-30 s of CPU work at a few GFLOP/s)
    return int(max(16, min(w.T, 2e10 // max(per_tok, 1))))


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args, name):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from mixture_experts_ffn_fp32_gb300 import workloads as W
    w = W.WORKLOADS[name]
    cores = os.cpu_count() or 1
    n = max(cores, oracle_sample_tokens(name) // max(1, args.steps + args.warmup))
    pool = _pool(cores)
    try:
        for _ in range(args.warmup):
            cpu_oracle_tokens_per_s(name, n, pool, cores)
        rates, secs = [], 0.0
        for _ in range(args.steps):
            r, info = cpu_oracle_tokens_per_s(name, n, pool, cores)
            rates.append(r)
            secs += info["wall_s"]
    finally:
        pool.close()
    value = statistics.median(rates)
    sample = (f"{n} of {w.T} tokens per step (evenly spaced), full layer per token, "
              f"float64 NumPy oracle, {cores} spawned single-threaded workers")
    line = {"metric": METRIC, "impl": "reference", "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * w.T / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "T": w.T, "d": w.d, "d_ff": w.d_ff, "E": w.E,
                       "K": w.K, "n_shared": w.n_shared, "shared_d_ff": w.shared_d_ff,
                       "latent_dim": w.latent_dim, "gate": w.gate},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


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

    w = W.WORKLOADS[name]
    spec = api.LayerSpec.of(w, out_dtype=args.out_dtype)
    inp = W.make_inputs(w, device=dev, seed=rank)
    ws = api.alloc_workspace(spec, dev)
    out = torch.empty((w.T, w.d), dtype=spec.torch_out_dtype, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        api.forward(spec, inp["x"], inp, out=out, ws=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    st = api.workspace_status(ws, stream)
    if st != api.MOE_OK:
        raise RuntimeError(f"device status after warm-up: {api.status_string(st)}")
    counts = api.workspace_views(spec, ws)["counts"].cpu().tolist()

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[local])
        except ValueError:
            gpu_index = local
    clocks = Clocks(gpu_index)
    clocks.start()
    barrier()
    n0 = api.launch_count()
    timer = api.StageTimer(args.steps, stages=["gate_up"])
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    barrier()
    t_wall = time.perf_counter() - t_wall0
    stages, ncalls = timer.finish()
    launches = api.launch_count() - n0
    clk = clocks.stop()
    st = api.workspace_status(ws, stream)
    if st != api.MOE_OK:
        raise RuntimeError(f"device status after the timed steps: {api.status_string(st)}")
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(sum(per) / len(per), dev)
    # per-stage breakdown from a separate instrumented pass (events between every stage)
    n_inst = min(args.steps, 20)
    timer2 = api.StageTimer(n_inst)
    for i in range(n_inst):
        flush.fill_(i & 0xFF)
        step()
    breakdown, nb = timer2.finish()

    # routing diagnostics (Switch loss, z-loss; moe_routing_stats): their own
    # pass, outside the timed forward region
    diag = None
    if world == 1:
        dws = api.alloc_workspace(spec)
        api.routing_stats(spec, inp["x"], inp["W_router"], inp["bias"], ws=dws, stream=stream)
        d_ms = []
        for i in range(min(args.steps, 10)):
            flush.fill_(i & 0xFF)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            api.routing_stats(spec, inp["x"], inp["W_router"], inp["bias"], ws=dws,
                              stream=stream, read=False)
            b.record(stream)
            torch.cuda.synchronize()
            d_ms.append(a.elapsed_time(b))
        g = api.routing_stats(spec, inp["x"], inp["W_router"], inp["bias"], ws=dws, stream=stream)
        diag = {"ms": sum(d_ms) / len(d_ms), "aux": g["aux"], "z": g["z"],
                "note": "moe_routing_stats (router + diagnostics reduction) timed alone with "
                        "CUDA events, L2 flushed before each call"}
        del dws

    # backward (moe_backward after the forward on ws): its own pass, outside the
    # timed forward region
    bwd = None
    if world == 1 and not args.no_backward:
        torch.manual_seed(1)
        dout = torch.randn(w.T, w.d, device=dev, dtype=torch.float32)
        de = w.latent_dim or w.d
        tc = (w.dtype == "bf16" and w.d % 64 == 0 and w.d_ff % 64 == 0 and de % 64 == 0
              and (w.n_shared == 0 or w.shared_d_ff % 64 == 0))
        n_bw = max(1, min(args.steps, 5))

        def time_backward(bspec):
            """Forward then backward on one workspace, each timed with CUDA events
            (L2 flushed before each forward); averages over n_bw steps after 2."""
            bws_ = torch.empty(api.backward_workspace_size(bspec), dtype=torch.uint8, device=dev)
            fws = ws if bspec is spec else torch.empty(api.workspace_size(bspec), dtype=torch.uint8,
                                                       device=dev)
            grads = {n: torch.empty(s_, dtype=torch.float32, device=dev)
                     for n, s_ in api.grad_shapes(bspec).items()}
            f_ms, b_ms = [], []
            for i in range(n_bw + 2):
                flush.fill_(i & 0xFF)
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                ev[0].record(stream)
                api.forward(bspec, inp["x"], inp, out=out, ws=fws, stream=stream)
                ev[1].record(stream)
                api.backward(bspec, inp["x"], inp, dout, fws, grads=grads, bws=bws_, stream=stream)
                ev[2].record(stream)
                torch.cuda.synchronize()
                if i >= 2:
                    f_ms.append(ev[0].elapsed_time(ev[1]))
                    b_ms.append(ev[1].elapsed_time(ev[2]))
            st_ = api.workspace_status(fws, stream)
            if st_ != api.MOE_OK:
                raise RuntimeError(f"device status after the backward: {api.status_string(st_)}")
            del bws_, grads
            return sum(f_ms) / len(f_ms), sum(b_ms) / len(b_ms)

        f_re, b_re = time_backward(spec)
        bfl = backward_flops(w)
        pk0 = peaks()
        bpk = pk0["bf16_tflops"] if tc else pk0["fp32_tflops"]
        if tc:
            # training form: the forward keeps its gate/up products, the backward reads them
            tspec = api.LayerSpec.of(w, save_gate_up=True)
            f_sv, bms = time_backward(tspec)
        else:
            f_sv, bms = f_re, b_re
        bwd = {"ms": bms, "tflops": bfl / (bms / 1e3) / 1e12, "flops_per_step": bfl,
               "bound": "tensor" if tc else "alu", "peak": bpk, "unit": "TFLOP/s",
               "frac": bfl / (bms / 1e3) / 1e12 / bpk,
               "forward_ms": f_sv, "training_step_ms": f_sv + bms,
               "recompute": {"ms": b_re, "forward_ms": f_re, "training_step_ms": f_re + b_re},
               "note": ("moe_backward (all gradients) after a forward on the same workspace; "
                        + ("the forward keeps its BF16 gate/up products (save_gate_up) and the "
                           "backward reads them ('recompute': the backward recomputes them "
                           "instead); expert contractions on tcgen05 (BF16 operands, FP32 "
                           "sums), peak = measured BF16 burst; " if tc else
                           "FP32 FFMA grouped GEMMs, peak = FP32 FFMA; ")
                        + "L2 flushed before each forward; CUDA events around the forward "
                          "and the backward separately; FLOPs exclude recomputed products")}
        del dout

    # end to end through the host-buffer entry point (copies inside the timed region)
    e2e = None
    if not args.no_e2e:
        xh = inp["x"].cpu().pin_memory()
        oh = torch.empty((w.T, w.d), dtype=spec.torch_out_dtype).pin_memory()
        for _ in range(max(1, args.warmup)):
            api.forward_host(spec, xh, inp, oh, ws, stream=stream)
        e_ms = []
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            api.forward_host(spec, xh, inp, oh, ws, stream=stream)
            b.record(stream)
            b.synchronize()
            e_ms.append(a.elapsed_time(b))
        em = max_over_ranks(sum(e_ms) / len(e_ms), dev)
        e2e = {"value": job_tokens_per_s(w.T, world, em), "unit": "tokens/s",
               "h2d_bytes_per_step": xh.numel() * xh.element_size(),
               "d2h_bytes_per_step": oh.numel() * oh.element_size(), "ms_per_step": em}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    pk = peaks()
    flops = w.flops()
    tflops = flops / (ms / 1e3) / 1e12
    gu_ms = stages.get("gate_up", 0.0) / max(1, ncalls)
    gu_flops = gate_up_flops(w)
    gu_bytes = gate_up_bytes(w, counts)
    traffic = profiled_traffic(name)
    t_flop = flops / (pk["bf16_tflops"] * 1e12)
    t_hbm = layer_bytes(w, counts) / (pk["hbm_gbs"] * 1e9)
    # the gate/up launch is tensor-bound on prefill and weight-streaming
    # (HBM-bound) on decode: report it against the roof that bounds it
    f32 = w.dtype == "f32"
    flop_peak = pk["fp32_tflops"] if f32 else pk["bf16_tflops"]
    gu_hbm = gu_bytes / (pk["hbm_gbs"] * 1e9) > gu_flops / (flop_peak * 1e12)
    if f32:
        # the FP32 layer's grouped GEMMs run on the CUDA cores (FFMA)
        achieved = gu_flops / (gu_ms / 1e3) / 1e12 if gu_ms > 0 else None
        roof = {"bound": "alu", "achieved": achieved, "peak": flop_peak, "unit": "TFLOP/s",
                "peak_source": "FP32 FFMA: 152 SMs x 128 lanes x 2 FLOP x max SM clock",
                "flops_per_launch": gu_flops}
    elif gu_hbm:
        achieved = gu_bytes / (gu_ms / 1e3) / 1e9 if gu_ms > 0 else None
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "peak_source": f"{pk['source']} HBM copy", "bytes_per_launch": gu_bytes}
    else:
        achieved = gu_flops / (gu_ms / 1e3) / 1e12 if gu_ms > 0 else None
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "peak_source": f"{pk['source']} bf16 burst",
                "flops_per_launch": gu_flops}
    roof["frac"] = (achieved / roof["peak"]) if achieved else None
    roof["traffic"] = traffic
    roof["avg_launch_ms"] = gu_ms
    line = {
        "metric": METRIC, "value": job_tokens_per_s(w.T, world, ms), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": name, "T": w.T, "d": w.d, "d_ff": w.d_ff, "E": w.E, "K": w.K,
                   "n_shared": w.n_shared, "shared_d_ff": w.shared_d_ff,
                   "latent_dim": w.latent_dim, "gate": w.gate, "out_dtype": args.out_dtype,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed between timed steps (256 MB write, outside the events)"},
        "tflops": tflops * world, "tflops_per_gpu": tflops,
        "layer_roofline": {"t_flop_ms": t_flop * 1e3, "t_hbm_ms": t_hbm * 1e3,
                           "bound": "tensor" if t_flop >= t_hbm else "hbm",
                           "frac": max(t_flop, t_hbm) * 1e3 / ms,
                           "peak_source": pk["source"]},
        "roofline": {"kernel": ("simt_grouped_gemm_kernel (gate_up)" if f32 else
                                "tc_grouped_gemm_kernel<SwiGLU> (gate_up)"), **roof},
        "stage_ms": {k: v / max(1, nb) for k, v in breakdown.items() if v > 0},
        "stage_ms_note": "separate instrumented pass (an event between every stage)",
        "routing_diagnostics": diag,
        "backward": bwd,
        "gpu_launches": int(launches),
        "wall_s_timed": t_wall,
        "clocks": clk,
        "e2e": e2e,
    }
    if not args.no_cpu_baseline and world == 1:
        cores = os.cpu_count() or 1
        n = oracle_sample_tokens(name)
        pool = _pool(cores)
        try:
            v, info = cpu_oracle_tokens_per_s(name, n, pool, cores)
        finally:
            pool.close()
        line["cpu_baseline"] = {
            "value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": (f"{info['tokens']} of {w.T} tokens (evenly spaced), full layer per token, "
                       f"float64 NumPy oracle, {cores} spawned single-threaded workers, "
                       f"{info['cpu_seconds']:.1f} CPU-s")}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


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
