"""Benchmark of the MoE FFN forward pass on GB300.

One step = one whole layer forward (route -> permute -> grouped gate/up+SwiGLU
-> grouped down -> shared MLP -> combine) over one batch of synthetic tokens,
through moe_layer_forward.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the fp64 CPU oracle on a sample)

The headline workload is the DeepSeek-V3-shaped prefill (T=8192, H=7168,
E=256, k=8, I=2048, one shared expert of width 2048), the largest layer that
fits one GPU; the line also carries the route + permute + combine stages
against their HBM floor and, under "per_config", the same measurements for
every other workload shape (fewer steps each).

Timing: W untimed warm-up steps, then K timed steps, each preceded by an L2
flush (a 256 MiB device write outside the timed interval); CUDA events on the
launching stream; barrier + synchronize around the timed region; max over
ranks.  Multi-GPU runs are independent replicas (every token is independent;
the layer has no exchange step without expert parallelism), so scaling is weak.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "deepseek-v3-shape-T8192"
# measured after the headline, in the same process (value, stages, fractions)
PER_CONFIG = ("tiny-f32-T64", "qwen3-30b-a3b-shape-T4096", "qwen2-moe-shape-T2048",
              "qwen2-moe-shape-T64", "qwen2-moe-shape-T8", "qwen2-moe-shape-T1",
              "adversarial-all-e0-T128", "adversarial-all-e0-T16384",
              "adversarial-zipf-T128", "adversarial-zipf-T16384",
              "gemma4-26b-a4b-shape-T4096")
METRIC = "MoE layer tokens/s and grouped-GEMM TFLOP/s (% bf16 peak) on 1 GB300"

# dram__bytes_read.sum + dram__bytes_write.sum of one gate/up grouped-GEMM
# launch, from an ncu capture, keyed by workload; valid only while the device
# code of the engine that ran it hashes to the recorded value.
# Nominal HBM3e bandwidth of a GB300 (the fractions against it sit beside the
# ones against the measured copy bandwidth).
NOMINAL_HBM_GBS = 7900.0

NCU_TRAFFIC = {
    # profiles/launches_qwen3-30b-a3b-shape-T4096.md (one-SM engine: K = 2048
    # and 128-row groups keep this layer off the SM-pair engine; first forward)
    "qwen3-30b-a3b-shape-T4096": {"bytes": 984256000, "kernel_hash": "7d2ea5ed3b98bf80"},
    # profiles/launches_deepseek-v3-shape-T8192.md (SM-pair engine; the launch
    # of the first forward: 16 206 901 504 B read + 265 844 224 B written)
    "deepseek-v3-shape-T8192": {"bytes": 16472745728, "kernel_hash": "6468578d8bae2304"},
}


def _kernel_hash(engine: str = "tc_gemm_kernel") -> str:
    """Hash of a grouped GEMM engine's device code: its PTX wrappers and the
    part of its source above the host-side launcher."""
    d = os.path.join(ROOT, "mixture_experts_ffn_04_gb300", "csrc")
    if engine == "tc2_gemm_kernel":
        src = open(os.path.join(d, "gemm_tc2.cu"), "rb").read()
        h = hashlib.sha256(open(os.path.join(d, "tcgen05.cuh"), "rb").read())
        h.update(open(os.path.join(d, "tc_pair.cuh"), "rb").read())
        h.update(src[:src.index(b"cudaError_t launch_gemm_tc2(")])
        return h.hexdigest()[:16]
    src = open(os.path.join(d, "gemm_tc.cu"), "rb").read()
    h = hashlib.sha256(open(os.path.join(d, "tcgen05.cuh"), "rb").read())
    h.update(src[:src.index(b"// host side")])
    return h.hexdigest()[:16]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def _dist():
    n = int(os.environ.get("WORLD_SIZE", "1"))
    if n > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist, dist.get_rank(), n
    return None, 0, 1


def max_over_ranks(v: float, dist) -> float:
    """The slowest rank's value (the job is done when the last replica is)."""
    if dist is None:
        return v
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank runs its own batch of tokens (weak scaling)."""
    return world * tokens_per_rank / (ms_per_step / 1000.0)


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def algorithmic(wl, counts: np.ndarray):
    """Algorithmic FLOPs and bytes (touched experts only, each weight byte once,
    activations once) of the gate/up GEMM, of the whole layer, and of the
    route, permute and combine stages:
      route    x + router weights read, topk_idx + topk_w (+ gate) written;
      permute  topk_idx read, x read once, its T*k grouped copies written,
               scatter_index + row_token written;
      combine  T*k grouped output rows (+ the shared row, + x for a residual)
               read, y written, scatter_index + topk_w read."""
    b = wl.esize
    # expert weights: the activation type, or packed MXFP8 (1 + 1/8 bytes a weight)
    wb = 1.125 if getattr(wl, "weights", "act") == "mxfp8" else b
    T, H, I, k, Ish = wl.T, wl.H, wl.I, wl.k, wl.I_sh
    touched = int((counts > 0).sum())
    rows = T * k
    gu_flops = 4.0 * rows * H * I
    gu_bytes = touched * 2.0 * I * H * wb + rows * H * b + rows * I * b
    dn_flops = 2.0 * rows * H * I
    layer_flops = wl.flops()
    n_router = (wl.E + (1 if wl.shared_gate else 0)) if wl.routing == "router" else 0
    layer_bytes = touched * 3.0 * I * H * wb + 3.0 * Ish * H * wb + T * H * b * 2 + n_router * H * b
    if getattr(wl, "input_norm", False):   # x_norm written once (x itself read already)
        layer_bytes += T * H * b + H * b
    if getattr(wl, "residual", False):     # x read again by the combine
        layer_bytes += T * H * b
    route_bytes = (T * H * b + n_router * H * b + rows * 8.0 + (T * 4.0 if wl.shared_gate else 0)
                   if wl.routing == "router" else 0.0)
    permute_bytes = rows * 4.0 + T * H * b + rows * H * b + rows * 8.0
    combine_bytes = (rows * H * b + (T * H * b if Ish else 0) + T * H * b + rows * 8.0
                     + (T * H * b if getattr(wl, "residual", False) else 0))
    return dict(gu_flops=gu_flops, gu_bytes=gu_bytes, dn_flops=dn_flops,
                gemm_flops=gu_flops + dn_flops + 6.0 * T * H * Ish,
                layer_flops=layer_flops, layer_bytes=layer_bytes, touched=touched,
                route_bytes=route_bytes, permute_bytes=permute_bytes,
                combine_bytes=combine_bytes)


class OracleSample:
    """The fp64 oracle (routing + expert FFNs + combine) on a fixed seeded
    sample of a workload's tokens.  The sample is sized once so that one run
    takes about target_s seconds; the expert weights it uses are staged on the
    host once (input preparation, not timed), so every run times only the
    oracle."""

    def __init__(self, wl, inputs, target_s: float, threads: int):
        from oracle import oracle as O
        self.O, self.wl, self.threads = O, wl, threads
        self.hin = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()
                    if k in ("x", "w_router", "routes_idx", "routes_w", "sh_gate", "sh_up",
                             "sh_down")}
        self.inputs = inputs
        rng = np.random.Generator(np.random.PCG64(99))
        self.order = rng.permutation(wl.T)
        n0 = min(wl.T, 8)
        self._prepare(n0)
        dt = self.run()
        n1 = int(max(1, min(wl.T, n0 * target_s / max(dt, 1e-9))))
        if n1 > n0:
            self._prepare(n1)

    def _prepare(self, n):
        self.tokens = np.sort(self.order[:n])
        r = self.O.route(self.wl, self.hin, self.tokens, nthreads=self.threads)
        used = np.unique(r["idx"])
        sel = torch.as_tensor(used, dtype=torch.long)
        self.w = [t.index_select(0, sel.to(t.device)).cpu()
                  for t in (self.inputs["w_gate"], self.inputs["w_up"], self.inputs["w_down"])]
        self.remap = np.zeros(self.wl.E, np.int32)
        self.remap[used] = np.arange(len(used), dtype=np.int32)
        self.n = n

    def run(self) -> float:
        """One timed pass over the sample; seconds."""
        O, h = self.O, self.hin
        t0 = time.perf_counter()
        r = O.route(self.wl, h, self.tokens, nthreads=self.threads)
        O.moe_ffn(h["x"], self.remap[r["idx"]], r["weights"], r["gate"], *self.w,
                  h.get("sh_gate"), h.get("sh_up"), h.get("sh_down"), tokens=self.tokens,
                  nthreads=self.threads)
        return time.perf_counter() - t0

    def describe(self, dt):
        return ("%d of the workload's %d tokens, seeded sample (routing + expert FFNs + "
                "combine in fp64), %.2f s a pass" % (self.n, self.wl.T, dt))


def run_reference(args, wl, rank, world):
    """--impl reference: the fp64 CPU oracle as it stands, on a bounded sample
    of the workload's tokens; each step is one pass over the sample, and
    ms_per_step is the time of that pass (the tokens it actually ran)."""
    if rank != 0:
        return
    from oracle import oracle as O
    O.load()
    threads = os.cpu_count() or 1
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inputs = _make_inputs(wl, dev)
    per_step_s = max(0.5, min(6.0, 120.0 / max(1, args.steps + args.warmup)))
    smp = OracleSample(wl, inputs, per_step_s, threads)
    times = []
    for i in range(args.warmup + args.steps):
        dt = smp.run()
        if i >= args.warmup:
            times.append(dt)
    sec = statistics.mean(times)
    value = smp.n / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * sec, "tokens_per_step": smp.n, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(wl),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": smp.describe(sec)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(wl):
    return {"workload": wl.name, "expert_weights": getattr(wl, "weights", "act"),
            "tokens": wl.T, "hidden": wl.H, "experts": wl.E,
            "top_k": wl.k, "moe_inter": wl.I, "shared_inter": wl.I_sh,
            "shared_gate": wl.shared_gate, "norm_topk": wl.norm_topk, "routing": wl.routing,
            "l2": "flushed before every timed step (256 MiB device write); e2e steps "
                  "unflushed, weights larger than L2",
            "description": wl.description}


def _make_inputs(wl, device):
    from mixture_experts_ffn_04_gb300 import workloads as W
    return W.make_inputs(wl, seed=0, device=device)


def train_step(m, wl, inputs, args, flush, peaks, dist):
    """Training step of the routed-expert op on the same inputs: the
    train-mode forward (which also keeps the gate/up pre-activations) and the
    backward (moe_layer_backward) with a seeded output gradient, timed with
    CUDA events after an L2 flush; W warm-up steps, K timed.  None for
    workloads whose backward the library does not cover (a shared expert or
    an input RMSNorm)."""
    if wl.I_sh or wl.input_norm or getattr(wl, "weights", "act") == "mxfp8":
        return None
    from mixture_experts_ffn_04_gb300 import workloads as W
    layer = m.MoELayer(wl, inputs, train=True)
    x = inputs["x"]
    ridx, rw = inputs.get("routes_idx"), inputs.get("routes_w")
    y = torch.empty_like(x)
    dy = W.make_output_grad(wl, seed=0, device="cuda")
    dx = torch.empty_like(x)
    dtw = torch.empty((wl.T, wl.k), device="cuda")
    E, I, H = wl.E, wl.I, wl.H
    dwg = torch.empty((E, I, H), device="cuda", dtype=wl.torch_dtype)
    dwu = torch.empty_like(dwg)
    dwd = torch.empty((E, H, I), device="cuda", dtype=wl.torch_dtype)
    grads = m.grads_for(dwg, dwu, dwd)
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def step():
        flush.fill_(1)
        ev[0].record(stream)
        layer.forward(x, y, ridx, rw)
        ev[1].record(stream)
        layer.backward(dy, dx, dtw, grads)
        ev[2].record(stream)
        ev[2].synchronize()
        return ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])

    for _ in range(args.warmup):
        step()
    launches = m.moe_last_launch_count()
    if dist is not None:
        dist.barrier()
    times = [step() for _ in range(args.steps)]
    st, bits = layer.device_status()
    if st != m.MOE_OK:
        raise RuntimeError("device status %d (bits %#x) in the training steps" % (st, bits))
    fwd_ms = max_over_ranks(sum(t[0] for t in times), dist) / args.steps
    bwd_ms = max_over_ranks(sum(t[1] for t in times), dist) / args.steps
    world = dist.get_world_size() if dist is not None else 1
    rows = wl.T * wl.k
    # dgrad through down 2RHI, dgrad through gate/up 4RHI, weight gradients
    # of down 2RHI and of gate/up 4RHI
    bwd_flops = 12.0 * rows * H * I
    bwd_tflops = bwd_flops / (bwd_ms / 1000.0) / 1e12
    return {
        "what": "train-mode forward + moe_layer_backward (routed experts: dx, routing-weight "
                "and expert weight gradients), seeded dy, L2 flushed before each step",
        "ms_per_step": fwd_ms + bwd_ms, "forward_ms": fwd_ms, "backward_ms": bwd_ms,
        "tokens_per_s": world * wl.T / ((fwd_ms + bwd_ms) / 1000.0),
        "backward_tflops": bwd_tflops, "backward_frac_bf16_peak": bwd_tflops / peaks["bf16"],
        "backward_launches": launches,
    }


def measure_layer(m, wl, inputs, steps, warmup, flush, peaks, dist, use_graph=True,
                  clocks=None):
    """Time moe_layer_forward on one workload: graph replays (or host launches)
    between CUDA events, each after an L2 flush; then a second pass through
    moe_layer_forward_traced for the per-stage times.  Returns the measured
    figures (max over ranks)."""
    world = dist.get_world_size() if dist is not None else 1
    layer = m.MoELayer(wl, inputs)
    x = inputs["x"]
    ridx, rw = inputs.get("routes_idx"), inputs.get("routes_w")
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    nst = len(m.STAGES)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)]
    for e in evs:
        e.record(stream)   # materialise the CUDA events
    torch.cuda.synchronize()
    for _ in range(warmup):
        flush.fill_(1)
        layer.forward(x, y, ridx, rw)
    torch.cuda.synchronize()
    st, bits = layer.device_status()
    if st != m.MOE_OK:
        raise RuntimeError("device status %d (bits %#x) after warm-up" % (st, bits))
    launches_per_step = m.moe_last_launch_count()

    # A timed step = L2 flush (untimed), then moe_layer_forward between two
    # CUDA events.  With a graph the forward is captured once and replayed, so
    # the device never waits on host-side launch work; the kernels are the
    # same.  Stage times come from a second pass of the same steps through
    # moe_layer_forward_traced (events between stages, which also separate
    # the stages' launches).
    graph = graph_traced = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            m.moe_layer_forward(layer.shape, layer.weights, x, ridx, rw, y, layer.ws)
        graph_traced = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_traced):
            flush.fill_(1)
            m.moe_layer_forward_traced(layer.shape, layer.weights, x, ridx, rw, y, layer.ws,
                                       evs)
        for _ in range(warmup):
            flush.fill_(1)
            graph.replay()
            graph_traced.replay()
        torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def one_step():
        flush.fill_(1)
        ev0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            m.moe_layer_forward(layer.shape, layer.weights, x, ridx, rw, y, layer.ws, stream)
        ev1.record(stream)
        ev1.synchronize()
        return ev0.elapsed_time(ev1)

    def one_traced_step():
        if graph_traced is not None:
            graph_traced.replay()
        else:
            flush.fill_(1)
            m.moe_layer_forward_traced(layer.shape, layer.weights, x, ridx, rw, y, layer.ws,
                                       evs, stream)
        evs[nst].synchronize()
        return [evs[s].elapsed_time(evs[s + 1]) for s in range(nst)]

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
        time.sleep(0.05)   # let the sampler start
    t_wall = time.perf_counter()
    step_ms = [one_step() for _ in range(steps)]
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if dist is not None:
        dist.barrier()
    clk = clocks.stop() if clocks is not None else None
    st, bits = layer.device_status()
    if st != m.MOE_OK:
        raise RuntimeError("device status %d (bits %#x) in the timed region" % (st, bits))
    per_stage = [one_traced_step() for _ in range(steps)]
    stage_ms = [max_over_ranks(statistics.mean(p[s] for p in per_stage), dist)
                for s in range(nst)]
    ms_per_step = max_over_ranks(sum(step_ms), dist) / steps
    stage = dict(zip(m.STAGES, stage_ms))

    counts = layer.views()["counts"].cpu().numpy()
    alg = algorithmic(wl, counts)
    gu_ms, dn_ms, sh_ms = stage["gate_up"], stage["down"], stage["shared"]
    gemm_ms = gu_ms + dn_ms + sh_ms
    gemm_tflops = alg["gemm_flops"] / (gemm_ms / 1000.0) / 1e12
    layer_roof_ms = 1000.0 * max(alg["layer_flops"] / (peaks["bf16"] * 1e12),
                                 alg["layer_bytes"] / (peaks["hbm"] * 1e9))
    rpc_ms = stage["route"] + stage["permute"] + stage["combine"]
    rpc_bytes = alg["route_bytes"] + alg["permute_bytes"] + alg["combine_bytes"]
    rpc_floor_ms = 1000.0 * rpc_bytes / (peaks["hbm"] * 1e9)
    out = {
        "value": replica_throughput(world, wl.T, ms_per_step), "unit": "tokens/s",
        "ms_per_step": ms_per_step, "cuda_graph": graph is not None,
        "grouped_gemm_tflops": gemm_tflops,
        "grouped_gemm_frac_bf16_peak": gemm_tflops / peaks["bf16"],
        # the same against the sustained bf16 peak (a cuBLAS GEMM looped for
        # seconds under the power cap), the reference for kernels timed
        # inside a long step
        "grouped_gemm_frac_bf16_sustained": gemm_tflops / peaks["bf16_sustained"],
        "layer_roofline_frac": layer_roof_ms / ms_per_step,
        "rpc_frac_hbm": rpc_floor_ms / rpc_ms if rpc_ms > 0 else None,
        "rpc": {"ms": rpc_ms, "algorithmic_bytes": rpc_bytes, "floor_ms": rpc_floor_ms,
                "achieved_gbs": rpc_bytes / (rpc_ms / 1000.0) / 1e9 if rpc_ms > 0 else None,
                "frac_nominal_hbm": (rpc_bytes / (rpc_ms / 1000.0) / 1e9 / NOMINAL_HBM_GBS
                                     if rpc_ms > 0 else None),
                "route_bytes": alg["route_bytes"], "permute_bytes": alg["permute_bytes"],
                "combine_bytes": alg["combine_bytes"],
                "what": "route (router GEMM + top-k) + permute + combine stage times "
                        "against their algorithmic bytes at the measured copy bandwidth"},
        "stage_ms": stage,
        "gpu_launches_per_step": launches_per_step,
        "wall_s_timed_region": t_wall,
        "experts_touched": alg["touched"],
        "clocks": clk,
    }
    return out, layer, alg


def gate_up_roofline(wl, alg, gu_ms, peaks):
    """Roofline of the dominant kernel, the gate/up grouped GEMM + SwiGLU."""
    t_flop = alg["gu_flops"] / (peaks["bf16"] * 1e12)
    t_byte = alg["gu_bytes"] / (peaks["hbm"] * 1e9)
    if t_flop >= t_byte:
        ach = alg["gu_flops"] / (gu_ms / 1000.0) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16"]}
    else:
        ach = alg["gu_bytes"] / (gu_ms / 1000.0) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm"], "unit": "GB/s",
                "frac": ach / peaks["hbm"], "frac_nominal": ach / NOMINAL_HBM_GBS}
    tr = NCU_TRAFFIC.get(wl.name)
    roof["kernel"] = gate_up_kernel_name(wl)
    engine = roof["kernel"].split(" ")[0]
    roof["traffic"] = (tr["bytes"] if tr and tr.get("kernel_hash") == _kernel_hash(engine)
                       else None)
    roof["kernel_ms"] = gu_ms
    roof["peak_source"] = peaks["source"] + (" burst" if roof["bound"] == "tensor" else " copy")
    roof["algorithmic_per_launch"] = (alg["gu_flops"] if roof["bound"] == "tensor"
                                      else alg["gu_bytes"])
    roof["algorithmic_flops"] = alg["gu_flops"]
    roof["algorithmic_bytes"] = alg["gu_bytes"]
    return roof


def gate_up_kernel_name(wl):
    """The engine the library picks for the routed gate/up call (T*k rows)."""
    if wl.T * wl.k <= 4:
        return "skinny_kernel (decode engine: gate/up + SwiGLU)"
    if wl.weights == "mxfp8" and wl.H % 128 == 0:
        return "tc_mx_kernel (gate/up grouped GEMM + SwiGLU, MXFP8 weights)"
    if wl.dtype == "f32":
        return "simt_gemm_kernel (gate/up grouped GEMM + SwiGLU, fp32 on the CUDA cores)"
    rows = wl.T * wl.k
    if rows >= 512 and (rows // wl.E >= 1024 or wl.H >= 3072):
        return "tc2_gemm_kernel (gate/up grouped GEMM + SwiGLU on SM pairs)"
    return "tc_gemm_kernel (gate/up grouped GEMM + SwiGLU)"


def e2e_measure(m, layer, wl, inputs, steps, warmup, world):
    """End to end through the public API, host buffers.  Every step copies its
    tokens in from pinned host memory, runs moe_layer_forward on them and
    copies its output back, on three streams so that step i+1's upload and
    step i-1's download overlap step i's forward (double-buffered device and
    host tensors; the forwards run in order on one stream and share the
    workspace).  No L2 flush here: the expert weights are larger than L2."""
    x = inputs["x"]
    ridx, rw = inputs.get("routes_idx"), inputs.get("routes_w")
    x_host = x.cpu().pin_memory()
    y_host = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    ridx_h = ridx.cpu().pin_memory() if ridx is not None else None
    rw_h = rw.cpu().pin_memory() if rw is not None else None
    xd = [torch.empty_like(x) for _ in range(2)]
    yd = [torch.empty_like(x) for _ in range(2)]
    rid = [torch.empty_like(ridx) for _ in range(2)] if ridx is not None else [None, None]
    rwd = [torch.empty_like(rw) for _ in range(2)] if rw is not None else [None, None]
    stream = torch.cuda.current_stream()
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_cmp + ev_out:
        e.record(stream)
    torch.cuda.synchronize()

    def e2e_steps(n):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_cmp[b])          # the forward that read xd[b] is done
                xd[b].copy_(x_host, non_blocking=True)
                if rid[b] is not None:
                    rid[b].copy_(ridx_h, non_blocking=True)
                    rwd[b].copy_(rw_h, non_blocking=True)
                ev_in[b].record(s_in)
            s_cmp.wait_event(ev_in[b])
            s_cmp.wait_event(ev_out[b])             # yd[b]'s last download is done
            layer.forward(xd[b], yd[b], rid[b], rwd[b], stream=s_cmp)
            ev_cmp[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[b])
                y_host[b].copy_(yd[b], non_blocking=True)
                ev_out[b].record(s_out)

    e2e_steps(warmup)
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(s_in)
    e2e_steps(steps)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    e_end.record(s_out)
    e_end.synchronize()
    e2e_ms = e_start.elapsed_time(e_end) / steps
    h2d = x.numel() * x.element_size() + (0 if ridx is None else
                                            ridx.numel() * 4 + rw.numel() * 4)
    d2h = x.numel() * x.element_size()
    return {"value": world * wl.T / (e2e_ms / 1000.0), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure the named workload only")
    ap.add_argument("--weights", default="act", choices=["act", "mxfp8"],
                    help="expert weights in the activation type or packed MXFP8 (no CPU "
                         "baseline or training step with MXFP8)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every step from the host instead of replaying a CUDA graph")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from mixture_experts_ffn_04_gb300 import workloads as W
    wl = W.get(args.workload)
    if args.weights == "mxfp8":
        import dataclasses
        wl = dataclasses.replace(wl, weights="mxfp8")
        args.no_cpu_baseline = True
    dist, rank, world = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if torch.cuda.is_available():
        torch.cuda.set_device(local)

    if args.impl == "reference":
        run_reference(args, wl, rank, world)
        if dist is not None:
            dist.barrier()
        return

    import mixture_experts_ffn_04_gb300 as m
    m.lib()
    peaks = _peaks()
    inputs = _make_inputs(wl, "cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    res, layer, alg = measure_layer(m, wl, inputs, args.steps, args.warmup, flush, peaks, dist,
                                    use_graph=not args.no_graph, clocks=Clocks(local))
    e2e = e2e_measure(m, layer, wl, inputs, args.steps, args.warmup, world)
    roof = gate_up_roofline(wl, alg, res["stage_ms"]["gate_up"], peaks)
    train = train_step(m, wl, inputs, args, flush, peaks, dist)

    line = {
        "metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
        "config": _config(wl),
        "cuda_graph": res["cuda_graph"],
        "grouped_gemm_tflops": res["grouped_gemm_tflops"],
        "grouped_gemm_frac_bf16_peak": res["grouped_gemm_frac_bf16_peak"],
        "grouped_gemm_frac_bf16_sustained": res["grouped_gemm_frac_bf16_sustained"],
        "layer_roofline_frac": res["layer_roofline_frac"],
        "rpc_frac_hbm": res["rpc_frac_hbm"],
        "rpc": res["rpc"],
        "stage_ms": res["stage_ms"],
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": res["gpu_launches_per_step"] * args.steps,
        "clocks": res["clocks"],
        "wall_s_timed_region": res["wall_s_timed_region"],
        "experts_touched": res["experts_touched"],
        "peaks": {"hbm_gbs": peaks["hbm"], "bf16_tflops": peaks["bf16"],
                  "bf16_tflops_sustained": peaks["bf16_sustained"], "source": peaks["source"]},
    }
    if train is not None:
        line["train_step"] = train
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import oracle as O
        O.load()
        threads = os.cpu_count() or 1
        smp = OracleSample(wl, inputs, 10.0, threads)
        dt = smp.run()
        line["cpu_baseline"] = {"value": smp.n / dt, "unit": "tokens/s", "cores": threads,
                                "kind": "oracle", "sample": smp.describe(dt)}
        del smp
    del layer, inputs
    torch.cuda.empty_cache()

    if not args.no_per_config and args.weights == "act" and args.workload == DEFAULT_WORKLOAD:
        per = {}
        for name in PER_CONFIG:
            w2 = W.get(name)
            inp2 = _make_inputs(w2, "cuda")
            r2, l2, a2 = measure_layer(m, w2, inp2, min(args.steps, 10), 3, flush, peaks, dist,
                                       use_graph=not args.no_graph)
            r2.pop("clocks", None)
            r2["roofline"] = gate_up_roofline(w2, a2, r2["stage_ms"]["gate_up"], peaks)
            r2["steps"] = min(args.steps, 10)
            per[name] = r2
            del l2, inp2
            torch.cuda.empty_cache()
        line["per_config"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()


if __name__ == "__main__":
    main()
