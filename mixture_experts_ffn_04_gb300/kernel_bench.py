"""Time one grouped-GEMM step of the layer, or one training step, on synthetic
seeded operands (CUDA events, L2 flushed before each timed launch), e.g. to
reproduce a profile of one kernel at chosen sizes:

    python -m mixture_experts_ffn_04_gb300.kernel_bench --op wgrad \\
        --groups 64 --rows-per-group 256 --hidden 7168 --inter 2048

ops: gate_up (forward grouped GEMM + SwiGLU), down (forward), dgrad_down
(dgrad through down with the SwiGLU derivative), dgrad_gate_up, wgrad
(the down projection's weight gradient), layer (moe_layer_forward of a named
workload, --workload, launched from the host: every kernel of the forward in
order, for launch lists and per-kernel DRAM counters), train_step (train-mode
forward and backward of a named workload).  Group sizes alternate between
rows-per-group +- 13 rows, so every group ends inside a 64-row block.
Prints one JSON line; exits non-zero if the device status word is set."""
from __future__ import annotations

import argparse
import json
import statistics
import sys

import torch

import mixture_experts_ffn_04_gb300 as m
from mixture_experts_ffn_04_gb300 import workloads as W


def _time(fn, flush, steps, warmup):
    for _ in range(warmup):
        flush.fill_(1)
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = []
    for _ in range(steps):
        flush.fill_(1)
        a.record()
        fn()
        b.record()
        b.synchronize()
        out.append(a.elapsed_time(b) * 1e3)
    return statistics.median(out)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", required=True,
                    choices=["gate_up", "down", "dgrad_down", "dgrad_gate_up", "wgrad",
                             "layer", "train_step"])
    ap.add_argument("--groups", type=int, default=64)
    ap.add_argument("--rows-per-group", type=int, default=256)
    ap.add_argument("--hidden", type=int, default=7168)
    ap.add_argument("--inter", type=int, default=2048)
    ap.add_argument("--workload", default="qwen3-30b-a3b-shape-T4096")
    ap.add_argument("--weights", default="act", choices=["act", "mxfp8"],
                    help="gate_up / down: expert weights packed as MXFP8 (moe_quantize_mxfp8); "
                         "layer: the workload's expert weights drawn as packed MXFP8")
    ap.add_argument("--engine", type=int, default=0,
                    help="grouped-GEMM engine forced for the run (moe_testing_set_gemm_engine; "
                         "0 = the library's choice)")
    ap.add_argument("--fork-sms", type=int, default=0,
                    help="layer: SMs the shared MLP may take on its forked stream at decode "
                         "sizes (moe_testing_set_fork_sms; 0 = the library's choice, -1 = all)")
    ap.add_argument("--graph", action="store_true",
                    help="layer: time the replay of one forward captured in a CUDA graph "
                         "(as the benchmark does) instead of the launches from the host")
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=2)
    a = ap.parse_args(argv)
    torch.cuda.set_device(0)
    m.moe_testing_set_gemm_engine(a.engine)
    m.moe_testing_set_fork_sms(a.fork_sms)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(0)

    if a.op == "layer":
        wl = W.get(a.workload)
        if a.weights == "mxfp8":
            import dataclasses
            wl = dataclasses.replace(wl, weights="mxfp8")
        dev = W.make_inputs(wl, seed=0, device="cuda")
        layer = m.MoELayer(wl, dev)
        x = dev["x"]
        y = torch.empty_like(x)
        fwd = lambda: layer.forward(x, y, dev.get("routes_idx"), dev.get("routes_w"))
        if a.graph:
            fwd()                      # first call outside the capture (side stream, tables)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                fwd()
            us = _time(graph.replay, flush, a.steps, a.warmup)
        else:
            us = _time(fwd, flush, a.steps, a.warmup)
        st = layer.device_status()[0]
        print(json.dumps({"op": a.op, "workload": wl.name, "weights": a.weights,
                          "engine": a.engine, "fork_sms": a.fork_sms, "graph": a.graph,
                          "us": us,
                          "launches": m.moe_last_launch_count(), "status": st}))
        return 0 if st == m.MOE_OK else 1

    if a.op == "train_step":
        wl = W.get(a.workload)
        dev = W.make_inputs(wl, seed=0, device="cuda")
        layer = m.MoELayer(wl, dev, train=True)
        x = dev["x"]
        y = torch.empty_like(x)
        dy = W.make_output_grad(wl, seed=0, device="cuda")
        dx = torch.empty_like(x)
        dtw = torch.empty((wl.T, wl.k), device="cuda")
        dwg = torch.empty((wl.E, wl.I, wl.H), device="cuda", dtype=wl.torch_dtype)
        dwu = torch.empty_like(dwg)
        dwd = torch.empty((wl.E, wl.H, wl.I), device="cuda", dtype=wl.torch_dtype)
        grads = m.grads_for(dwg, dwu, dwd)

        def fn():
            layer.forward(x, y, dev.get("routes_idx"), dev.get("routes_w"))
            layer.backward(dy, dx, dtw, grads)
        us = _time(fn, flush, a.steps, a.warmup)
        st = layer.device_status()[0]
        print(json.dumps({"op": a.op, "workload": wl.name, "us": us, "status": st}))
        return 0 if st == m.MOE_OK else 1

    E, H, I = a.groups, a.hidden, a.inter
    counts = torch.full((E,), a.rows_per_group, dtype=torch.int64)
    counts[::2] += 13
    counts[1::2] -= 13
    counts.clamp_(min=0)
    offsets = torch.cat([torch.zeros(1, dtype=torch.int64), counts.cumsum(0)]).to(torch.int32).cuda()
    R = int(counts.sum())
    wl = W.small(W.DEEPSEEK_V3, T=max(1, R // 8), H=H, I=I, E=E, k=8, I_sh=0)
    mx = a.weights == "mxfp8" and a.op in ("gate_up", "down")
    if mx:
        import dataclasses
        wl = dataclasses.replace(wl, weights="mxfp8")
    s = m.shape_for(wl)
    ws = m.alloc_workspace(s, full=False)
    rnd = lambda *shape, sc=0.1: (torch.randn(*shape, generator=g, device="cuda") * sc).bfloat16()
    if a.op in ("gate_up", "dgrad_gate_up"):
        wg, wu = rnd(E, I, H, sc=0.02), rnd(E, I, H, sc=0.02)
    if a.op in ("down", "dgrad_down"):
        wd = rnd(E, H, I, sc=0.02)
    gs, ds = I * H, H * I   # expert strides (elements; bytes when packed)
    if mx and a.op == "gate_up":
        wg, wu = m.mxfp8_pack(wg), m.mxfp8_pack(wu)
        gs = wg.shape[1]
    if mx and a.op == "down":
        wd = m.mxfp8_pack(wd)
        ds = wd.shape[1]
    if a.op == "gate_up":
        xp, h = rnd(R, H), torch.empty(R, I, device="cuda", dtype=torch.bfloat16)
        fn = lambda: m.moe_grouped_swiglu(s, xp, wg, wu, gs, offsets, E, R, I, h, ws)
        flops = 4.0 * R * H * I
    elif a.op == "down":
        h, yp = rnd(R, I), torch.empty(R, H, device="cuda", dtype=torch.bfloat16)
        fn = lambda: m.moe_grouped_down(s, h, wd, ds, offsets, E, R, I, yp, ws)
        flops = 2.0 * R * H * I
    elif a.op == "dgrad_down":
        gf, fc1 = rnd(R, H), rnd(R, 2 * I, sc=1.0)
        dfc1 = torch.empty(R, 2 * I, device="cuda", dtype=torch.bfloat16)
        fn = lambda: m.moe_grouped_down_dgrad(s, gf, wd, H * I, fc1, offsets, E, R, I, dfc1, ws)
        flops = 2.0 * R * H * I
    elif a.op == "dgrad_gate_up":
        dfc1, dxp = rnd(R, 2 * I), torch.empty(R, H, device="cuda", dtype=torch.bfloat16)
        fn = lambda: m.moe_grouped_gate_up_dgrad(s, dfc1, wg, wu, I * H, offsets, E, R, I, dxp, ws)
        flops = 4.0 * R * H * I
    else:
        gf, h = rnd(R, H), rnd(R, I)
        dw = torch.empty(E, H, I, device="cuda", dtype=torch.bfloat16)
        fn = lambda: m.moe_grouped_wgrad(s, gf, H, h, I, offsets, E, R, H, I, dw, H * I, ws)
        flops = 2.0 * R * H * I
    us = _time(fn, flush, a.steps, a.warmup)
    st = m.moe_get_device_status(ws)[0]
    print(json.dumps({"op": a.op, "engine": a.engine, "weights": a.weights, "groups": E,
                      "rows": R, "hidden": H,
                      "inter": I, "us": us,
                      "tflops": flops / us / 1e6, "status": st}))
    return 0 if st == m.MOE_OK else 1


if __name__ == "__main__":
    sys.exit(main())
