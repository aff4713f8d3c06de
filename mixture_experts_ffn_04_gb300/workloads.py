"""Workload shapes and seeded synthetic inputs for the MoE FFN forward pass.

This module is the only code that both the CUDA path and the fp64 oracle
consume: it draws random tensors and nothing else.  It contains none of the
layer's arithmetic (no routing, no activation, no reduction).

Value recipe (per workload):
  x ~ N(0, 1); expert gate/up ~ N(0, 1/sqrt(H)); expert down ~ N(0, 1/sqrt(I));
  shared gate/up ~ N(0, 1/sqrt(H)); shared down ~ N(0, 1/sqrt(I_sh));
  router rows ~ N(0, router_std) (1/sqrt(H) when unset); the Qwen2-MoE-style
  shared-gate weight (router row E) ~ N(0, 1/sqrt(H)), so its logit is ~N(0, 1).
  Input RMSNorm weight (workloads with input preparation) ~ 1 + N(0, 0.1^2).
  Direct routes: "all_to_e0" sends every slot to expert 0 with weight 1/k;
  "zipf" draws each slot independently with P(e) proportional to (e+1)^-s
  (duplicates allowed) and per-slot weights U(0,1) normalised to sum 1.

Randomness: one stream per tensor, keyed by (seed, tensor name).  On the host
the stream is numpy's PCG64; on a CUDA device it is torch's Philox generator
(used for the multi-GB weight sets).  A test draws all inputs of one case on
one device and hands the same values to both sides.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Dict, Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    I_sh: int = 0
    shared_gate: bool = False
    norm_topk: bool = True
    dtype: str = "bf16"          # "f32" or "bf16"
    routing: str = "router"      # "router", "all_to_e0" or "zipf"
    router_std: Optional[float] = None
    zipf_s: float = 1.2
    input_norm: bool = False     # input RMSNorm before the router and experts
    residual: bool = False       # y = x + MoE(x_norm)
    norm_eps: float = 1e-6
    weights: str = "act"         # expert weights: "act" (activation type) or "mxfp8" (packed)
    description: str = ""

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def esize(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def with_tokens(self, T: int) -> "Workload":
        return dataclasses.replace(self, T=T, name="%s-T%d" % (self.name.split("-T")[0], T))

    def flops(self) -> float:
        """Algorithmic FLOPs of one forward pass (multiply-add = 2)."""
        f = 6.0 * self.T * self.k * self.H * self.I + 6.0 * self.T * self.H * self.I_sh
        if self.routing == "router":
            f += 2.0 * self.T * self.H * (self.E + (1 if self.shared_gate else 0))
        return f


# The five workloads; names say what they are and give their sizes.
WORKLOADS: Dict[str, Workload] = {}


def _add(w: Workload):
    WORKLOADS[w.name] = w
    return w


TINY_F32 = _add(Workload(
    "tiny-f32-T64", T=64, H=256, E=8, k=2, I=128, dtype="f32", norm_topk=True,
    description="tiny fp32 layer: T=64, H=256, E=8, k=2, I=128, no shared expert"))
QWEN3_30B_A3B = _add(Workload(
    "qwen3-30b-a3b-shape-T4096", T=4096, H=2048, E=128, k=8, I=768, norm_topk=True,
    router_std=0.02,
    description="Qwen3-30B-A3B-shaped prefill: T=4096, H=2048, E=128, k=8, I=768, "
                "no shared expert, renormalised top-k softmax"))
DEEPSEEK_V3 = _add(Workload(
    "deepseek-v3-shape-T8192", T=8192, H=7168, E=256, k=8, I=2048, I_sh=2048,
    norm_topk=False, router_std=0.02,
    description="DeepSeek-V3-shaped prefill: T=8192, H=7168, E=256, k=8, I=2048, "
                "one ungated shared expert of width 2048, top-k of the full softmax"))
QWEN2_MOE = _add(Workload(
    "qwen2-moe-shape-T2048", T=2048, H=3584, E=60, k=4, I=2560, I_sh=20480,
    shared_gate=True, norm_topk=False, router_std=0.02,
    description="Qwen2-MoE-shaped: T=2048 (also T=64, 8, 1), H=3584, E=60, k=4, "
                "I=2560, shared MLP width 20480 with a sigmoid gate"))
for _t in (64, 8, 1):
    _add(QWEN2_MOE.with_tokens(_t))
ADV_E0 = _add(Workload(
    "adversarial-all-e0-T128", T=128, H=4096, E=64, k=6, I=1408, I_sh=2816,
    routing="all_to_e0",
    description="adversarial direct routes: every slot to expert 0, weight 1/6; "
                "H=4096, E=64, k=6, I=1408, two shared experts fused to 2816"))
_add(ADV_E0.with_tokens(16384))
ADV_ZIPF = _add(Workload(
    "adversarial-zipf-T128", T=128, H=4096, E=64, k=6, I=1408, I_sh=2816,
    routing="zipf",
    description="adversarial direct routes: Zipf(1.2) expert popularity, duplicates "
                "allowed; H=4096, E=64, k=6, I=1408, shared width 2816"))
_add(ADV_ZIPF.with_tokens(16384))
GEMMA4_26B_A4B = _add(Workload(
    "gemma4-26b-a4b-shape-T512", T=512, H=2816, E=128, k=8, I=704, norm_topk=False,
    router_std=0.02, input_norm=True, residual=True,
    description="Gemma-4-26B-A4B-shaped prefill with the sublayer's input preparation: "
                "T=512 (also 4096), H=2816, E=128, k=8, I=704, no shared expert, input "
                "RMSNorm (eps 1e-6) before routing and experts, residual added after "
                "the combine, top-k of the full softmax"))
_add(GEMMA4_26B_A4B.with_tokens(4096))


def get(name: str) -> Workload:
    return WORKLOADS[name]


def small(w: Workload, T: Optional[int] = None, H: Optional[int] = None,
          I: Optional[int] = None, I_sh: Optional[int] = None, E: Optional[int] = None,
          k: Optional[int] = None) -> Workload:
    """A reduced copy of a workload (same routing style, gate and dtype)."""
    d = dict(T=T or w.T, H=H or w.H, I=I or w.I, E=E or w.E, k=k or w.k)
    d["I_sh"] = w.I_sh if I_sh is None else I_sh
    if w.I_sh == 0:
        d["I_sh"] = 0
    name = "%s-reduced-T%d-H%d-E%d-k%d-I%d-Ish%d" % (w.name.split("-T")[0], d["T"], d["H"],
                                                     d["E"], d["k"], d["I"], d["I_sh"])
    return dataclasses.replace(w, name=name, **d)


# ---------------------------------------------------------------------------
# seeded streams
# ---------------------------------------------------------------------------
def _key(seed: int, name: str) -> int:
    return (int(seed) * 0x9E3779B1 + zlib.crc32(name.encode())) & 0x7FFFFFFFFFFFFFFF


def _normal(seed: int, name: str, shape, std: float, dtype, device) -> torch.Tensor:
    n = int(np.prod(shape))
    if torch.device(device).type == "cpu":
        rng = np.random.Generator(np.random.PCG64(_key(seed, name)))
        a = rng.standard_normal(n, dtype=np.float32)
        a *= np.float32(std)
        return torch.from_numpy(a).reshape(shape).to(dtype)
    g = torch.Generator(device=device)
    g.manual_seed(_key(seed, name))
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    chunk = 1 << 28
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        tmp = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        tmp.mul_(std)
        flat[s:e].copy_(tmp)
        del tmp
    return out


def _routes(w: Workload, seed: int):
    T, k, E = w.T, w.k, w.E
    if w.routing == "all_to_e0":
        idx = np.zeros((T, k), dtype=np.int32)
        wt = np.full((T, k), 1.0 / k, dtype=np.float32)
        return torch.from_numpy(idx), torch.from_numpy(wt)
    rng = np.random.Generator(np.random.PCG64(_key(seed, "routes")))
    p = (np.arange(1, E + 1, dtype=np.float64)) ** (-w.zipf_s)
    p /= p.sum()
    idx = rng.choice(E, size=(T, k), p=p).astype(np.int32)
    u = rng.uniform(0.0, 1.0, size=(T, k)) + 1e-3
    wt = (u / u.sum(axis=1, keepdims=True)).astype(np.float32)
    return torch.from_numpy(idx), torch.from_numpy(wt)


def _mxfp8_packed(seed: int, name: str, batch: int, N: int, K: int, std: float,
                  device) -> torch.Tensor:
    """Seeded packed MXFP8 matrices [batch, N*K*9/8] drawn directly as codes and
    scales (no quantisation): e4m3 codes with a random sign, exponent field
    4..9 and mantissa 0..7 (magnitudes 0.125 .. 7.5), and per-block scale
    bytes within one of 127 + round(log2(std / 4)), so the values have about
    the standard deviation `std`."""
    g = torch.Generator(device=device)
    g.manual_seed(_key(seed, name))
    nk = N * K
    out = torch.empty((batch, nk // 8 * 9), dtype=torch.uint8, device=device)
    for b in range(batch):
        sign = torch.randint(0, 2, (nk,), generator=g, device=device, dtype=torch.int32)
        ex = torch.randint(4, 10, (nk,), generator=g, device=device, dtype=torch.int32)
        man = torch.randint(0, 8, (nk,), generator=g, device=device, dtype=torch.int32)
        out[b, :nk] = ((sign << 7) | (ex << 3) | man).to(torch.uint8)
        base = 127 + int(round(math.log2(std / 4.0)))
        sc = torch.randint(-1, 2, (nk // 8,), generator=g, device=device, dtype=torch.int32) + base
        out[b, nk:] = sc.to(torch.uint8)
    return out


def make_output_grad(w: Workload, seed: int = 0, device="cpu") -> torch.Tensor:
    """dy = dL/dy [T, H] for the backward: standard normal in the activation type."""
    return _normal(seed, "dy", (w.T, w.H), 1.0, w.torch_dtype, device)


def make_inputs(w: Workload, seed: int = 0, device="cpu", with_experts: bool = True):
    """All input tensors of one workload, drawn on ``device``.

    Keys: x [T,H]; norm_weight [H] or None; w_router [E(+1),H] or None;
    w_gate, w_up [E,I,H];
    w_down [E,H,I]; sh_gate, sh_up [I_sh,H] and sh_down [H,I_sh] or None;
    routes_idx [T,k] int32 and routes_w [T,k] fp32 (direct routes) or None.
    """
    dt = w.torch_dtype
    T, H, E, k, I, I_sh = w.T, w.H, w.E, w.k, w.I, w.I_sh
    d = {}
    d["x"] = _normal(seed, "x", (T, H), 1.0, dt, device)
    if w.input_norm:
        d["norm_weight"] = (_normal(seed, "norm_weight", (H,), 0.1, torch.float32, device)
                            + 1.0).to(dt)
    else:
        d["norm_weight"] = None
    if w.routing == "router":
        std = w.router_std if w.router_std is not None else 1.0 / math.sqrt(H)
        wr = _normal(seed, "w_router", (E, H), std, dt, device)
        if w.shared_gate:
            wsg = _normal(seed, "w_shared_gate", (1, H), 1.0 / math.sqrt(H), dt, device)
            wr = torch.cat([wr, wsg], dim=0).contiguous()
        d["w_router"] = wr
        d["routes_idx"] = d["routes_w"] = None
    else:
        d["w_router"] = None
        ri, rw = _routes(w, seed)
        d["routes_idx"], d["routes_w"] = ri.to(device), rw.to(device)
    mx = w.weights == "mxfp8"
    if with_experts and mx:
        # packed MXFP8 [E, N*K*9/8] (include/moe.h, moe_weight_format)
        d["w_gate"] = _mxfp8_packed(seed, "w_gate", E, I, H, 1.0 / math.sqrt(H), device)
        d["w_up"] = _mxfp8_packed(seed, "w_up", E, I, H, 1.0 / math.sqrt(H), device)
        d["w_down"] = _mxfp8_packed(seed, "w_down", E, H, I, 1.0 / math.sqrt(I), device)
    elif with_experts:
        d["w_gate"] = _normal(seed, "w_gate", (E, I, H), 1.0 / math.sqrt(H), dt, device)
        d["w_up"] = _normal(seed, "w_up", (E, I, H), 1.0 / math.sqrt(H), dt, device)
        d["w_down"] = _normal(seed, "w_down", (E, H, I), 1.0 / math.sqrt(I), dt, device)
    if I_sh > 0 and mx:
        d["sh_gate"] = _mxfp8_packed(seed, "sh_gate", 1, I_sh, H, 1.0 / math.sqrt(H), device)[0]
        d["sh_up"] = _mxfp8_packed(seed, "sh_up", 1, I_sh, H, 1.0 / math.sqrt(H), device)[0]
        d["sh_down"] = _mxfp8_packed(seed, "sh_down", 1, H, I_sh, 1.0 / math.sqrt(I_sh), device)[0]
    elif I_sh > 0:
        d["sh_gate"] = _normal(seed, "sh_gate", (I_sh, H), 1.0 / math.sqrt(H), dt, device)
        d["sh_up"] = _normal(seed, "sh_up", (I_sh, H), 1.0 / math.sqrt(H), dt, device)
        d["sh_down"] = _normal(seed, "sh_down", (H, I_sh), 1.0 / math.sqrt(I_sh), dt, device)
    else:
        d["sh_gate"] = d["sh_up"] = d["sh_down"] = None
    return d
