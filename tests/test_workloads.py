"""The seeded input recipe (workloads.py) draws what it states: determinism
per (seed, tensor name), the value distributions of each tensor, the direct
routes of the adversarial workloads (all-to-one with weight 1/k; Zipf(1.2)
over 64 experts, whose most and least popular experts are drawn with
probability about 0.29 and 0.002, duplicates allowed, weights summing to 1),
and the packed MXFP8 weights (finite normal e4m3 codes, scales near the
target standard deviation).  CPU only; reduced widths keep it fast."""
import dataclasses
import math

import numpy as np
import pytest
import torch

from mixture_experts_ffn_04_gb300 import workloads as W


def _std(t):
    return float(t.double().std())


def test_same_seed_same_values_other_seed_or_name_other_values():
    wl = W.small(W.QWEN2_MOE, T=64, H=256, I=128, I_sh=256, E=8, k=2)
    a = W.make_inputs(wl, seed=0)
    b = W.make_inputs(wl, seed=0)
    c = W.make_inputs(wl, seed=1)
    for key in ("x", "w_router", "w_gate", "w_up", "w_down", "sh_gate", "sh_up", "sh_down"):
        assert torch.equal(a[key], b[key]), key
        assert not torch.equal(a[key], c[key]), key
    # one stream per tensor name: gate and up weights are not the same draw
    g = a["w_gate"].double().flatten()
    u = a["w_up"].double().flatten()
    assert abs(float(torch.corrcoef(torch.stack([g, u]))[0, 1])) < 0.02


def test_value_distributions():
    H, I, I_sh = 512, 256, 384
    wl = W.small(W.QWEN2_MOE, T=512, H=H, I=I, I_sh=I_sh, E=16, k=4)
    d = W.make_inputs(wl, seed=0)
    assert abs(_std(d["x"]) - 1.0) < 0.02 and abs(float(d["x"].double().mean())) < 0.01
    assert abs(_std(d["w_gate"]) * math.sqrt(H) - 1.0) < 0.02
    assert abs(_std(d["w_up"]) * math.sqrt(H) - 1.0) < 0.02
    assert abs(_std(d["w_down"]) * math.sqrt(I) - 1.0) < 0.02
    assert abs(_std(d["sh_gate"]) * math.sqrt(H) - 1.0) < 0.02
    assert abs(_std(d["sh_down"]) * math.sqrt(I_sh) - 1.0) < 0.02
    # router rows N(0, 0.02); the shared-gate row (last) N(0, 1/sqrt(H))
    wr = d["w_router"]
    assert wr.shape == (wl.E + 1, H)
    assert abs(_std(wr[:-1]) / 0.02 - 1.0) < 0.03
    assert abs(_std(wr[-1]) * math.sqrt(H) - 1.0) < 0.15
    # a workload without a stated router std: 1/sqrt(H)
    t = W.make_inputs(W.small(W.TINY_F32, T=64), seed=0)
    assert abs(_std(t["w_router"]) * math.sqrt(W.TINY_F32.H) - 1.0) < 0.05
    assert t["x"].dtype == torch.float32 and d["x"].dtype == torch.bfloat16


def test_input_norm_weight_near_one():
    wl = W.small(W.GEMMA4_26B_A4B, T=16, H=4096, I=64, E=4, k=2)
    d = W.make_inputs(wl, seed=0, with_experts=False)
    nw = d["norm_weight"].double()
    assert abs(float(nw.mean()) - 1.0) < 0.01 and abs(float(nw.std()) - 0.1) < 0.01


def test_all_to_one_routes():
    wl = W.small(W.ADV_E0, T=100, H=64, I=64, I_sh=64)
    d = W.make_inputs(wl, seed=0, with_experts=False)
    assert d["w_router"] is None
    assert (d["routes_idx"] == 0).all()
    assert torch.equal(d["routes_w"], torch.full((100, wl.k), 1.0 / wl.k, dtype=torch.float32))


def test_zipf_routes():
    wl = W.small(W.ADV_ZIPF, T=16384, H=64, I=64, I_sh=64)
    assert (wl.E, wl.k, wl.zipf_s) == (64, 6, 1.2)
    d = W.make_inputs(wl, seed=0, with_experts=False)
    idx = d["routes_idx"].numpy()
    freq = np.bincount(idx.reshape(-1), minlength=64) / idx.size
    assert abs(freq[0] - 0.29) < 0.01
    assert abs(freq[63] - 0.002) < 0.001
    assert (np.diff(freq[:8]) < 0).all()       # the head is monotone in the rank
    dup = np.array([len(set(r)) < wl.k for r in idx])
    assert dup.mean() > 0.5                    # duplicates are allowed and common
    w = d["routes_w"].double().numpy()
    assert (w > 0).all()
    assert np.abs(w.sum(axis=1) - 1.0).max() < 1e-6


def test_mxfp8_packed_weights():
    H, I = 256, 128
    wl = dataclasses.replace(W.small(W.QWEN2_MOE, T=8, H=H, I=I, I_sh=128, E=4, k=2),
                             weights="mxfp8")
    d = W.make_inputs(wl, seed=0)
    wg = d["w_gate"]
    assert wg.dtype == torch.uint8 and wg.shape == (4, I * H * 9 // 8)
    codes = wg[:, :I * H].to(torch.int32)
    exp_field = (codes >> 3) & 0xF
    assert int(exp_field.min()) >= 4 and int(exp_field.max()) <= 9   # normal, finite
    scales = wg[:, I * H:].to(torch.int32)
    base = 127 + int(round(math.log2((1.0 / math.sqrt(H)) / 4.0)))
    assert int(scales.min()) >= base - 1 and int(scales.max()) <= base + 1
    # dequantised values: e4m3 (torch's decode) times 2^(scale - 127), per block of 8
    vals = codes.to(torch.uint8).view(torch.float8_e4m3fn).double().reshape(4, I, H // 8, 8)
    vals = vals * torch.exp2(scales.double() - 127.0).reshape(4, I, H // 8, 1)
    assert 0.7 < float(vals.std()) * math.sqrt(H) < 1.5
