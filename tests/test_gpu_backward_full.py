"""The routed-expert backward at full benchmark sizes, in the configuration
bench.py times (moe_layer_backward after a train-mode moe_layer_forward),
checked on samples the fp64 oracle computes one by one:

* dx and the routing-weight gradient of sampled tokens: a token's gradients
  depend only on its own k routed pairs, so the oracle runs on those tokens
  alone;
* the whole weight gradient of sampled experts: dW[e] depends only on the
  pairs routed to e, so the oracle runs on those pairs as one-slot tokens;
* every value of every output finite, and experts without rows exactly zero.

Routes are the oracle's own routing of the workload (Qwen3-30B-A3B shape) or
seeded Zipf routes (DeepSeek-V3 expert shape), passed to both sides."""
import dataclasses

import numpy as np
import pytest
import torch

import mixture_experts_ffn_04_gb300 as m
from mixture_experts_ffn_04_gb300 import workloads as W
from oracle import moe_backward as MB
from oracle import oracle as O

from gpu_util import TOL, rel_l2

pytestmark = pytest.mark.gpu

FULL = [
    W.QWEN3_30B_A3B,
    dataclasses.replace(W.DEEPSEEK_V3, I_sh=0, routing="zipf", zipf_s=0.6,
                        name="deepseek-v3-experts-zipf-T8192"),
]


@pytest.mark.parametrize("wl", FULL, ids=[w.name for w in FULL])
def test_full_size_backward_sampled(wl):
    dev = W.make_inputs(wl, seed=0, device="cuda")
    if wl.routing == "router":
        host = {"x": dev["x"].cpu(), "w_router": dev["w_router"].cpu(), "routes_idx": None,
                "routes_w": None, "norm_weight": None}
        r = O.route(wl, host)
        idx = r["idx"].astype(np.int32)
        wts = r["weights"].astype(np.float32)
    else:
        idx = dev["routes_idx"].cpu().numpy()
        wts = dev["routes_w"].cpu().numpy()
    dy = W.make_output_grad(wl, seed=0, device="cuda")
    wl_d = dataclasses.replace(wl, routing="zipf", shared_gate=False)
    layer = m.MoELayer(wl_d, dev, train=True)
    ridx = torch.from_numpy(idx).cuda()
    rw = torch.from_numpy(wts).cuda()
    layer.forward(dev["x"], routes_idx=ridx, routes_w=rw)
    E, I, H, T, k = wl.E, wl.I, wl.H, wl.T, wl.k
    nan = float("nan")
    dwg = torch.full((E, I, H), nan, device="cuda", dtype=torch.bfloat16)
    dwu = torch.full((E, I, H), nan, device="cuda", dtype=torch.bfloat16)
    dwd = torch.full((E, H, I), nan, device="cuda", dtype=torch.bfloat16)
    dx = torch.full_like(dev["x"], float("nan"))
    dtw = torch.full((T, k), float("nan"), device="cuda")
    layer.backward(dy, dx, dtw, m.grads_for(dwg, dwu, dwd))
    st, bits = layer.device_status()
    assert st == m.MOE_OK, (st, bits)
    for t in (dx, dtw, dwg, dwu, dwd):
        assert bool(torch.isfinite(t.float()).all())
    counts = np.bincount(idx.reshape(-1), minlength=E)
    for e in np.nonzero(counts == 0)[0][:4]:
        assert bool((dwg[e] == 0).all() and (dwu[e] == 0).all() and (dwd[e] == 0).all())
    tol = TOL["bf16"]
    rng = np.random.default_rng(0)
    xh = dev["x"]
    dyh = dy
    # sampled tokens, one at a time (only its k experts leave the device): dx
    # and d_topk_w
    for t in np.sort(rng.choice(T, size=6, replace=False)):
        used, inv = np.unique(idx[t], return_inverse=True)
        sel = torch.from_numpy(used).long().cuda()
        ref = MB.backward(xh[t:t + 1].cpu(), inv.reshape(1, k).astype(np.int32), wts[t:t + 1],
                          dev["w_gate"].index_select(0, sel).cpu(),
                          dev["w_up"].index_select(0, sel).cpu(),
                          dev["w_down"].index_select(0, sel).cpu(), dyh[t:t + 1].cpu())
        assert rel_l2(dx[t:t + 1].double().cpu().numpy(), ref["dx"]) <= tol, t
        assert rel_l2(dtw[t:t + 1].double().cpu().numpy(), ref["dw"]) <= tol, t
    # sampled experts: the whole weight gradient from the pairs routed to them
    busy = np.argsort(-counts)
    for e in (int(busy[0]), int(busy[E // 2])):
        tt, ss = np.nonzero(idx == e)
        sel = torch.tensor([e], device="cuda").long()
        ref = MB.backward(xh[tt].cpu(), np.zeros((tt.size, 1), np.int32), wts[tt, ss][:, None],
                          dev["w_gate"].index_select(0, sel).cpu(),
                          dev["w_up"].index_select(0, sel).cpu(),
                          dev["w_down"].index_select(0, sel).cpu(), dyh[tt].cpu())
        for got, key in ((dwg, "dw_gate"), (dwu, "dw_up"), (dwd, "dw_down")):
            err = rel_l2(got[e].double().cpu().numpy(), ref[key][0])
            assert err <= tol, (e, key, err)
