"""Hash-MoE routing (moe_hash_route) on the GPU against the oracle's lookup,
and the layer driven by it ("Fused MoE Kernel Notes", Duplicate top-k routes:
a token-to-expert lookup can send both slots of a token to one expert).

* routes and weights bit-exact against oracle.hash_route, with duplicate
  slots, and token ids outside the table flagged (MOE_ERR_DEVICE_ROUTE) and
  dropped;
* the notes' example: 128 tokens, top-k 2, every slot on expert 0 -> one
  group of 256 rows; forward and backward finite and equal to the oracle;
* a Zipf-like table at the Qwen3-30B-A3B widths, forward and backward
  against the oracle (bf16 within 1e-2 relative L2)."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_04_gb300 as m
from mixture_experts_ffn_04_gb300 import workloads as W
from oracle import moe_backward as MB
from oracle import oracle as O

from gpu_util import TOL, rel_l2

pytestmark = pytest.mark.gpu


def _table(vocab, k, E, seed, dup_all=False):
    rng = np.random.default_rng(seed)
    if dup_all:
        return np.zeros((vocab, k), np.int32)
    p = np.arange(1, E + 1, dtype=np.float64) ** -0.8
    tab = rng.choice(E, size=(vocab, k), p=p / p.sum()).astype(np.int32)
    tab[::7, 1] = tab[::7, 0]   # explicit duplicates in every seventh row
    return tab


def test_hash_route_matches_oracle_and_flags_bad_ids():
    wl = W.small(W.QWEN3_30B_A3B, T=1000, H=256, I=128, E=64, k=8)
    s = m.shape_for(wl)
    ws = m.alloc_workspace(s, full=False)
    vocab = 500
    tab = _table(vocab, wl.k, wl.E, 1)
    ids = np.random.default_rng(2).integers(0, vocab, size=wl.T).astype(np.int32)
    for bad in (False, True):
        if bad:
            ids[[3, 500, 999]] = [-1, vocab, 1 << 30]
        idx = torch.full((wl.T, wl.k), 77, dtype=torch.int32, device="cuda")
        w = torch.full((wl.T, wl.k), -1.0, device="cuda")
        m.moe_hash_route(s, torch.from_numpy(ids).cuda(), torch.from_numpy(tab).cuda(), vocab,
                         idx, w, ws)
        st, bits = m.moe_get_device_status(ws)
        ridx, rw = O.hash_route(ids, tab, wl.k)
        assert np.array_equal(idx.cpu().numpy(), ridx)
        assert np.array_equal(w.cpu().numpy(), rw.astype(np.float32))
        assert st == (m.MOE_ERR_DEVICE_ROUTE if bad else m.MOE_OK), (st, bits)
    assert any(len(set(r)) < wl.k for r in ridx.tolist())   # duplicate slots present


@pytest.mark.parametrize("case", ["all-to-expert-0-T128-k2", "zipf-table-qwen3-widths"])
def test_layer_forward_and_backward_on_hash_routes(case):
    if case.startswith("all"):
        wl = W.small(W.ADV_E0, T=128, H=256, I=128, E=8, k=2, I_sh=0)
        vocab, tab = 64, _table(64, 2, 8, 0, dup_all=True)
    else:
        wl = W.small(W.QWEN3_30B_A3B, T=512, H=2048, I=768, E=128, k=8)
        vocab, tab = 5000, _table(5000, 8, 128, 3)
    host = W.make_inputs(wl, seed=4)
    dy = W.make_output_grad(wl, seed=4)
    ids = np.random.default_rng(5).integers(0, vocab, size=wl.T).astype(np.int32)
    dev = {k: (v.cuda() if v is not None else None) for k, v in host.items()}
    layer = m.MoELayer(wl, dev, train=True)
    idx = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.k), device="cuda")
    m.moe_hash_route(layer.shape, torch.from_numpy(ids).cuda(), torch.from_numpy(tab).cuda(),
                     vocab, idx, w, layer.ws)
    y = layer.forward(dev["x"], routes_idx=idx, routes_w=w)
    E, I, H = wl.E, wl.I, wl.H
    dwg = torch.empty((E, I, H), device="cuda", dtype=torch.bfloat16)
    dwu = torch.empty_like(dwg)
    dwd = torch.empty((E, H, I), device="cuda", dtype=torch.bfloat16)
    dx = torch.empty_like(dev["x"])
    dtw = torch.empty((wl.T, wl.k), device="cuda")
    layer.backward(dy.cuda(), dx, dtw, m.grads_for(dwg, dwu, dwd))
    st, bits = layer.device_status()
    assert st == m.MOE_OK, (st, bits)
    ridx, rw = O.hash_route(ids, tab, wl.k)
    counts = np.bincount(ridx.reshape(-1), minlength=E)
    if case.startswith("all"):
        assert counts[0] == 2 * wl.T   # one group of T*k rows, far more than T
    yref = O.moe_ffn(host["x"], ridx, rw.astype(np.float32).astype(np.float64), None,
                     host["w_gate"], host["w_up"], host["w_down"])
    assert rel_l2(y.double().cpu().numpy(), yref) <= TOL["bf16"]
    ref = MB.backward(host["x"], ridx, rw.astype(np.float32), host["w_gate"], host["w_up"],
                      host["w_down"], dy)
    for got, key in ((dx, "dx"), (dtw, "dw"), (dwg, "dw_gate"), (dwu, "dw_up"),
                     (dwd, "dw_down")):
        g = got.double().cpu().numpy()
        assert np.isfinite(g).all(), key
        assert rel_l2(g, ref[key]) <= TOL["bf16"], (key, rel_l2(g, ref[key]))
