"""GPU parity of the routed-expert backward (include/moe_backward.h) against
the fp64 backward oracle (oracle/moe_backward.py), through the C ABI.

Routes are inputs of this op: router workloads take the oracle's own routing
(fp32 weights) as direct routes, the adversarial workloads their direct
routes, so both sides see the same routes and nothing the CUDA path computed
feeds the oracle.  Tolerances as for the forward: bf16 within 1e-2 relative
L2 of the oracle (every value finite), fp32 within 1e-4.  Gradient buffers
start as NaN, so a row or an expert the kernels skip shows up.

Cases: reduced Qwen3-30B-A3B / DeepSeek-V3 / Gemma-4 (with the residual)
shapes; the tiny fp32 layer; "Fused MoE Kernel Notes", Duplicate top-k
routes (every slot of every token on expert 0, so one group holds T*k rows);
Zipf routing with duplicates and empty experts; a moe_inter that is not a
multiple of 64 (the gate/up dgrad then runs on the CUDA cores); 1100 experts
(tile schedule and offsets in global memory); a single token with top-1; each
bf16 case on the tensor-core path and on the CUDA-core path."""
import dataclasses

import numpy as np
import pytest
import torch

import mixture_experts_ffn_04_gb300 as m
from mixture_experts_ffn_04_gb300 import workloads as W
from oracle import moe_backward as MB
from oracle import oracle as O

from gpu_util import TOL, rel_l2, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    W.small(W.QWEN3_30B_A3B, T=300, H=256, I=192, E=8, k=4),
    W.small(W.DEEPSEEK_V3, T=160, H=512, I=256, E=16, k=8, I_sh=0),
    dataclasses.replace(W.small(W.GEMMA4_26B_A4B, T=128, H=320, I=704, E=6, k=4),
                        input_norm=False, residual=True, name="gemma4-shape-residual-T128"),
    W.TINY_F32,
    W.small(W.ADV_E0, T=96, H=256, I=128, E=8, k=6, I_sh=0),
    W.small(W.ADV_ZIPF, T=128, H=384, I=320, E=16, k=6, I_sh=0),
    W.small(W.QWEN3_30B_A3B, T=70, H=136, I=200, E=5, k=3),
    # more groups than the kernels keep in shared memory (device-built global
    # tile schedule, offsets read from global memory), most of them empty
    W.small(W.QWEN3_30B_A3B, T=40, H=128, I=64, E=1100, k=2),
    # one token, one slot
    W.small(W.QWEN3_30B_A3B, T=1, H=64, I=64, E=4, k=1),
]


def _cases():
    for wl in CASES:
        for e in ([0] if wl.dtype == "f32" else [0, 1]):
            yield pytest.param(wl, e, id="%s-%s" % (wl.name, "auto" if e == 0 else "cuda-core"))


def _routes(wl, host):
    """Direct routes for both sides: the oracle's routing or the workload's."""
    if wl.routing == "router":
        r = O.route(wl, {"x": host["x"], "w_router": host["w_router"], "routes_idx": None,
                         "routes_w": None, "norm_weight": None})
        return r["idx"].astype(np.int32), r["weights"].astype(np.float32)
    return host["routes_idx"].numpy(), host["routes_w"].numpy()


def run_backward(wl, host, idx, wts, dy, engine=0):
    dev = to_dev(host)
    ridx = torch.from_numpy(idx).cuda()
    rw = torch.from_numpy(wts).cuda()
    wl_direct = dataclasses.replace(wl, routing="zipf", shared_gate=False)
    prev = m.moe_testing_set_gemm_engine(engine)
    try:
        layer = m.MoELayer(wl_direct, dev, train=True)
        for t in m.moe_backward_views(layer.shape, layer.ws).values():
            t.fill_(float("nan"))
        y = layer.forward(dev["x"], routes_idx=ridx, routes_w=rw)
        E, I, H = wl.E, wl.I, wl.H
        nan = float("nan")
        dwg = torch.full((E, I, H), nan, device="cuda").to(wl.torch_dtype)
        dwu = torch.full((E, I, H), nan, device="cuda").to(wl.torch_dtype)
        dwd = torch.full((E, H, I), nan, device="cuda").to(wl.torch_dtype)
        dx = torch.full_like(dev["x"], nan)
        dtw = torch.full((wl.T, wl.k), nan, device="cuda")
        layer.backward(dy.cuda(), dx, dtw, m.grads_for(dwg, dwu, dwd))
        st, bits = layer.device_status()
        launches = m.moe_last_launch_count()
    finally:
        m.moe_testing_set_gemm_engine(prev)
    assert st == m.MOE_OK, (st, bits)
    return dict(y=y.cpu(), dx=dx.cpu(), dw=dtw.cpu(), dw_gate=dwg.cpu(), dw_up=dwu.cpu(),
                dw_down=dwd.cpu(), launches=launches)


@pytest.mark.parametrize("wl,engine", list(_cases()))
def test_layer_backward_matches_oracle(wl, engine):
    host = W.make_inputs(wl, seed=3)
    dy = W.make_output_grad(wl, seed=3)
    idx, wts = _routes(wl, host)
    got = run_backward(wl, host, idx, wts, dy, engine)
    ref = MB.backward(host["x"], idx, wts, host["w_gate"], host["w_up"], host["w_down"], dy)
    if wl.residual:
        ref["dx"] = ref["dx"] + dy.double().numpy()
    tol = TOL[wl.dtype]
    used = np.zeros(wl.E, dtype=bool)
    used[np.unique(idx)] = True
    errs = {}
    for key in ("dx", "dw", "dw_gate", "dw_up", "dw_down"):
        g = got[key].double().numpy()
        assert np.isfinite(g).all(), "non-finite %s" % key
        errs[key] = rel_l2(g, ref[key])
        assert errs[key] <= tol, "%s rel L2 %.3e > %.0e" % (key, errs[key], tol)
    for key in ("dw_gate", "dw_up", "dw_down"):
        assert (got[key][torch.from_numpy(~used)] == 0).all(), "unused expert's %s not zero" % key
    # the train-mode forward is the forward
    yref = O.moe_ffn(host["x"], idx, wts.astype(np.float64), None, host["w_gate"],
                     host["w_up"], host["w_down"])
    if wl.residual:
        yref = yref + host["x"].double().numpy()
    assert rel_l2(got["y"].double().numpy(), yref) <= tol
    print("\n%s engine %d: %s, %d launches" % (wl.name, engine,
          ", ".join("%s %.2e" % kv for kv in errs.items()), got["launches"]))


def test_duplicate_routes_split_and_merged_fc1_agree():
    """The regression of "Fused MoE Kernel Notes", Duplicate top-k routes:
    every slot of every token on expert 0 (one group of T*k rows, far more
    than T) with equal routing weights; the split-fc1 and merged-fc1 weight
    layouts give bit-identical gradients, all finite, and both match the
    oracle."""
    wl = W.small(W.ADV_E0, T=128, H=256, I=128, E=4, k=2, I_sh=0)
    host = W.make_inputs(wl, seed=5)
    dy = W.make_output_grad(wl, seed=5)
    idx = np.zeros((wl.T, wl.k), np.int32)
    wts = np.full((wl.T, wl.k), 0.5, np.float32)
    split = run_backward(wl, host, idx, wts, dy)
    # merged fc1: [E, 2I, H], gate rows then up rows of each expert
    merged = torch.cat([host["w_gate"], host["w_up"]], dim=1).contiguous()
    dev = to_dev(host)
    dev_m = dict(dev)
    mg = merged.cuda()
    E, I, H = wl.E, wl.I, wl.H
    layer = m.MoELayer(dataclasses.replace(wl, routing="zipf"), dev_m, train=True)
    layer.weights.gate = mg.data_ptr()
    layer.weights.up = mg.data_ptr() + I * H * 2
    layer.weights.gate_up_stride = 2 * I * H
    layer.forward(dev["x"], routes_idx=torch.from_numpy(idx).cuda(),
                  routes_w=torch.from_numpy(wts).cuda())
    dfc1 = torch.full((E, 2 * I, H), float("nan"), device="cuda").bfloat16()
    dwd = torch.full((E, H, I), float("nan"), device="cuda").bfloat16()
    g = m.MoEExpertGrads()
    g.gate, g.up = dfc1.data_ptr(), dfc1.data_ptr() + I * H * 2
    g.gate_up_stride = 2 * I * H
    g.down, g.down_stride = dwd.data_ptr(), H * I
    dx = torch.empty_like(dev["x"])
    dtw = torch.empty((wl.T, wl.k), device="cuda")
    layer.backward(dy.cuda(), dx, dtw, g)
    assert layer.device_status()[0] == m.MOE_OK
    dfc1 = dfc1.cpu()
    assert torch.equal(dx.cpu().view(torch.int16), split["dx"].view(torch.int16))
    assert torch.equal(dfc1[:, :I].view(torch.int16), split["dw_gate"].view(torch.int16))
    assert torch.equal(dfc1[:, I:].view(torch.int16), split["dw_up"].view(torch.int16))
    assert torch.equal(dwd.cpu().view(torch.int16), split["dw_down"].view(torch.int16))
    assert torch.equal(dtw.cpu(), split["dw"])
    assert torch.isfinite(split["dx"].float()).all() and torch.isfinite(dfc1.float()).all()
    ref = MB.backward(host["x"], idx, wts, host["w_gate"], host["w_up"], host["w_down"], dy)
    for key in ("dx", "dw", "dw_gate", "dw_up", "dw_down"):
        assert rel_l2(split[key].double().numpy(), ref[key]) <= TOL["bf16"], key


@pytest.mark.parametrize("engine", [0, 1])
def test_grouped_wgrad_matches_definition(engine):
    """moe_grouped_wgrad alone: ragged groups (empty, one row, 63, 64, 65 and
    several hundred rows), rows past the last group set to NaN (a group's
    tail block must not read them), M and N not multiples of the tile."""
    sizes = [0, 1, 63, 64, 65, 0, 300, 129]
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offsets[-1])
    bound = rows + 40
    M, N = 200, 328
    g = torch.Generator().manual_seed(11)
    a = (torch.randn(bound, M, generator=g) * 0.5).bfloat16()
    b = (torch.randn(bound, N, generator=g) * 0.5).bfloat16()
    a[rows:] = float("nan")
    b[rows:] = float("nan")
    wl = W.small(W.QWEN3_30B_A3B, T=64, H=256, I=128, E=len(sizes), k=2)
    s = m.shape_for(wl)
    ws = m.alloc_workspace(s, full=False)
    G = len(sizes)
    dw = torch.full((G, M, N), float("nan"), device="cuda").bfloat16()
    prev = m.moe_testing_set_gemm_engine(engine)
    try:
        m.moe_grouped_wgrad(s, a.cuda(), M, b.cuda(), N, torch.from_numpy(offsets).cuda(), G,
                            bound, M, N, dw, M * N, ws)
        assert m.moe_get_device_status(ws)[0] == m.MOE_OK
    finally:
        m.moe_testing_set_gemm_engine(prev)
    ref = MB.group_weight_grads(a[:rows], b[:rows], offsets)
    got = dw.cpu().double().numpy()
    assert np.isfinite(got).all()
    for gi, n in enumerate(sizes):
        if n == 0:
            assert (got[gi] == 0).all()
        else:
            assert rel_l2(got[gi], ref[gi]) <= TOL["bf16"], (gi, rel_l2(got[gi], ref[gi]))


def test_scatter_grad_and_gather_grad_steps():
    """The two non-GEMM steps through their own entry points: grad_fc2 rows
    are topk_w * dy rounded once, d_topk_w the fp32 dot with y_perm, and the
    gather sums each token's rows (plus the residual gradient)."""
    wl = W.small(W.ADV_ZIPF, T=96, H=256, I=128, E=8, k=6, I_sh=0)
    host = W.make_inputs(wl, seed=9)
    dy = W.make_output_grad(wl, seed=9)
    idx = host["routes_idx"].numpy()
    wts = host["routes_w"].numpy()
    counts, offsets, sidx, row_token = O.permute(idx, wl.E)
    R = wl.T * wl.k
    g = torch.Generator().manual_seed(2)
    y_perm = torch.randn(R, wl.H, generator=g).bfloat16()
    s = m.shape_for(wl)
    gf = torch.full((R, wl.H), float("nan"), device="cuda").bfloat16()
    dtw = torch.full((wl.T, wl.k), float("nan"), device="cuda")
    sidx_d = torch.from_numpy(sidx).cuda()
    m.moe_scatter_grad(s, dy.cuda(), sidx_d, torch.from_numpy(wts).cuda(), y_perm.cuda(), gf,
                       dtw)
    torch.cuda.synchronize()
    dyd = dy.double().numpy()
    exp_g = np.zeros((R, wl.H))
    exp_w = np.zeros((wl.T, wl.k))
    yp = y_perm.double().numpy()
    for t in range(wl.T):
        for j in range(wl.k):
            r = sidx[t, j]
            exp_g[r] = wts[t, j] * dyd[t]
            exp_w[t, j] = float(np.dot(dyd[t], yp[r]))
    # grad_fc2: the product rounded once (fp32 product of two exact values)
    want = torch.from_numpy(exp_g).float().bfloat16()
    assert torch.equal(gf.cpu().view(torch.int16), want.view(torch.int16))
    np.testing.assert_allclose(dtw.cpu().double().numpy(), exp_w, rtol=1e-4, atol=1e-3)
    # gather with a residual gradient
    dxp = torch.randn(R, wl.H, generator=g).bfloat16()
    dx = torch.empty((wl.T, wl.H), device="cuda").bfloat16()
    m.moe_gather_grad(s, dxp.cuda(), sidx_d, dy.cuda(), dx)
    exp = dyd.copy()
    dxpd = dxp.double().numpy()
    for t in range(wl.T):
        for j in range(wl.k):
            exp[t] += dxpd[sidx[t, j]]
    assert rel_l2(dx.cpu().double().numpy(), exp) <= 4e-3


def test_train_forward_keeps_bit_identical_h():
    """moe_grouped_swiglu_save writes the same h as moe_grouped_swiglu, and
    its fc1 rows are the gate / up pre-activations (oracle values rounded
    once, so within one bf16 rounding)."""
    wl = W.small(W.QWEN3_30B_A3B, T=200, H=256, I=192, E=8, k=4)
    host = W.make_inputs(wl, seed=1)
    idx, _ = _routes(wl, host)
    counts, offsets, sidx, row_token = O.permute(idx, wl.E)
    x_perm = host["x"][torch.from_numpy(row_token).long()].contiguous().cuda()
    s = m.shape_for(wl)
    ws = m.alloc_workspace(s, full=False)
    R, I = wl.T * wl.k, wl.I
    off = torch.from_numpy(offsets).cuda()
    dev = to_dev(host)
    for engine in (0, 1):
        prev = m.moe_testing_set_gemm_engine(engine)
        try:
            h0 = torch.empty((R, I), device="cuda").bfloat16()
            h1 = torch.empty((R, I), device="cuda").bfloat16()
            fc1 = torch.empty((R, 2 * I), device="cuda").bfloat16()
            m.moe_grouped_swiglu(s, x_perm, dev["w_gate"], dev["w_up"], I * wl.H, off, wl.E, R,
                                 I, h0, ws)
            m.moe_grouped_swiglu_save(s, x_perm, dev["w_gate"], dev["w_up"], I * wl.H, off,
                                      wl.E, R, I, h1, fc1, ws)
            assert m.moe_get_device_status(ws)[0] == m.MOE_OK
        finally:
            m.moe_testing_set_gemm_engine(prev)
        assert torch.equal(h0.view(torch.int16), h1.view(torch.int16))
        X = host["x"].double().numpy()[row_token]
        e_of_row = np.repeat(np.arange(wl.E), counts)
        wg = host["w_gate"].double().numpy()[e_of_row]
        wu = host["w_up"].double().numpy()[e_of_row]
        a = np.einsum("rh,rih->ri", X, wg)
        b = np.einsum("rh,rih->ri", X, wu)
        got = fc1.cpu().double().numpy()
        assert rel_l2(got[:, :I], a) <= 4e-3 and rel_l2(got[:, I:], b) <= 4e-3
