"""Helpers for the GPU parity tests: run the CUDA path through the C ABI, run
the fp64 oracle on the same seeded inputs, and compare.

Tolerances (from the layer's numeric contract): fp32 layers within 1e-4
relative L2 of the oracle, bf16 layers within 1e-2 relative L2 with every
value finite; routing indices, counts, offsets and scatter_index bit-exact,
except tokens whose oracle top-(k+1) logits have a neighbour gap below 1e-6
(a near-tie: either order is a correct answer), which are reported.
"""
import numpy as np
import torch

import mixture_experts_ffn_04_gb300 as m
from mixture_experts_ffn_04_gb300 import workloads as W
from oracle import oracle as O

TOL = {"f32": 1e-4, "bf16": 1e-2}
# bound on each token's own relative L2 in the full-size checks: twice the
# pooled bar (one row's rounding noise is noisier than a pool of rows)
ROW_TOL = {"f32": 2e-4, "bf16": 2e-2}
TILE_ROWS = 128
TIE_GAP = 1e-6
W_ATOL = 2e-5   # routing weights: fp32 softmax of fp32 logits


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def to_dev(inputs):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()}


def run_gpu(wl, dev, engine=0, poison=True):
    """Whole layer through moe_layer_forward; returns y and host copies of the
    routing views and the device status."""
    prev = m.moe_testing_set_gemm_engine(engine)
    try:
        layer = m.MoELayer(wl, dev)
        if poison:
            v = layer.views()
            for key in ("x_perm", "h", "y_perm", "shared_out"):
                if v[key] is not None:
                    v[key].fill_(float("nan"))
        y = layer.forward(dev["x"], routes_idx=dev.get("routes_idx"), routes_w=dev.get("routes_w"))
        st, bits = layer.device_status()
        launches = m.moe_last_launch_count()
        v = layer.views()
        out = {k: (t.cpu() if t is not None else None) for k, t in v.items()
               if k in ("topk_idx", "topk_w", "gate", "counts", "offsets", "scatter_index",
                        "row_token")}
    finally:
        m.moe_testing_set_gemm_engine(prev)
    out.update(y=y, status=st, bits=bits, launches=launches)
    return out


def oracle_ffn(wl, host_x, dev_or_host, tokens, idx, w, gate):
    """Oracle FFN + combine for `tokens`, pulling only the experts those
    tokens use (compact copy on the host, indices remapped)."""
    used = np.unique(idx)
    sel = torch.as_tensor(used, dtype=torch.long)
    if len(used) == wl.E:
        pick = lambda t: t.cpu()
    else:
        pick = lambda t: t.index_select(0, sel.to(t.device)).cpu()
    wg, wu, wd = pick(dev_or_host["w_gate"]), pick(dev_or_host["w_up"]), pick(dev_or_host["w_down"])
    remap = np.zeros(wl.E, dtype=np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    sh = [dev_or_host.get(k) for k in ("sh_gate", "sh_up", "sh_down")]
    sh = [None if t is None else t.cpu() for t in sh]
    return O.moe_ffn(host_x, remap[idx], w, gate, wg, wu, wd, sh[0], sh[1], sh[2],
                     tokens=np.asarray(tokens, dtype=np.int64))


def host_routing_inputs(dev):
    d = {"x": dev["x"].cpu()}
    for k in ("w_router", "routes_idx", "routes_w", "norm_weight"):
        d[k] = None if dev.get(k) is None else dev[k].cpu()
    return d


def tile_sample(counts, offsets, row_token):
    """Tokens whose rows cover every 128-row tile of every expert group: for
    each group its first row, and the last row of each of its 128-row tiles
    (the group's last row for the ragged tail).  Taken from the oracle's
    grouping, so a tile computed wrong, or not at all, at any group or tile
    position is in the sample."""
    rows = []
    for g in range(len(counts)):
        c = int(counts[g])
        if c == 0:
            continue
        o = int(offsets[g])
        rows.append(o)
        for t0 in range(0, c, TILE_ROWS):
            rows.append(o + min(t0 + TILE_ROWS, c) - 1)
    return np.unique(row_token[np.asarray(rows, dtype=np.int64)])


def check_layer(wl, dev, res, sample=None, report=None):
    """Compare a GPU result with the oracle.  sample: token subset for the
    FFN/combine comparison (all tokens when None; "tiles": tile_sample of the
    oracle's grouping).  The pooled relative L2 must be within TOL and every
    checked token's own within ROW_TOL.  Returns a dict of the measured
    errors."""
    T = wl.T
    assert res["status"] == m.MOE_OK, (res["status"], res["bits"])
    y = res["y"]
    assert bool(torch.isfinite(y).all()), "non-finite output"
    hin = host_routing_inputs(dev)
    xin = O.layer_input(wl, hin)                   # x, or its input RMSNorm
    r_all = O.route(wl, hin, xin=xin)              # every token
    gidx = res["topk_idx"].numpy() if res["topk_idx"] is not None else None
    if wl.routing == "router":
        mism = (gidx != r_all["idx"]).any(axis=1)
        allowed = r_all["gap"] < TIE_GAP
        bad = np.nonzero(mism & ~allowed)[0]
        assert bad.size == 0, "routing differs at tokens %s (gaps %s)" % (
            bad[:8].tolist(), r_all["gap"][bad[:8]].tolist())
        ok = ~mism
        gw = res["topk_w"].numpy()
        np.testing.assert_allclose(gw[ok], r_all["weights"][ok], atol=W_ATOL, rtol=1e-4)
        if wl.shared_gate:
            np.testing.assert_allclose(res["gate"].numpy(), r_all["gate"], atol=1e-5, rtol=1e-5)
        route_idx = gidx
        n_ties = int(mism.sum())
    else:
        route_idx = r_all["idx"]
        ok = np.ones(T, dtype=bool)
        n_ties = 0
    # grouping: bit-exact against the oracle's permutation of the same routes
    counts, offsets, sidx, row_token = O.permute(route_idx, wl.E)
    assert np.array_equal(res["counts"].numpy(), counts)
    assert np.array_equal(res["offsets"].numpy(), offsets)
    assert np.array_equal(res["scatter_index"].numpy(), sidx)
    assert np.array_equal(res["row_token"].numpy(), row_token)
    # layer output
    if isinstance(sample, str) and sample == "tiles":
        sample = tile_sample(counts, offsets, row_token)
    tokens = np.arange(T) if sample is None else np.asarray(sample)
    tokens = tokens[ok[tokens]]
    ref = oracle_ffn(wl, xin, dev, tokens, r_all["idx"][tokens], r_all["weights"][tokens],
                     None if r_all["gate"] is None else r_all["gate"][tokens])
    if wl.residual:
        ref = ref + hin["x"].double().numpy()[tokens]
    yg = y.index_select(0, torch.as_tensor(tokens, device=y.device)).double().cpu().numpy()
    err = rel_l2(yg, ref)
    tol = TOL[wl.dtype]
    assert err <= tol, "rel L2 %.3e > %.0e" % (err, tol)
    # every sampled token on its own (a wrong tile shows up in its rows even
    # when the pooled error stays small)
    per = (np.linalg.norm(yg - ref, axis=1)
           / np.maximum(np.linalg.norm(ref, axis=1), 1e-300)) if len(tokens) else np.zeros(0)
    worst = float(per.max()) if per.size else 0.0
    assert worst <= ROW_TOL[wl.dtype], "token %d: rel L2 %.3e > %.0e" % (
        int(tokens[int(per.argmax())]), worst, ROW_TOL[wl.dtype])
    out = dict(rel_l2=err, worst_token_rel_l2=worst, tokens_checked=int(len(tokens)),
               ties=n_ties, max_group=int(counts.max()) if counts.size else 0,
               launches=res["launches"])
    if report is not None:
        report.append((wl.name, out))
    return out
