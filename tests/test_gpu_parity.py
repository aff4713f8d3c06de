"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Reduced shapes keep each workload's routing structure (E, k, gate, top-k
convention, direct routes) at sizes the oracle checks in full; they span
several 128-row tiles, ragged group tails and partial N and K tiles.  Full
sizes run in the launch configuration the benchmark times and are checked
on routing (every token, bit-exact), grouping (bit-exact) and a seeded token
sample of the output.  Intermediates are poisoned with NaN before each run, so
a row the kernels failed to write shows up as a non-finite output.
"""
import dataclasses

import numpy as np
import pytest
import torch

import mixture_experts_ffn_04_gb300 as m
from mixture_experts_ffn_04_gb300 import workloads as W

from gpu_util import TOL, check_layer, rel_l2, run_gpu, to_dev

pytestmark = pytest.mark.gpu

REDUCED = [
    W.small(W.TINY_F32, T=300),
    W.small(W.QWEN3_30B_A3B, T=300, H=512, I=256),
    W.small(W.QWEN3_30B_A3B, T=77, H=392, I=200, E=16, k=3),      # ragged N and K
    W.small(W.DEEPSEEK_V3, T=260, H=512, I=256, I_sh=256),
    W.small(W.QWEN2_MOE, T=300, H=512, I=256, I_sh=512),
    W.small(W.QWEN2_MOE, T=5, H=512, I=256, I_sh=512),            # decode-sized
    W.small(W.QWEN2_MOE, T=1, H=512, I=256, I_sh=512),            # one token: one-row decode tiles
    W.small(W.QWEN2_MOE, T=3, H=512, I=256, I_sh=512),            # shared MLP in one decode tile
    W.small(W.ADV_E0, T=1, H=512, I=256, I_sh=256, k=3),          # one token's 3 routes to one expert
    W.small(W.ADV_E0, T=300, H=512, I=256, I_sh=256),
    W.small(W.ADV_ZIPF, T=300, H=512, I=256, I_sh=256),
    W.small(W.QWEN3_30B_A3B, T=100, H=256, I=128, E=64, k=40),    # k+1 > 32: warp top-k
    W.small(W.QWEN3_30B_A3B, T=200, H=256, I=128, E=300, k=4),    # E > 256
    W.small(W.QWEN3_30B_A3B, T=600, H=256, I=128, E=2048, k=4),   # > 1024 groups, > 512 columns
    W.small(W.GEMMA4_26B_A4B, T=300, H=704, I=176, E=16, k=4),    # input RMSNorm + residual
    dataclasses.replace(W.small(W.TINY_F32, T=200), input_norm=True, residual=True,
                        name="tiny-f32-norm-residual-T200"),
]
ENGINES = {0: "auto", 1: "cuda-core", 2: "tensor-core", 3: "skinny", 4: "tensor-core-pairs"}


def _cases():
    for wl in REDUCED:
        engines = [0, 3] if wl.dtype == "f32" else [0, 1, 2, 3, 4]
        for e in engines:
            yield pytest.param(wl, e, id="%s-%s" % (wl.name, ENGINES[e]))


@pytest.mark.parametrize("wl,engine", list(_cases()))
def test_reduced_parity(wl, engine):
    inp = W.make_inputs(wl, seed=0, device="cpu")
    dev = to_dev(inp)
    res = run_gpu(wl, dev, engine=engine)
    out = check_layer(wl, dev, res)
    assert out["launches"] > 0
    if wl.routing == "all_to_e0":
        assert out["max_group"] == wl.T * wl.k


# Full sizes: the output is checked on every token when the oracle can take
# them all, else ("tiles") on the tokens that own the first row of every
# expert group and the last row of each of its 128-row tiles.
FULL = [
    (W.TINY_F32, None),
    (W.QWEN3_30B_A3B, "tiles"),
    (W.DEEPSEEK_V3, "tiles"),
    (W.get("qwen2-moe-shape-T2048"), "tiles"),
    (W.get("qwen2-moe-shape-T64"), None),
    (W.get("qwen2-moe-shape-T8"), None),
    (W.get("qwen2-moe-shape-T1"), None),
    (W.get("adversarial-all-e0-T128"), None),
    (W.get("adversarial-all-e0-T16384"), "tiles"),
    (W.get("adversarial-zipf-T128"), None),
    (W.get("adversarial-zipf-T16384"), "tiles"),
    (W.get("gemma4-26b-a4b-shape-T512"), "tiles"),
    (W.get("gemma4-26b-a4b-shape-T4096"), "tiles"),
]


@pytest.mark.parametrize("wl,sample", FULL, ids=[f[0].name for f in FULL])
def test_full_size_parity(wl, sample):
    dev = W.make_inputs(wl, seed=0, device="cuda")
    res = run_gpu(wl, dev, poison=False)
    out = check_layer(wl, dev, res, sample=sample)
    print("%s: rel_l2=%.3e worst token %.3e over %d tokens near_ties=%d max_group=%d "
          "launches=%d" % (wl.name, out["rel_l2"], out["worst_token_rel_l2"],
                           out["tokens_checked"], out["ties"], out["max_group"], out["launches"]))
    if sample == "tiles":
        assert out["tokens_checked"] >= min(wl.T, 64)
    del dev, res
    torch.cuda.empty_cache()


def test_step_api_matches_layer_and_merged_fc1():
    """route -> permute -> grouped gate/up -> grouped down -> shared -> combine
    through the individual entry points gives the layer's grouped rows h and
    y_perm bit for bit (merged fc1, [E, 2I, H] with stride 2*I*H, gives the
    split result), and the combine of those rows with the layer's shared
    output gives the layer's output bit for bit.  The shared MLP itself agrees
    to rounding: at this size the layer splits its gate/up over K (fp32
    partial sums added in split order), the one-group step call does not."""
    wl = W.small(W.QWEN2_MOE, T=300, H=512, I=256, I_sh=512)
    dev = to_dev(W.make_inputs(wl, seed=3, device="cpu"))
    layer = m.MoELayer(wl, dev)
    y_ref = layer.forward(dev["x"])
    s = layer.shape
    T, H, I, E, k, Ish = wl.T, wl.H, wl.I, wl.E, wl.k, wl.I_sh
    ws = m.alloc_workspace(s, full=False)
    i32 = dict(dtype=torch.int32, device="cuda")
    idx, tw = torch.empty(T, k, **i32), torch.empty(T, k, dtype=torch.float32, device="cuda")
    gate = torch.empty(T, dtype=torch.float32, device="cuda")
    m.moe_route(s, dev["x"], dev["w_router"], idx, tw, gate, ws)
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    sidx, row_token = torch.empty(T, k, **i32), torch.empty(T * k, **i32)
    x_perm = torch.empty(T * k, H, dtype=torch.bfloat16, device="cuda")
    m.moe_permute(s, dev["x"], idx, counts, offsets, sidx, row_token, x_perm, ws)
    h = torch.empty(T * k, I, dtype=torch.bfloat16, device="cuda")
    merged = torch.cat([dev["w_gate"], dev["w_up"]], dim=1).contiguous()
    m.moe_grouped_swiglu(s, x_perm, merged, None, 2 * I * H, offsets, E, T * k, I, h, ws,
                         w_up_ptr=merged.data_ptr() + I * H * 2)
    y_perm = torch.empty(T * k, H, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_down(s, h, dev["w_down"], H * I, offsets, E, T * k, I, y_perm, ws)
    one = torch.tensor([0, T], **i32)
    hs = torch.empty(T, Ish, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_swiglu(s, dev["x"], dev["sh_gate"], dev["sh_up"], 0, one, 1, T, Ish, hs, ws)
    sh = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_down(s, hs, dev["sh_down"], 0, one, 1, T, Ish, sh, ws)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws)[0] == m.MOE_OK
    v = layer.views()
    assert torch.equal(h.view(torch.int16), v["h"].view(torch.int16))
    assert torch.equal(y_perm.view(torch.int16), v["y_perm"].view(torch.int16))
    sh_layer = v["shared_out"].clone()
    assert rel_l2(sh.double().cpu().numpy(), sh_layer.double().cpu().numpy()) < 2e-3
    torch.testing.assert_close(sh.float(), sh_layer.float(), rtol=2.0 ** -6, atol=1e-3)
    y = torch.empty_like(dev["x"])
    m.moe_combine(s, y_perm, sidx, tw, sh_layer, gate, y)   # no residual: this workload has none
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)


@pytest.mark.parametrize("engine", [1, 2, 3])
def test_gathered_rows_match_copied_rows(engine):
    """moe_permute without x_perm writes the same routing arrays, and
    moe_grouped_swiglu_gather on x + row_token gives h bit for bit equal to
    moe_grouped_swiglu on the grouped copy, on every engine (ragged K: H is not
    a multiple of 64; groups span several 128-row tiles)."""
    wl = W.small(W.QWEN3_30B_A3B, T=333, H=328, I=136, E=12, k=4)
    dev = to_dev(W.make_inputs(wl, seed=5, device="cpu"))
    s = m.shape_for(wl)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    ws = m.alloc_workspace(s, full=False)
    i32 = dict(dtype=torch.int32, device="cuda")
    idx, tw = torch.empty(T, k, **i32), torch.empty(T, k, dtype=torch.float32, device="cuda")
    m.moe_route(s, dev["x"], dev["w_router"], idx, tw, None, ws)
    outs = []
    for copy in (True, False):
        counts, offsets = torch.full((E,), -7, **i32), torch.full((E + 1,), -7, **i32)
        sidx, row_token = torch.full((T, k), -7, **i32), torch.full((T * k,), -7, **i32)
        x_perm = torch.empty(T * k, H, dtype=torch.bfloat16, device="cuda") if copy else None
        m.moe_permute(s, dev["x"] if copy else None, idx, counts, offsets, sidx, row_token,
                      x_perm, ws)
        h = torch.full((T * k, I), float("nan"), dtype=torch.bfloat16, device="cuda")
        prev = m.moe_testing_set_gemm_engine(engine)
        try:
            if copy:
                m.moe_grouped_swiglu(s, x_perm, dev["w_gate"], dev["w_up"], I * H, offsets, E,
                                     T * k, I, h, ws)
            else:
                m.moe_grouped_swiglu_gather(s, dev["x"], row_token, dev["w_gate"], dev["w_up"],
                                            I * H, offsets, E, T * k, I, h, ws)
        finally:
            m.moe_testing_set_gemm_engine(prev)
        torch.cuda.synchronize()
        assert m.moe_get_device_status(ws)[0] == m.MOE_OK
        outs.append((counts, offsets, sidx, row_token, h))
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)
    assert torch.isfinite(outs[1][4].float()).all()


@pytest.mark.parametrize("engine", [1, 2, 3])
def test_bad_gather_token_sets_device_flag(engine):
    """A row_token entry outside [0, T) reads nothing, gives a zero row of h
    and raises MOE_ERR_GATHER; the other rows are unaffected."""
    wl = W.small(W.QWEN3_30B_A3B, T=150, H=256, I=128, E=8, k=2)
    dev = to_dev(W.make_inputs(wl, seed=6, device="cpu"))
    s = m.shape_for(wl)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    ws = m.alloc_workspace(s, full=False)
    i32 = dict(dtype=torch.int32, device="cuda")
    idx, tw = torch.empty(T, k, **i32), torch.empty(T, k, dtype=torch.float32, device="cuda")
    m.moe_route(s, dev["x"], dev["w_router"], idx, tw, None, ws)
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    sidx, row_token = torch.empty(T, k, **i32), torch.empty(T * k, **i32)
    m.moe_permute(s, None, idx, counts, offsets, sidx, row_token, None, ws)
    hs = []
    prev = m.moe_testing_set_gemm_engine(engine)
    try:
        for bad in (False, True):
            rt = row_token.clone()
            if bad:
                rt[5] = T + 7
                rt[9] = -3
            h = torch.full((T * k, I), float("nan"), dtype=torch.bfloat16, device="cuda")
            m.moe_grouped_swiglu_gather(s, dev["x"], rt, dev["w_gate"], dev["w_up"], I * H,
                                        offsets, E, T * k, I, h, ws)
            st, bits = m.moe_get_device_status(ws)
            assert (st, bits) == ((m.MOE_ERR_GATHER, 8) if bad else (m.MOE_OK, 0))
            hs.append(h)
    finally:
        m.moe_testing_set_gemm_engine(prev)
    good, bad = hs
    assert torch.equal(bad[5].float(), torch.zeros(I, device="cuda"))
    assert torch.equal(bad[9].float(), torch.zeros(I, device="cuda"))
    keep = torch.ones(T * k, dtype=torch.bool, device="cuda")
    keep[5] = keep[9] = False
    assert torch.equal(good[keep].view(torch.int16), bad[keep].view(torch.int16))


def test_bad_direct_route_sets_device_flag():
    wl = W.small(W.ADV_ZIPF, T=64, H=256, I=128, I_sh=256)
    dev = to_dev(W.make_inputs(wl, seed=0, device="cpu"))
    dev["routes_idx"][5, 2] = wl.E + 3
    layer = m.MoELayer(wl, dev)
    y = layer.forward(dev["x"], routes_idx=dev["routes_idx"], routes_w=dev["routes_w"])
    st, bits = layer.device_status()
    assert st == m.MOE_ERR_DEVICE_ROUTE and bits & 1
    assert int(layer.views()["counts"].sum()) == wl.T * wl.k - 1
    assert bool(torch.isfinite(y).all())
    assert layer.device_status()[0] == m.MOE_OK  # read-and-clear


@pytest.mark.parametrize("engine", [1, 2, 3, 4])
def test_rows_beyond_bound_set_device_flag(engine):
    wl = W.small(W.QWEN3_30B_A3B, T=64, H=256, I=128, E=4, k=2)
    s = m.shape_for(wl)
    ws = m.alloc_workspace(s, full=False)
    offsets = torch.tensor([0, 40, 80, 100, 128], dtype=torch.int32, device="cuda")
    xp = torch.randn(128, 256, device="cuda").bfloat16()
    wg = torch.randn(4, 128, 256, device="cuda").bfloat16()
    h = torch.full((128, 128), 7.0, device="cuda").bfloat16()
    prev = m.moe_testing_set_gemm_engine(engine)
    try:
        m.moe_grouped_swiglu(s, xp, wg, wg, 128 * 256, offsets, 4, 100, 128, h, ws)
    finally:
        m.moe_testing_set_gemm_engine(prev)
    assert m.moe_get_device_status(ws)[0] == m.MOE_ERR_ROWS
    assert bool((h.float() == 7.0).all())  # nothing was computed


@pytest.mark.parametrize("groups", [[1000], [300, 0, 513, 7, 256, 257],
                                    [1, 16, 17, 33, 0, 255, 257, 384, 385, 512, 8, 9, 130]],
                         ids=["one-group", "ragged-groups", "small-and-half-tile-edges"])
def test_sm_pair_engine_matches_one_sm_engine(groups):
    """The SM-pair engine (256-row tiles over two CTAs; a group's last tile of
    at most 128 rows as an M = 128 half tile) gives the one-SM engine's h and
    y_perm bit for bit: the same fp32 sums in the same k order, one rounding.
    Ragged N and K (N = 200, K = 328), empty groups, groups of one tile and
    of one row past a tile, and groups whose last tile has 1, 128 and 129
    rows (half tile, half tile, full tile).  Both engines also give the same
    bits with per-group A maps (the rows past a group's end load as zeros)
    as with the global map (they load the next group's rows)."""
    G = len(groups)
    rows = sum(groups)
    H, I = 328, 200
    wl = W.small(W.QWEN3_30B_A3B, T=rows, H=H, I=I, E=max(G, 2), k=1)
    s = m.shape_for(wl)
    ws = m.alloc_workspace(s, full=False)
    g = torch.Generator(device="cuda").manual_seed(11)
    offs = torch.tensor([0] + list(np.cumsum(groups)), dtype=torch.int32, device="cuda")
    xp = torch.randn(rows, H, device="cuda", generator=g).bfloat16()
    wg = (torch.randn(G, I, H, device="cuda", generator=g) * 0.05).bfloat16()
    wu = (torch.randn(G, I, H, device="cuda", generator=g) * 0.05).bfloat16()
    wd = (torch.randn(G, H, I, device="cuda", generator=g) * 0.05).bfloat16()
    out = {}
    for zp in (-1, 1):
        for e in (2, 4):
            h = torch.full((rows, I), float("nan"), device="cuda").bfloat16()
            yp = torch.full((rows, H), float("nan"), device="cuda").bfloat16()
            prev = m.moe_testing_set_gemm_engine(e)
            prev_zp = m.moe_testing_set_zero_pad(zp)
            try:
                m.moe_grouped_swiglu(s, xp, wg, wu, I * H, offs, G, rows, I, h, ws)
                m.moe_grouped_down(s, h, wd, H * I, offs, G, rows, I, yp, ws)
            finally:
                m.moe_testing_set_gemm_engine(prev)
                m.moe_testing_set_zero_pad(prev_zp)
            torch.cuda.synchronize()
            assert m.moe_get_device_status(ws)[0] == m.MOE_OK
            assert torch.isfinite(h.float()).all() and torch.isfinite(yp.float()).all()
            out[(zp, e)] = (h, yp)
    ref = out[(-1, 2)]
    for key, (h, yp) in out.items():
        assert torch.equal(ref[0].view(torch.int16), h.view(torch.int16)), key
        assert torch.equal(ref[1].view(torch.int16), yp.view(torch.int16)), key


def test_zero_tokens_is_a_no_op():
    wl = W.small(W.QWEN3_30B_A3B, T=1, H=256, I=128, E=8, k=2)
    dev = to_dev(W.make_inputs(wl, seed=0, device="cpu"))
    s = m.shape_for(wl, T=0)
    ws = m.alloc_workspace(s)
    x = dev["x"][:0]
    y = torch.empty_like(x)
    m.moe_layer_forward(s, m.weights_from(dev), x, None, None, y, ws)
    assert m.moe_last_launch_count() == 0


def test_near_ties_match_the_oracle():
    """Router rows that are copies of others, or differ from them by one bf16
    ulp in a few entries, give exact ties and logit gaps of ~1e-5..1e-3 --
    below the fp32 error bound the kernel guards against, above the 1e-6
    tie threshold.  The exact re-decision must reproduce the oracle's order
    there; exact ties go to the lower expert index on both sides."""
    from oracle import oracle as O
    wl = W.small(W.QWEN3_30B_A3B, T=1024, H=2048, I=128, E=128, k=8)
    inp = W.make_inputs(wl, seed=5, device="cpu", with_experts=False)
    wr = inp["w_router"].clone()
    g = torch.Generator().manual_seed(7)
    for src, dst, nflip in [(3, 5, 0), (10, 11, 1), (20, 40, 2), (60, 61, 4), (70, 90, 8)]:
        row = wr[src].clone()
        if nflip:
            pos = torch.randperm(wl.H, generator=g)[:nflip]
            bits = row.view(torch.int16)
            bits[pos] += 1                       # one ulp up on a few entries
        wr[dst] = row
    s = m.shape_for(wl)
    ws = m.alloc_workspace(s, full=False)
    x = inp["x"].cuda()
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    tw = torch.empty(wl.T, wl.k, dtype=torch.float32, device="cuda")
    m.moe_route(s, x, wr.cuda(), idx, tw, None, ws)
    torch.cuda.synchronize()
    lg = O.router_logits(inp["x"], wr)
    ridx, rw, gap = O.topk_softmax(lg, wl.E, wl.k, True)
    gi = idx.cpu().numpy()
    mism = (gi != ridx).any(axis=1)
    assert not (mism & (gap >= 1e-6)).any(), np.nonzero(mism & (gap >= 1e-6))[0][:10]
    close = (gap < 1e-3).sum()
    assert close > 20, close   # the construction really produced near-ties
    print("near-tie tokens (gap < 1e-3): %d, exact ties: %d, mismatches: %d" % (
        close, int((gap == 0).sum()), int(mism.sum())))


@pytest.mark.parametrize("wl", [W.QWEN3_30B_A3B, W.DEEPSEEK_V3, W.get("qwen2-moe-shape-T2048"),
                                W.TINY_F32], ids=lambda w: w.name)
def test_router_logit_error_within_tie_bound(wl):
    """The fp32 router logits (tensor-core or FMA sums, split-K partials added
    in order) stay well inside the kernel's near-tie bound
    tau >= 2^-20 * sqrt(H): that bound is what makes the exact re-decision
    complete.  Also reports how many tokens were re-decided."""
    from oracle import oracle as O
    T = min(wl.T, 2048)
    inp = W.make_inputs(wl, seed=0, device="cuda", with_experts=False)
    x = inp["x"][:T].contiguous()
    s = m.shape_for(wl, T=T)
    ws = m.alloc_workspace(s, full=False)
    ncols = inp["w_router"].shape[0]
    lg = torch.empty(T, ncols, dtype=torch.float32, device="cuda")
    m.moe_testing_router_logits(s, x, inp["w_router"], lg, ws)
    idx = torch.empty(T, wl.k, dtype=torch.int32, device="cuda")
    tw = torch.empty(T, wl.k, dtype=torch.float32, device="cuda")
    gate = torch.empty(T, dtype=torch.float32, device="cuda") if wl.shared_gate else None
    m.moe_route(s, x, inp["w_router"], idx, tw, gate, ws)
    redecided = m.moe_get_route_stats(ws)
    ref = O.router_logits(x.cpu(), inp["w_router"].cpu())
    err = np.abs(lg.double().cpu().numpy() - ref).max()
    bound = 2.0 ** -20 * np.sqrt(wl.H)
    print("%s: max |fp32 logit - exact| = %.3e (%.3f of the smallest tie bound), "
          "re-decided %d of %d tokens" % (wl.name, err, err / bound, redecided, T))
    assert err < 0.5 * bound


@pytest.mark.parametrize("dtype,size", [("bf16", "small"), ("f32", "small"), ("bf16", "full")])
def test_residual_setup_matches_oracle(dtype, size):
    """moe_residual_setup against the oracle's RMSNorm (fp64, rounded once):
    bf16 bit for bit; fp32 within one ulp (the kernel's double-float value
    can sit on the other side of an fp32 rounding boundary about once in 2^22
    elements).  The full Gemma-4 size checks 11.5 M bf16 elements, a few
    thousand of them with exact values close to a bf16 rounding midpoint."""
    from oracle import oracle as O
    if size == "full":
        wl = W.GEMMA4_26B_A4B
    else:
        wl = W.small(W.GEMMA4_26B_A4B, T=300, H=704, I=176, E=16, k=4)
    wl = dataclasses.replace(wl, dtype=dtype)
    inp = W.make_inputs(wl, seed=9, with_experts=False)
    x = inp["x"] * 3.0 + 0.5          # an offset and a scale: rms far from 1
    ref = O.rmsnorm(x, inp["norm_weight"], wl.norm_eps)
    s = m.shape_for(wl)
    xd, wd = x.cuda(), inp["norm_weight"].cuda()
    out = torch.empty_like(xd)
    m.moe_residual_setup(s, xd, wd, out)
    got = out.cpu()
    if dtype == "bf16":
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    else:
        diff = (got.view(torch.int32).long() - ref.view(torch.int32).long()).abs()
        assert int(diff.max()) <= 1


def test_step_api_with_input_norm_and_residual():
    """residual_setup -> route -> permute -> gate/up -> down -> combine with
    the residual, through the individual entry points, equals the layer bit
    for bit."""
    wl = W.small(W.GEMMA4_26B_A4B, T=300, H=704, I=176, E=16, k=4)
    dev = to_dev(W.make_inputs(wl, seed=3, device="cpu"))
    layer = m.MoELayer(wl, dev)
    y_ref = layer.forward(dev["x"])
    s = layer.shape
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    ws = m.alloc_workspace(s, full=False)
    i32 = dict(dtype=torch.int32, device="cuda")
    xn = torch.empty_like(dev["x"])
    m.moe_residual_setup(s, dev["x"], dev["norm_weight"], xn)
    idx, tw = torch.empty(T, k, **i32), torch.empty(T, k, dtype=torch.float32, device="cuda")
    m.moe_route(s, xn, dev["w_router"], idx, tw, None, ws)
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    sidx, row_token = torch.empty(T, k, **i32), torch.empty(T * k, **i32)
    x_perm = torch.empty(T * k, H, dtype=torch.bfloat16, device="cuda")
    m.moe_permute(s, xn, idx, counts, offsets, sidx, row_token, x_perm, ws)
    h = torch.empty(T * k, I, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_swiglu(s, x_perm, dev["w_gate"], dev["w_up"], I * H, offsets, E, T * k, I, h, ws)
    y_perm = torch.empty(T * k, H, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_down(s, h, dev["w_down"], H * I, offsets, E, T * k, I, y_perm, ws)
    y = torch.empty_like(dev["x"])
    m.moe_combine(s, y_perm, sidx, tw, None, None, y, residual=dev["x"])
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws)[0] == m.MOE_OK
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


@pytest.mark.parametrize("T", [1, 8, 64, 2048])
def test_forked_shared_mlp_in_a_graph_matches_eager(T):
    """The shared MLP runs on a second stream forked from and joined back into
    the caller's stream (held to part of the SMs at decode sizes).  The same
    forward captured in a CUDA graph (the fork becomes a graph branch) gives
    the eager result bit for bit, and the eager result equals the traced entry
    point's, which keeps one stream."""
    wl = W.get("qwen2-moe-shape-T%d" % T)
    dev = W.make_inputs(wl, seed=4, device="cuda")
    layer = m.MoELayer(wl, dev)
    x = dev["x"]
    y_eager = torch.empty_like(x)
    layer.forward(x, y_eager)
    torch.cuda.synchronize()
    y_graph = torch.full_like(x, float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.moe_layer_forward(layer.shape, layer.weights, x, None, None, y_graph, layer.ws)
    g.replay()
    torch.cuda.synchronize()
    assert layer.device_status()[0] == m.MOE_OK
    assert torch.equal(y_eager.view(torch.int16), y_graph.view(torch.int16))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(m.STAGES) + 1)]
    for e in evs:
        e.record()
    y_traced = torch.empty_like(x)
    m.moe_layer_forward_traced(layer.shape, layer.weights, x, None, None, y_traced, layer.ws, evs)
    torch.cuda.synchronize()
    assert torch.equal(y_eager.view(torch.int16), y_traced.view(torch.int16))


@pytest.mark.parametrize("T", [1, 8, 64, 300, 2048])
def test_forked_shared_mlp_sm_cap_keeps_results(T):
    """The shared MLP's GEMMs on the forked stream may be held to fewer SMs
    (their CTAs then loop over the remaining column blocks or tiles; the
    SM-pair engine's K split, T = 300, keeps the split count of the whole
    GPU); every cap gives the uncapped result bit for bit."""
    if T == 300:
        wl = W.small(W.QWEN2_MOE, T=300, H=512, I=256, I_sh=512)
    else:
        wl = W.get("qwen2-moe-shape-T%d" % T)
    dev = W.make_inputs(wl, seed=6, device="cuda")
    layer = m.MoELayer(wl, dev)
    prev = m.moe_testing_set_fork_sms(-1)
    try:
        ref = layer.forward(dev["x"])
        for sms in (1, 7, 60, 151):
            m.moe_testing_set_fork_sms(sms)
            y = torch.full_like(ref, float("nan"))
            layer.forward(dev["x"], y)
            torch.cuda.synchronize()
            assert layer.device_status()[0] == m.MOE_OK
            assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), sms
    finally:
        m.moe_testing_set_fork_sms(prev)


def test_forked_shared_mlp_from_two_host_threads():
    """Two host threads, each with its own layer, workspace and stream, call
    the decode-sized forward at once; they share the library's side stream
    (one per device, its fork and join taken under a lock), and every output
    equals that layer's single-threaded result bit for bit."""
    import threading
    layers, xs, refs, outs, streams = [], [], [], [], []
    for i, T in enumerate((1, 8)):
        wl = W.get("qwen2-moe-shape-T%d" % T)
        dev = W.make_inputs(wl, seed=20 + i, device="cuda")
        layer = m.MoELayer(wl, dev)
        ref = torch.empty_like(dev["x"])
        layer.forward(dev["x"], ref)
        layers.append(layer)
        xs.append(dev["x"])
        refs.append(ref)
        outs.append([torch.full_like(dev["x"], float("nan")) for _ in range(24)])
        streams.append(torch.cuda.Stream())
    torch.cuda.synchronize()
    errors = []
    start = threading.Barrier(2)

    def run(i):
        try:
            start.wait()
            with torch.cuda.stream(streams[i]):
                for y in outs[i]:
                    layers[i].forward(xs[i], y, stream=streams[i])
            streams[i].synchronize()
        except Exception as exc:   # reported by the main thread
            errors.append(exc)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    torch.cuda.synchronize()
    for i in range(2):
        assert layers[i].device_status()[0] == m.MOE_OK
        for y in outs[i]:
            assert torch.equal(y.view(torch.int16), refs[i].view(torch.int16))
