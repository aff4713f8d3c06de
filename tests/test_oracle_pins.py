"""Pins for the fp64 oracle, independent of the oracle's own code.

Each ``check_*`` function compares the oracle with something the pages or the
mathematics fix: values printed on the pages (tests/golden), brute force on
tiny inputs, closed forms, and library routines in the special cases where the
layer reduces to one.  ``test_oracle_mutations.py`` re-runs these checks
against deliberately broken copies of the oracle and expects them to fail.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import expit, softmax

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


# --------------------------------------------------------------------------
# routing shape word (compiler page, Group A)
# --------------------------------------------------------------------------
def check_shape_words():
    g = _golden("topk_shape_words.json")
    for row in g["valid"]:
        w = O.topk_pack(row["num_experts"], row["top_k"])
        assert w == row["word"], (row, w)
        assert O.topk_unpack(w) == (row["num_experts"], row["top_k"])
        assert w < (1 << 22)  # fits the 22-bit immediate
    for row in g["invalid"]:
        assert O.topk_pack(row["num_experts"], row["top_k"]) == 0, row
    assert O.topk_unpack(0) is None          # never-set register is an error
    assert O.topk_unpack(1 << 22) is None


def test_shape_words(orc):
    check_shape_words()


def test_topk_rejects_missing_shape(orc):
    with pytest.raises(ValueError):
        O.topk_softmax(np.zeros((1, 4)), 4, 2, True, word=0)


# --------------------------------------------------------------------------
# top-k selection: brute force over all subsets on tiny shapes
# --------------------------------------------------------------------------
def _brute_topk(l, k):
    """The unique k-subset whose members all beat all non-members under the
    order (value descending, index ascending); slots sorted by that order."""
    E = len(l)
    better = lambda a, b: (l[a] > l[b]) or (l[a] == l[b] and a < b)
    found = []
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if all(better(a, b) for a in S for b in rest):
            found.append(S)
    assert len(found) == 1
    S = list(found[0])
    # order slots: repeatedly the member that beats all the others left
    out = []
    while S:
        top = [a for a in S if all(a == b or better(a, b) for b in S)][0]
        out.append(top)
        S.remove(top)
    return out


def check_topk_bruteforce():
    rng = _rng(11)
    for trial in range(60):
        E = int(rng.integers(2, 9))
        k = int(rng.integers(1, E + 1))
        n = 5
        if trial % 3 == 0:   # many exact ties
            lg = rng.integers(-2, 3, size=(n, E)).astype(np.float64)
        else:
            lg = rng.standard_normal((n, E))
        for norm in (True, False):
            idx, w, gap = O.topk_softmax(lg, E, k, norm)
            for t in range(n):
                ref = _brute_topk(list(lg[t]), k)
                assert list(idx[t]) == ref, (lg[t], k, idx[t], ref)
                if norm:
                    ref_w = softmax(lg[t, ref])
                else:
                    ref_w = softmax(lg[t])[ref]
                np.testing.assert_allclose(w[t], ref_w, rtol=1e-13, atol=1e-15)
                srt = sorted(lg[t], reverse=True)
                m = min(k + 1, E)
                ref_gap = min((srt[i] - srt[i + 1] for i in range(m - 1)), default=math.inf)
                assert gap[t] == ref_gap


def test_topk_bruteforce(orc):
    check_topk_bruteforce()


def check_topk_wide_blocks():
    """256 experts across several vector-unit-wide blocks must be able to
    select expert 255 (simulator page: DeepSeek-V3 selects expert 255)."""
    rng = _rng(3)
    for E, k in [(16, 1), (60, 4), (64, 6), (128, 8), (256, 8), (32, 4)]:
        lg = rng.standard_normal((4, E))
        lg[0, E - 1] = 10.0
        lg[1, :] = 0.0                     # all tied: lowest indices win
        idx, w, _ = O.topk_softmax(lg, E, k, True)
        assert idx[0, 0] == E - 1
        assert list(idx[1]) == list(range(k))
        np.testing.assert_allclose(w[1], np.full(k, 1.0 / k), rtol=1e-15)
        for t in (2, 3):
            assert list(idx[t]) == list(np.argsort(-lg[t], kind="stable")[:k])


def test_topk_wide_blocks(orc):
    check_topk_wide_blocks()


# --------------------------------------------------------------------------
# grouping (Fused MoE Kernel Notes)
# --------------------------------------------------------------------------
def check_grouping_golden():
    for c in _golden("grouping_examples.json")["cases"]:
        idx = np.tile(np.array(c["slot_experts"], dtype=np.int32), (c["tokens"], 1))
        counts, offsets, sidx, row_token = O.permute(idx, c["num_experts"])
        assert list(counts) == c["counts"]
        assert offsets[-1] == c["tokens"] * c["topk"]
        assert sorted(sidx.ravel().tolist()) == list(range(c["tokens"] * c["topk"]))


def test_grouping_golden(orc):
    check_grouping_golden()


def check_permute_bruteforce():
    rng = _rng(5)
    for trial in range(30):
        T = int(rng.integers(1, 40))
        E = int(rng.integers(1, 9))
        k = int(rng.integers(1, 5))
        idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
        if trial % 5 == 0:
            idx[:] = 0
        counts, offsets, sidx, row_token = O.permute(idx, E)
        pairs = sorted((int(idx[t, s]), t, s) for t in range(T) for s in range(k))
        for r, (e, t, s) in enumerate(pairs):
            assert sidx[t, s] == r
            assert row_token[r] == t
        assert list(counts) == [int((idx == e).sum()) for e in range(E)]
        assert list(offsets) == [0] + list(np.cumsum(counts))


def test_permute_bruteforce(orc):
    check_permute_bruteforce()


def test_permute_rejects_bad_route(orc):
    with pytest.raises(ValueError):
        O.permute(np.array([[0, 3]], dtype=np.int32), 3)


# --------------------------------------------------------------------------
# expert FFN and combine
# --------------------------------------------------------------------------
def _t64(a):
    return torch.as_tensor(np.asarray(a, dtype=np.float64))


def _swiglu_torch(x, wg, wu, wd):
    """Textbook SwiGLU MLP, torch fp64 library ops: down(silu(gate x) * up x)."""
    return F.linear(F.silu(F.linear(x, wg)) * F.linear(x, wu), wd)


def _rand_layer(seed, T, H, E, I, I_sh, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: (torch.randn(*s, generator=g) / math.sqrt(s[-1])).to(dtype)
    d = dict(x=torch.randn(T, H, generator=g).to(dtype), w_gate=r(E, I, H),
             w_up=r(E, I, H), w_down=r(E, H, I))
    if I_sh:
        d.update(sh_gate=r(I_sh, H), sh_up=r(I_sh, H), sh_down=r(H, I_sh))
    return d


def check_single_expert_textbook():
    """E = 1, k = 1, weight 1: the layer is one SwiGLU MLP.  H != I so a
    transposed operand cannot pass."""
    for dtype in (torch.float32, torch.bfloat16):
        L = _rand_layer(1, T=7, H=24, E=1, I=40, I_sh=0, dtype=dtype)
        idx = np.zeros((7, 1), np.int32)
        y = O.moe_ffn(L["x"], idx, np.ones((7, 1)), None, L["w_gate"], L["w_up"],
                      L["w_down"])
        ref = _swiglu_torch(L["x"].double(), L["w_gate"][0].double(), L["w_up"][0].double(),
                            L["w_down"][0].double())
        np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_single_expert_textbook(orc):
    check_single_expert_textbook()


def check_dense_masked_form():
    """Dense all-expert form (every expert evaluated, each scaled by its route
    value masked by the k-th-largest threshold; the persistent dense-expert
    path of the Spyre adapter page) equals the routed oracle on tie-free,
    duplicate-free inputs, for both weight conventions and with a shared
    expert, gated and ungated."""
    T, H, E, k, I, I_sh = 9, 20, 6, 2, 12, 16
    L = _rand_layer(2, T, H, E, I, I_sh)
    x = L["x"].double()
    g = torch.Generator().manual_seed(9)
    wr = (torch.randn(E + 1, H, generator=g) / math.sqrt(H)).float()
    for norm, gated in [(True, False), (False, True), (False, False), (True, True)]:
        lg = x @ wr.double().T
        probs = torch.softmax(lg[:, :E], dim=1)
        kth = torch.topk(probs, k, dim=1).values[:, -1:]
        route = torch.where(probs >= kth, probs, torch.zeros_like(probs))
        if norm:
            route = route / route.sum(1, keepdim=True)
        dense = torch.zeros(T, H, dtype=torch.float64)
        for e in range(E):
            ye = _swiglu_torch(x, L["w_gate"][e].double(), L["w_up"][e].double(),
                               L["w_down"][e].double())
            dense += route[:, e:e + 1] * ye
        sh = _swiglu_torch(x, L["sh_gate"].double(), L["sh_up"].double(),
                           L["sh_down"].double())
        gate = torch.sigmoid(lg[:, E:E + 1]) if gated else 1.0
        dense += gate * sh
        olg = O.router_logits(L["x"], wr)
        np.testing.assert_allclose(olg, lg.numpy(), rtol=1e-12, atol=1e-12)
        idx, w, _ = O.topk_softmax(olg, E, k, norm)
        og = O.sigmoid(olg[:, E]) if gated else None
        y = O.moe_ffn(L["x"], idx, w, og, L["w_gate"], L["w_up"], L["w_down"],
                      L["sh_gate"], L["sh_up"], L["sh_down"])
        np.testing.assert_allclose(y, dense.numpy(), rtol=1e-11, atol=1e-11)


def test_dense_masked_form(orc):
    check_dense_masked_form()


def check_all_duplicate_closed_form():
    """Every slot on expert 0 with weight 1/k: y = shared(x) + expert_0(x), and
    the grouping is one group of T*k rows (Duplicate top-k routes)."""
    T, H, E, k, I, I_sh = 10, 16, 4, 6, 8, 12
    L = _rand_layer(3, T, H, E, I, I_sh, dtype=torch.bfloat16)
    idx = np.zeros((T, k), np.int32)
    w = np.full((T, k), 1.0 / k)
    y = O.moe_ffn(L["x"], idx, w, None, L["w_gate"], L["w_up"], L["w_down"],
                  L["sh_gate"], L["sh_up"], L["sh_down"])
    x = L["x"].double()
    ref = _swiglu_torch(x, L["w_gate"][0].double(), L["w_up"][0].double(),
                        L["w_down"][0].double())
    ref += _swiglu_torch(x, L["sh_gate"].double(), L["sh_up"].double(), L["sh_down"].double())
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
    counts, offsets, sidx, _ = O.permute(idx, E)
    assert list(counts) == [T * k, 0, 0, 0]
    assert list(sidx.ravel()) == list(range(T * k))


def test_all_duplicate_closed_form(orc):
    check_all_duplicate_closed_form()


def check_shared_fusion_identity():
    """n_shared experts stored as one MLP of width moe_inter * n_shared equal
    the sum of the individual experts (compiler page, Group C), to fp64
    rounding -- not bitwise."""
    T, H, I, n = 5, 16, 8, 3
    parts = [_rand_layer(10 + j, T, H, 1, I, 0) for j in range(n)]
    x = parts[0]["x"]
    fused_g = torch.cat([p["w_gate"][0] for p in parts], 0)
    fused_u = torch.cat([p["w_up"][0] for p in parts], 0)
    fused_d = torch.cat([p["w_down"][0] for p in parts], 1)
    zero_idx = np.zeros((T, 1), np.int32)
    zero_w = np.zeros((T, 1))
    dummy = parts[0]
    y_fused = O.moe_ffn(x, zero_idx, zero_w, None, dummy["w_gate"], dummy["w_up"],
                        dummy["w_down"], fused_g, fused_u, fused_d)
    y_sum = np.zeros_like(y_fused)
    for p in parts:
        y_sum += O.moe_ffn(x, zero_idx, zero_w, None, dummy["w_gate"], dummy["w_up"],
                           dummy["w_down"], p["w_gate"][0], p["w_up"][0], p["w_down"][0])
    np.testing.assert_allclose(y_fused, y_sum, rtol=1e-12, atol=1e-13)
    ref = _swiglu_torch(x.double(), fused_g.double(), fused_u.double(), fused_d.double())
    np.testing.assert_allclose(y_fused, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_shared_fusion_identity(orc):
    check_shared_fusion_identity()


def check_gate():
    """sigmoid(0) = 1/2 exactly; with a zero gate weight the gated layer is the
    ungated layer minus half the shared output.  Logits of +-16 saturate the
    gate to exactly 1.0 once rounded to bf16 (simulator page, Tests), but not in
    fp64."""
    assert O.sigmoid(np.array([0.0]))[0] == 0.5
    s = O.sigmoid(np.array([16.0, -16.0, 3.0, -2.5]))
    np.testing.assert_allclose(s, expit([16.0, -16.0, 3.0, -2.5]), rtol=1e-15)
    assert s[0] < 1.0
    assert torch.tensor(s[0]).to(torch.bfloat16).item() == 1.0
    T, H, E, k, I, I_sh = 6, 16, 4, 2, 8, 12
    L = _rand_layer(4, T, H, E, I, I_sh)
    rng = _rng(4)
    idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
    w = rng.uniform(0.1, 1.0, size=(T, k))
    args = (L["w_gate"], L["w_up"], L["w_down"], L["sh_gate"], L["sh_up"], L["sh_down"])
    y1 = O.moe_ffn(L["x"], idx, w, None, *args)
    yh = O.moe_ffn(L["x"], idx, w, np.full(T, 0.5), *args)
    sh = _swiglu_torch(L["x"].double(), L["sh_gate"].double(), L["sh_up"].double(),
                       L["sh_down"].double()).numpy()
    np.testing.assert_allclose(yh, y1 - 0.5 * sh, rtol=1e-11, atol=1e-12)
    z = rng.standard_normal(T)
    yg = O.moe_ffn(L["x"], idx, w, O.sigmoid(z), *args)
    np.testing.assert_allclose(yg, y1 - (1 - expit(z))[:, None] * sh, rtol=1e-11, atol=1e-12)


def test_gate(orc):
    check_gate()


def check_combine_is_k_sum():
    """The combine is the per-token sum over the k slots of weight times the
    slot's expert output (the Spyre adapter's decode combine, a K-axis sum),
    duplicates included."""
    T, H, E, k, I = 6, 16, 3, 4, 8
    L = _rand_layer(5, T, H, E, I, 0)
    rng = _rng(6)
    idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
    idx[0, :] = 1                                            # duplicate routes
    w = rng.uniform(0.1, 1.0, size=(T, k))
    y = O.moe_ffn(L["x"], idx, w, None, L["w_gate"], L["w_up"], L["w_down"])
    x = L["x"].double()
    ref = torch.zeros(T, H, dtype=torch.float64)
    for t in range(T):
        for s in range(k):
            e = int(idx[t, s])
            ref[t] += w[t, s] * _swiglu_torch(x[t:t + 1], L["w_gate"][e].double(),
                                              L["w_up"][e].double(),
                                              L["w_down"][e].double())[0]
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_combine_is_k_sum(orc):
    check_combine_is_k_sum()


def check_expert_strides_and_tokens():
    """Merged fc1 (gate and up rows of one expert adjacent, stride 2*I*H) and a
    token subset give the same result as split fc1 over all tokens."""
    T, H, E, k, I = 8, 16, 3, 2, 8
    L = _rand_layer(7, T, H, E, I, 0, dtype=torch.bfloat16)
    rng = _rng(8)
    idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
    w = rng.uniform(0.1, 1.0, size=(T, k))
    y = O.moe_ffn(L["x"], idx, w, None, L["w_gate"], L["w_up"], L["w_down"])
    merged = torch.cat([L["w_gate"], L["w_up"]], dim=1).contiguous()   # [E, 2I, H]
    up_view = merged.view(-1)[I * H:]
    tok = np.array([6, 1, 3])
    ym = O.moe_ffn(L["x"], idx[tok], w[tok], None, merged, up_view, L["w_down"],
                   tokens=tok, gate_stride=2 * I * H, up_stride=2 * I * H, moe_inter=I)
    np.testing.assert_allclose(ym, y[tok], rtol=0, atol=0)
    # split gate (stride I*H) next to the merged buffer's up half (stride 2*I*H)
    yx = O.moe_ffn(L["x"], idx, w, None, L["w_gate"], up_view, L["w_down"],
                   gate_stride=I * H, up_stride=2 * I * H, moe_inter=I)
    np.testing.assert_allclose(yx, y, rtol=0, atol=0)


def test_expert_strides_and_tokens(orc):
    check_expert_strides_and_tokens()


def test_workload_gate_stays_interior():
    """The Qwen2-MoE-shaped workload's gate weight keeps sigmoid(z) strictly
    inside (0, 1) after bf16 rounding, so an unapplied gate cannot pass."""
    from mixture_experts_ffn_04_gb300 import workloads as W
    wl = W.small(W.QWEN2_MOE, T=256)
    d = W.make_inputs(wl, seed=0, with_experts=False)
    z = (d["x"].double() @ d["w_router"][wl.E].double())
    g = torch.sigmoid(z).to(torch.bfloat16).float()
    assert bool(((g > 0) & (g < 1)).all())


# ---------------------------------------------------------------------------
# Input preparation: activation rounding, input RMSNorm, residual
# ("MoE: shared experts, arbitrary V_TOPK expert shapes, and an enforced
# stage-marker contract", Group E: residual_setup = residual copy + input
# RMSNorm + norm-weight multiply)
# ---------------------------------------------------------------------------
def _bf16_nearest_exact(v):
    """Nearest bf16 value to v with ties to even, by exact rational
    arithmetic (Fraction) -- an independent statement of the rounding rule."""
    from fractions import Fraction
    if v == 0:
        return 0.0
    a = Fraction(abs(v))
    if a < Fraction(2) ** -126:
        q = Fraction(2) ** -133
    else:
        e = 0
        while Fraction(2) ** (e + 1) <= a:
            e += 1
        while Fraction(2) ** e > a:
            e -= 1
        q = Fraction(2) ** (e - 7)        # 8 significant bits over [2^e, 2^(e+1))
    r = round(a / q) * q                  # Python rounds Fractions half to even
    if r > Fraction(255) * Fraction(2) ** 120:
        return math.copysign(math.inf, v)
    return math.copysign(float(r), v)


def check_round_act():
    rng = _rng(21)
    vals = list(rng.standard_normal(400) * 10.0 ** rng.integers(-6, 6, size=400))
    one = 1.0
    for m in range(128, 256, 7):           # exact midpoints and just either side
        mid = (m + 0.5) / 128.0
        vals += [mid, mid + 2 ** -30, mid - 2 ** -30, -mid]
    vals += [1 + 2 ** -8 + 2 ** -30, one, 2.0 ** -130, 3.3e-39, 3.0e38, 3.4e38, -7.0e-41]
    for v in vals:
        got = O.round_act(v, "bf16")
        want = _bf16_nearest_exact(v)
        assert got == want, (v, got, want)
        assert O.round_act(v, "f32") == float(np.float32(v)), v


def test_round_act(orc):
    check_round_act()


def check_rmsnorm_closed_forms():
    H = 16
    w1 = torch.ones(H, dtype=torch.bfloat16)
    # constant rows: x / |x| = sign(x), for eps = 0
    x = torch.tensor([[3.0] * H, [-0.25] * H], dtype=torch.bfloat16)
    out = O.rmsnorm(x, w1, 0.0).float()
    assert torch.equal(out, torch.tensor([[1.0] * H, [-1.0] * H]))
    # alternating +-a: rms = a; the norm weight multiplies per column
    x = torch.tensor([[5.0, -5.0] * (H // 2)], dtype=torch.bfloat16)
    w = torch.tensor([0.5, 2.0, -1.0, 1.5] * (H // 4), dtype=torch.bfloat16)
    out = O.rmsnorm(x, w, 0.0).float()
    assert torch.equal(out, torch.tensor([[1.0, -1.0] * (H // 2)]) * w.float())
    # eps enters under the square root: x = 1 everywhere, eps = 3 -> 1/2
    out = O.rmsnorm(torch.ones(1, H, dtype=torch.bfloat16), w1, 3.0).float()
    assert torch.equal(out, torch.full((1, H), 0.5))
    # scale invariance (eps = 0, power-of-two scale: exact)
    x = torch.from_numpy(_rng(22).standard_normal((3, H)).astype(np.float32)).to(torch.bfloat16)
    a = O.rmsnorm(x, w1, 0.0)
    b = O.rmsnorm(x * 8.0, w1, 0.0)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_rmsnorm_closed_forms(orc):
    check_rmsnorm_closed_forms()


def check_rmsnorm_high_precision():
    """Random rows against a 60-digit evaluation of the definition, rounded
    by the exact rule above: bit for bit."""
    import mpmath
    mpmath.mp.dps = 60
    rng = _rng(23)
    T, H = 5, 24
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy((1 + 0.2 * rng.standard_normal(H)).astype(np.float32)).to(torch.bfloat16)
    eps = 1e-3
    got = O.rmsnorm(x, w, eps).float().numpy()
    xs, ws = x.float().numpy().astype(np.float64), w.float().numpy().astype(np.float64)
    for t in range(T):
        ms = mpmath.fsum([mpmath.mpf(float(v)) ** 2 for v in xs[t]]) / H
        inv = 1 / mpmath.sqrt(ms + mpmath.mpf(eps))
        for h in range(H):
            exact = mpmath.mpf(float(xs[t, h])) * inv * mpmath.mpf(float(ws[h]))
            want = _bf16_nearest_exact(float(exact))
            # float(exact) is within 2^-53 relative; no case lands that close
            # to a bf16 midpoint here (checked below)
            q = abs(want) * 2.0 ** -8
            assert abs(abs(float(exact)) - abs(want)) < q, (t, h)
            assert got[t, h] == want, (t, h, got[t, h], want)


def test_rmsnorm_high_precision(orc):
    check_rmsnorm_high_precision()


def check_residual_identity():
    """y = x + MoE(rmsnorm(x)): with every expert weight zero the output is x
    exactly; otherwise the residual run minus x is the run without it."""
    import dataclasses
    from mixture_experts_ffn_04_gb300 import workloads as W
    wl = W.small(W.GEMMA4_26B_A4B, T=12, H=64, I=32, E=8, k=2)
    inp = W.make_inputs(wl, seed=4)
    zero = dict(inp, w_gate=torch.zeros_like(inp["w_gate"]),
                w_up=torch.zeros_like(inp["w_up"]), w_down=torch.zeros_like(inp["w_down"]))
    y0 = O.forward(wl, zero)["y"]
    np.testing.assert_array_equal(y0, inp["x"].double().numpy())
    y = O.forward(wl, inp)["y"]
    ynr = O.forward(dataclasses.replace(wl, residual=False), inp)["y"]
    np.testing.assert_allclose(y - inp["x"].double().numpy(), ynr, rtol=0, atol=1e-12)
    # the routed part sees the normalised input, not x
    xn = O.rmsnorm(inp["x"], inp["norm_weight"], wl.norm_eps)
    r = O.route(wl, dict(inp, x=xn, norm_weight=None),
                xin=xn)
    ym = O.moe_ffn(xn, r["idx"], r["weights"], None, inp["w_gate"], inp["w_up"],
                   inp["w_down"])
    np.testing.assert_allclose(ynr, ym, rtol=0, atol=0)


def test_residual_identity(orc):
    check_residual_identity()


def check_hash_route():
    """Hash-MoE lookup ("Fused MoE Kernel Notes", Duplicate top-k routes): a
    hand-worked table, an out-of-range token id, and the notes' example --
    128 tokens whose lookup sends both slots to expert 0 form one group of
    256 rows."""
    table = np.array([[3, 1], [2, 2], [0, 3]], dtype=np.int32)   # vocab 3, k 2
    idx, w = O.hash_route([2, 1, 0, 7, 1], table, 2)
    assert idx.tolist() == [[0, 3], [2, 2], [3, 1], [-1, -1], [2, 2]]
    assert w.shape == (5, 2) and (w == 0.5).all()
    idx, w = O.hash_route(np.arange(128) % 5, np.zeros((5, 2), np.int32), 2)
    counts, offsets, sidx, _ = O.permute(idx, 4)
    assert counts.tolist() == [256, 0, 0, 0] and offsets.tolist() == [0, 256, 256, 256, 256]
    assert sidx[127].tolist() == [254, 255]
    _, w3 = O.hash_route([0], np.zeros((1, 3), np.int32), 3)
    assert w3[0, 0] == 1.0 / 3.0


def test_hash_route():
    check_hash_route()
