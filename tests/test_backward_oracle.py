"""Pins of the fp64 backward oracle (oracle/moe_backward.py) to things other
than itself:

* central differences of the C forward oracle (a separate program, pinned in
  test_oracle_pins.py): the directional derivative of sum(dy * y) along a
  random direction of each input must equal <gradient, direction>;
* homogeneity: y is linear in w, in each W_down[e] and in each W_up[e], so
  <w, dw> = <W_down, dW_down> = <W_up, dW_up> = <dy, y> (Euler's theorem);
* a symbolic derivative (sympy) of a one-token, one-expert case;
* duplicate routes ("Fused MoE Kernel Notes", Duplicate top-k routes): two
  slots of a token on one expert with weights w1, w2 give the gradients of a
  single slot with weight w1 + w2, and the same dw in both slots;
* an expert no pair routes to gets zero weight gradients.

Each check takes the module under test, so the mutation test below can run the
same checks against mutated copies of it."""
import importlib.util
import os

import numpy as np
import pytest
import torch

from oracle import moe_backward as MB
from oracle import oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def _case(seed=0, T=7, H=16, I=8, E=4, k=2, dup=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g) * 0.7
    wg = torch.randn(E, I, H, generator=g) * 0.4
    wu = torch.randn(E, I, H, generator=g) * 0.4
    wd = torch.randn(E, H, I, generator=g) * 0.4
    idx = torch.randint(0, E - 1, (T, k), generator=g).to(torch.int32)   # expert E-1 unused
    if dup:
        idx[0, :] = 1   # one token with both slots on one expert
    w = torch.rand(T, k, generator=g, dtype=torch.float64) + 0.1
    dy = torch.randn(T, H, generator=g, dtype=torch.float64)
    return dict(x=x, wg=wg, wu=wu, wd=wd, idx=idx.numpy(), w=w.numpy(), dy=dy.numpy())


def _loss(c, x=None, w=None, wg=None, wu=None, wd=None):
    """sum(dy * y) from the C forward oracle (fp64 arithmetic, no rounding)."""
    y = O.moe_ffn(c["x"] if x is None else x, c["idx"], c["w"] if w is None else w, None,
                  c["wg"] if wg is None else wg, c["wu"] if wu is None else wu,
                  c["wd"] if wd is None else wd)
    return float(np.sum(c["dy"] * y))


def _fd(c, name, grad, eps=1e-4, seed=1):
    """Central difference of the C forward along a random direction v of input
    `name`; fp32 inputs move by the exact difference of the rounded points."""
    rng = np.random.default_rng(seed)
    base = c[name]
    if isinstance(base, torch.Tensor):
        v = torch.from_numpy(rng.standard_normal(tuple(base.shape))).float()
        plus, minus = base + eps * v, base - eps * v
        step = plus.double().numpy() - minus.double().numpy()
    else:
        v = rng.standard_normal(base.shape)
        plus, minus = base + eps * v, base - eps * v
        step = plus - minus
    d = _loss(c, **{name: plus}) - _loss(c, **{name: minus})
    return d, float(np.sum(grad * step))


def check_central_differences(B=MB):
    # the second case is square (H == I), where a transposed operand still fits
    for seed, H, I in ((0, 16, 8), (3, 8, 8)):
        c = _case(seed, H=H, I=I)
        gr = B.backward(c["x"], c["idx"], c["w"], c["wg"], c["wu"], c["wd"], c["dy"])
        for name, key in (("x", "dx"), ("w", "dw"), ("wg", "dw_gate"), ("wu", "dw_up"),
                          ("wd", "dw_down")):
            fd, an = _fd(c, name, gr[key], seed=seed + 1)
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (seed, name, fd, an)


def check_forward_matches_c_oracle(B=MB):
    c = _case(5)
    y, _ = B.forward(c["x"], c["idx"], c["w"], c["wg"], c["wu"], c["wd"])
    yc = O.moe_ffn(c["x"], c["idx"], c["w"], None, c["wg"], c["wu"], c["wd"])
    assert np.allclose(y, yc, rtol=1e-12, atol=1e-12)


def check_homogeneity(B=MB):
    c = _case(7)
    gr = B.backward(c["x"], c["idx"], c["w"], c["wg"], c["wu"], c["wd"], c["dy"])
    yc = O.moe_ffn(c["x"], c["idx"], c["w"], None, c["wg"], c["wu"], c["wd"])
    ref = float(np.sum(c["dy"] * yc))
    for v, dv in ((c["w"], gr["dw"]), (c["wd"].double().numpy(), gr["dw_down"]),
                  (c["wu"].double().numpy(), gr["dw_up"])):
        assert abs(float(np.sum(v * dv)) - ref) <= 1e-10 * max(1.0, abs(ref))


def check_symbolic(B=MB):
    sp = pytest.importorskip("sympy")
    x0, x1, wgt = sp.symbols("x0 x1 w")
    g0, g1, u0, u1, d0, d1 = sp.symbols("g0 g1 u0 u1 d0 d1")
    a = g0 * x0 + g1 * x1
    b = u0 * x0 + u1 * x1
    h = a / (1 + sp.exp(-a)) * b
    y = [wgt * d0 * h, wgt * d1 * h]
    vals = {x0: sp.Rational(3, 5), x1: sp.Rational(-7, 10), wgt: sp.Rational(2, 3),
            g0: sp.Rational(1, 2), g1: sp.Rational(-1, 4), u0: sp.Rational(3, 4),
            u1: sp.Rational(1, 3), d0: sp.Rational(-6, 5), d1: sp.Rational(2, 5)}
    dyv = [sp.Rational(5, 4), sp.Rational(-3, 8)]
    L = dyv[0] * y[0] + dyv[1] * y[1]
    num = lambda s: float(sp.N(sp.diff(L, s).subs(vals), 30))
    f = lambda s: float(vals[s])
    x = np.array([[f(x0), f(x1)]])
    gr = B.backward(x, np.zeros((1, 1), np.int32), np.array([[f(wgt)]]),
                    np.array([[[f(g0), f(g1)]]]), np.array([[[f(u0), f(u1)]]]),
                    np.array([[[f(d0)], [f(d1)]]]), np.array([[float(d) for d in dyv]]))
    pairs = [(gr["dx"][0, 0], x0), (gr["dx"][0, 1], x1), (gr["dw"][0, 0], wgt),
             (gr["dw_gate"][0, 0, 0], g0), (gr["dw_gate"][0, 0, 1], g1),
             (gr["dw_up"][0, 0, 0], u0), (gr["dw_up"][0, 0, 1], u1),
             (gr["dw_down"][0, 0, 0], d0), (gr["dw_down"][0, 1, 0], d1)]
    for got, s in pairs:
        assert abs(got - num(s)) <= 1e-13 * max(1.0, abs(num(s))), (s, got, num(s))


def check_duplicate_routes(B=MB):
    c = _case(9, k=2, dup=False)
    T = c["x"].shape[0]
    idx2 = np.zeros((T, 2), np.int32)
    w2 = c["w"]
    idx1 = np.zeros((T, 1), np.int32)
    w1 = (w2[:, 0] + w2[:, 1])[:, None]
    g2 = B.backward(c["x"], idx2, w2, c["wg"], c["wu"], c["wd"], c["dy"])
    g1 = B.backward(c["x"], idx1, w1, c["wg"], c["wu"], c["wd"], c["dy"])
    for key in ("dx", "dw_gate", "dw_up", "dw_down"):
        assert np.allclose(g2[key], g1[key], rtol=1e-12, atol=1e-12), key
    assert np.allclose(g2["dw"][:, 0], g1["dw"][:, 0], rtol=1e-12, atol=1e-12)
    assert np.allclose(g2["dw"][:, 1], g1["dw"][:, 0], rtol=1e-12, atol=1e-12)
    assert np.all(np.isfinite(g2["dx"]))


def check_unused_expert_has_zero_grads(B=MB):
    c = _case(11)
    gr = B.backward(c["x"], c["idx"], c["w"], c["wg"], c["wu"], c["wd"], c["dy"])
    E = c["wg"].shape[0]
    assert not np.any(c["idx"] == E - 1)
    for key in ("dw_gate", "dw_up", "dw_down"):
        assert np.all(gr[key][E - 1] == 0.0)
        assert np.any(gr[key][1] != 0.0)


def check_group_weight_grads_bruteforce(B=MB):
    """The grouped weight-gradient GEMM by explicit triple loops on tiny
    inputs, with an empty group and a group of one row."""
    rng = np.random.default_rng(4)
    a = rng.standard_normal((7, 3))
    b = rng.standard_normal((7, 2))
    offsets = [0, 3, 3, 4, 7]
    got = B.group_weight_grads(a, b, offsets)
    assert got.shape == (4, 3, 2)
    for g in range(4):
        for i in range(3):
            for j in range(2):
                ref = 0.0
                for r in range(offsets[g], offsets[g + 1]):
                    ref += a[r, i] * b[r, j]
                assert abs(got[g, i, j] - ref) <= 1e-14 * max(1.0, abs(ref)), (g, i, j)
    assert np.all(got[1] == 0.0)


CHECKS = [check_central_differences, check_forward_matches_c_oracle, check_homogeneity,
          check_symbolic, check_duplicate_routes, check_unused_expert_has_zero_grads,
          check_group_weight_grads_bruteforce]


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_backward_oracle_pin(check):
    check()


# (name, original text, mutated text): plausible slips in the backward, each of
# which the checks above must catch.
MUTANTS = [
    ("routing weight not carried by the scattered gradient",
     "dO = W[tok, slot][:, None] * dY[tok]", "dO = dY[tok]"),
    ("silu derivative without its second term",
     "dA = dH * B * sg * (1.0 + A * (1.0 - sg))", "dA = dH * B * sg"),
    ("gate and up gradients swapped", "dB = dH * A * sg", "dB = dH * B * sg"),
    ("down dgrad through the transposed weight", "dH = dO @ Wd[e]", "dH = dO @ Wd[e].T"),
    ("down weight gradient transposed", "dWd[e] = dO.T @ Hh", "dWd[e] = Hh.T @ dO"),
    ("up term dropped from the input gradient", "dXe = dA @ Wg[e] + dB @ Wu[e]", "dXe = dA @ Wg[e]"),
    ("routing-weight gradient from h, not o", "dw[tok, slot] = np.sum(dY[tok] * O, axis=1)",
     "dw[tok, slot] = np.sum(dY[tok][:, :Hh.shape[1]] * Hh, axis=1)"),
    ("gather keeps only the last slot", "np.add.at(dx, tok, dXe)", "dx[tok] = dXe"),
    ("gate weight gradient uses the up input", "dWg[e] = dA.T @ Xe", "dWg[e] = dB.T @ Xe"),
    ("weight-gradient groups off by one row", "r0, r1 = off[g], off[g + 1]",
     "r0, r1 = off[g], off[g + 1] + (1 if g + 1 < G else 0)"),
]


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_backward_mutant_is_caught(tmp_path, name, orig, mut):
    src = open(MB.__file__).read()
    assert src.count(orig) == 1, "mutation site not unique: %r" % orig
    p = tmp_path / "mutant_backward.py"
    p.write_text(src.replace(orig, mut))
    spec = importlib.util.spec_from_file_location("mutant_backward", str(p))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    caught = []
    for chk in CHECKS:
        try:
            chk(mod)
        except (AssertionError, ValueError, IndexError):
            caught.append(chk.__name__)
    assert caught, "mutant %r passed every backward pin" % name
