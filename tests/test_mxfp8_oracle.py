"""Pins of the MXFP8 oracle (oracle/mxfp8.py) to things other than itself:

* every e4m3 code decodes to torch's float8_e4m3fn value (a library
  routine), NaN codes included;
* round-to-nearest-even onto e4m3 agrees with torch's conversion on random
  in-range values and on exact midpoints between neighbouring codes;
* the pages' statement ("MoE: shared experts, arbitrary V_TOPK expert shapes,
  and an enforced stage-marker contract", Tests): MXFP8-representable inputs
  make quantisation the identity -- including blocks whose largest value has
  the mantissa 1.875;
* the block scale by brute force: the smallest power of two X over all
  candidates with max|V| / X <= 448;
* packing keeps codes then scales;
* a block holding a NaN or an infinity is stored as NaN (the reading taken
  for non-finite weights): scale 0xFF, which torch's e8m0 type also decodes
  to NaN, and e4m3 codes that torch decodes to NaN; the finite blocks of the
  same row quantise as they do alone.
Each check takes the module, so the mutation test can rerun them."""
import importlib.util

import numpy as np
import pytest
import torch

from oracle import mxfp8 as MX


def check_decode_matches_torch(X=MX):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([X.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])


def check_rounding_matches_torch(X=MX):
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(-440, 440, 4000), rng.standard_normal(4000) * 0.01,
                        rng.standard_normal(2000) * 2.0 ** -8])
    vals = np.array(sorted({X.e4m3_value(c) for c in range(0x7F)}))
    mids = (vals[:-1] + vals[1:]) / 2.0   # exact in float64: ties
    v = np.concatenate([v, mids, -mids]).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(v).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got_a = X.round_e4m3_array(v)
    assert np.array_equal(got_a, ref), np.nonzero(got_a != ref)[0][:5]
    got_s = np.array([X.round_e4m3(t) for t in v[::17]], dtype=np.uint8)
    assert np.array_equal(got_s, ref[::17])
    assert X.round_e4m3(1000.0) == 0x7E and X.round_e4m3(-1000.0) == 0xFE


def check_representable_is_identity(X=MX):
    rng = np.random.default_rng(1)
    N, K = 64, 64
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    codes = rng.choice(finite, size=(N, K)).astype(np.uint8)
    codes[::5, 0] = 0x77   # 1.875 * 2^7 = 240: the mantissa that breaks the floor rule
    scales = rng.integers(100, 140, size=(N, K // 8)).astype(np.uint8)
    v = X.dequantize(codes, scales)
    c2, s2 = X.quantize(v, K)
    assert np.array_equal(X.dequantize(c2, s2), v)


def check_scale_bruteforce(X=MX):
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((16, 64)) * np.exp2(rng.integers(-12, 6, size=(16, 1)))).astype(np.float32)
    _, s = X.quantize(w, 64)
    blocks = w.astype(np.float64).reshape(16, 8, 8)
    for n in range(16):
        for b in range(8):
            amax = np.max(np.abs(blocks[n, b]))
            best = None
            for e in range(-140, 140):
                if amax / 2.0 ** e <= 448.0:
                    best = e
                    break
            assert s[n, b] == best + 127, (n, b, s[n, b], best)


def check_pack_layout(X=MX):
    c = np.arange(16, dtype=np.uint8).reshape(2, 8)
    s = np.array([[120], [130]], np.uint8)
    buf = X.pack(c, s)
    assert buf.tolist() == list(range(16)) + [120, 130]
    c2, s2 = X.unpack(buf, 2, 8)
    assert np.array_equal(c2, c) and np.array_equal(s2, s)


def check_nonfinite_blocks_are_nan(X=MX):
    rng = np.random.default_rng(3)
    w = rng.standard_normal((4, 32))
    w[0, 3], w[1, 9], w[2, 30] = np.inf, np.nan, -np.inf
    c, s = X.quantize(w, 32)
    bad = {(0, 0), (1, 1), (2, 3)}
    for n in range(4):
        for b in range(4):
            if (n, b) in bad:
                assert s[n, b] == 0xFF and np.all(c[n, 8 * b:8 * b + 8] == 0x7F)
            else:
                c1, s1 = X.quantize(w[n, 8 * b:8 * b + 8], 8)
                assert s[n, b] == s1[0, 0] and np.array_equal(c[n, 8 * b:8 * b + 8], c1[0])
    v = X.dequantize(c, s)
    assert np.array_equal(np.isnan(v), np.repeat(s == 0xFF, 8, axis=1))
    code = torch.tensor([0x7F], dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    assert torch.isnan(code).all()
    if hasattr(torch, "float8_e8m0fnu"):
        sc = torch.tensor([0xFF], dtype=torch.uint8).view(torch.float8_e8m0fnu).float()
        assert torch.isnan(sc).all()


CHECKS = [check_decode_matches_torch, check_rounding_matches_torch,
          check_representable_is_identity, check_scale_bruteforce, check_pack_layout,
          check_nonfinite_blocks_are_nan]


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_mxfp8_oracle_pin(check):
    check()


MUTANTS = [
    ("OCP floor rule for the scale", "return E - 8 + (1 if amax > 1.75 * 2.0 ** E else 0)",
     "return E - 8"),
    ("ties away from zero", "pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))",
     "pick = np.where(dlo < dhi, lo, hi)"),
    ("non-finite blocks quantised like finite ones", "byte = np.where(bad, 255, byte)",
     "byte = byte"),
    ("subnormals scaled like normals", "return s * (m / 8.0) * 2.0 ** -6",
     "return s * (1.0 + m / 8.0) * 2.0 ** -7"),
]


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mxfp8_mutant_is_caught(tmp_path, name, orig, mut):
    src = open(MX.__file__).read()
    assert src.count(orig) == 1, orig
    p = tmp_path / "mutant_mxfp8.py"
    p.write_text(src.replace(orig, mut))
    spec = importlib.util.spec_from_file_location("mutant_mxfp8", str(p))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    caught = []
    for chk in CHECKS:
        try:
            chk(mod)
        except (AssertionError, ValueError, IndexError):
            caught.append(chk.__name__)
    assert caught, "mutant %r passed every MXFP8 pin" % name
