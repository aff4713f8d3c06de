"""MXFP8 expert weights for the oracle: e4m3 values with one e8m0 scale per
block of 8 along the reduced axis.

TEST INFRASTRUCTURE ONLY (imported by the tests, smoke() and bench.py's
CPU-baseline leg; shares nothing with the CUDA path).

The pages fix the format -- "MoE: shared experts, arbitrary V_TOPK expert
shapes, and an enforced stage-marker contract", the fusion identity: expert
weights are MXFP8, e4m3 with one e8m0 scale per block of 8 along the reduced
axis -- and that MXFP8-representable inputs make quantisation the identity
(ibid., Tests).  They do not give the quantisation rule.  The reading taken
is the one that identity implies: the scale of a block V of 8 values is the
smallest power of two X with max|V| / X <= 448 (the largest e4m3 value), so

    E = floor(log2(max|V|)),  shared = E - 8 + (max|V| > 1.75 * 2^E)
    (0 when V == 0), e8m0 byte = shared + 127 clamped to [0, 254]
    q_i = e4m3(V_i / 2^shared), round to nearest even, saturating at +-448

and the value of a stored weight is e4m3_value(q) * 2^(byte - 127).  The
pages say nothing of non-finite weights; the reading taken is that a block
holding a NaN or an infinity is stored as NaN -- scale byte 0xFF (the e8m0
NaN) and eight e4m3 NaN codes 0x7F -- rather than its finite values being
quantised against a scale that the infinity or NaN decides.  (The OCP
Microscaling rule, shared = floor(log2(max|V|)) - 8, would send a
representable block whose largest value has the mantissa 1.875 to 480 and
saturate it at 448, breaking the identity the pages state.)

Packed layout of one [N, K] matrix: N*K e4m3 bytes (row-major), then N*K/8
e8m0 bytes (row-major [N, K/8]).
"""
from __future__ import annotations

import numpy as np


def e4m3_value(code: int) -> float:
    """Value of an e4m3 (fn) byte: 1 sign, 4 exponent bits (bias 7), 3
    mantissa bits; exponent 0 is subnormal; S.1111.111 is NaN (no infinity)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_VALUES = np.array([e4m3_value(c) for c in range(256)])
_POS_CODES = [c for c in range(0x7F) if c < 0x7F]            # 0x00 .. 0x7E: +0 .. 448
_POS_VALUES = np.array([_VALUES[c] for c in _POS_CODES])


def round_e4m3(v: float) -> int:
    """e4m3 code nearest to v (exact arithmetic in float64 for the values the
    quantiser produces), ties to the even code, |v| > 448 saturating to 448."""
    a = abs(v)
    sign = 0x80 if (v < 0 or (v == 0 and np.signbit(v))) else 0
    if a >= 448.0:
        return sign | 0x7E
    i = int(np.searchsorted(_POS_VALUES, a))   # first value >= a
    if _POS_VALUES[i] == a:
        return sign | _POS_CODES[i]
    lo, hi = _POS_CODES[i - 1], _POS_CODES[i]
    dlo, dhi = a - _VALUES[lo], _VALUES[hi] - a
    if dlo < dhi:
        code = lo
    elif dhi < dlo:
        code = hi
    else:
        code = lo if lo % 2 == 0 else hi
    return sign | code


def block_shared_exponent(amax: float) -> int:
    """Exponent of the smallest power of two X with amax / X <= 448."""
    if amax == 0.0:
        return 0
    m, e = np.frexp(amax)          # amax = m * 2^e, m in [0.5, 1): E = e - 1
    E = int(e) - 1
    return E - 8 + (1 if amax > 1.75 * 2.0 ** E else 0)


def round_e4m3_array(v: np.ndarray) -> np.ndarray:
    """round_e4m3 over an array (same rule, vectorised)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    sign = np.where(np.signbit(v), 0x80, 0).astype(np.int64)
    codes = np.asarray(_POS_CODES, dtype=np.int64)
    i = np.clip(np.searchsorted(_POS_VALUES, a), 1, len(_POS_VALUES) - 1)
    lo, hi = codes[i - 1], codes[i]
    dlo, dhi = a - _POS_VALUES[i - 1], _POS_VALUES[i] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a == _POS_VALUES[i - 1], lo, pick)
    pick = np.where(a >= 448.0, 0x7E, pick)
    return (sign | pick).astype(np.uint8)


def quantize(w, K: int):
    """Quantise rows of K values (K a multiple of 8) into (codes [N, K] uint8,
    scales [N, K/8] uint8)."""
    W = np.asarray(w.detach().cpu().double().numpy() if hasattr(w, "detach") else w,
                   dtype=np.float64).reshape(-1, K)
    N = W.shape[0]
    blocks = W.reshape(N, K // 8, 8)
    bad = ~np.all(np.isfinite(blocks), axis=2)          # blocks stored as NaN
    amax = np.where(bad, 0.0, np.max(np.abs(np.where(np.isfinite(blocks), blocks, 0.0)), axis=2))
    shared = np.vectorize(block_shared_exponent, otypes=[np.int64])(amax)
    byte = np.clip(shared + 127, 0, 254)
    x = np.exp2(byte.astype(np.float64) - 127.0)
    finite = np.where(bad[:, :, None], 0.0, blocks)
    codes = round_e4m3_array((finite / x[:, :, None]).reshape(-1)).reshape(N, K)
    codes = np.where(np.repeat(bad, 8, axis=1), 0x7F, codes).astype(np.uint8)
    byte = np.where(bad, 255, byte)
    return codes, byte.astype(np.uint8)


def dequantize(codes, scales) -> np.ndarray:
    """float64 [N, K] values of quantised rows."""
    c = np.asarray(codes, np.uint8)
    s = np.asarray(scales, np.uint8)
    N, K = c.shape
    x = np.where(s == 255, np.nan, np.exp2(s.astype(np.float64) - 127.0))   # 0xFF: e8m0 NaN
    return _VALUES[c] * np.repeat(x, 8, axis=1)


def pack(codes, scales) -> np.ndarray:
    """The packed bytes of one matrix: codes then scales."""
    return np.concatenate([np.asarray(codes, np.uint8).reshape(-1),
                           np.asarray(scales, np.uint8).reshape(-1)])


def unpack(buf, N: int, K: int):
    b = np.asarray(buf, np.uint8).reshape(-1)
    return b[:N * K].reshape(N, K), b[N * K: N * K + N * K // 8].reshape(N, K // 8)
