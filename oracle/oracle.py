"""Python marshalling for the fp64 MoE oracle in ``moe_oracle.c``.

TEST INFRASTRUCTURE ONLY.  This module (and the C file it loads) is imported
by the test suite, by ``__graft_entry__.smoke()`` and by the CPU-baseline leg
of ``bench.py`` -- nowhere else.  The product library never touches it, and
it imports nothing from the product package: it shares no code with the CUDA
path.  Inputs are CPU torch tensors (fp32 or bf16) or numpy arrays; every
result comes back as float64 / int32 numpy arrays.

The functions follow these passages (page title, section):

* "MoE: shared experts, arbitrary V_TOPK expert shapes, and an enforced
  stage-marker contract" -- Group A (routing shape word), Group C (shared
  experts and the Qwen2-MoE sigmoid gate).
* "MoE: timing-replay harnesses, shared experts, parameterized V_TOPK
  routing" -- Part 2 (generic topk_softmax; SwiGLU expert).
* "Fused MoE Kernel Notes" -- Scatter/gather layout, Duplicate top-k routes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (no fast-math, so libm's exp and IEEE
    double arithmetic are what the definitions say)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def _bind(lib):
    c = ctypes
    P = c.c_void_p
    lib.oracle_topk_pack.restype = c.c_uint32
    lib.oracle_topk_pack.argtypes = [c.c_int32, c.c_int32]
    lib.oracle_topk_unpack.restype = c.c_int32
    lib.oracle_topk_unpack.argtypes = [c.c_uint32, c.POINTER(c.c_int32), c.POINTER(c.c_int32)]
    lib.oracle_router_logits.restype = None
    lib.oracle_router_logits.argtypes = [c.c_int64, P, c.c_int64, c.c_int64, P, c.c_int32,
                                         P, c.c_int32, P, c.c_int32]
    lib.oracle_topk_softmax.restype = c.c_int32
    lib.oracle_topk_softmax.argtypes = [c.c_int64, c.c_uint32, c.c_int32, P, c.c_int64,
                                        P, P, P]
    lib.oracle_sigmoid.restype = None
    lib.oracle_sigmoid.argtypes = [c.c_int64, P, c.c_int64, P]
    lib.oracle_permute.restype = c.c_int32
    lib.oracle_permute.argtypes = [c.c_int64, c.c_int32, c.c_int32, P, P, P, P, P]
    lib.oracle_round_act.restype = c.c_double
    lib.oracle_round_act.argtypes = [c.c_double, c.c_int32]
    lib.oracle_rmsnorm.restype = None
    lib.oracle_rmsnorm.argtypes = [c.c_int64, c.c_int64, P, c.c_int32, P, c.c_double, P]
    lib.oracle_moe_ffn.restype = None
    lib.oracle_moe_ffn.argtypes = [c.c_int64, P, c.c_int64, c.c_int64, c.c_int64, c.c_int32,
                                   P, c.c_int32, c.c_int32, P, P, P, P, c.c_int64, P,
                                   c.c_int64, P, c.c_int64, P, P, P, P, c.c_int32]
    return lib


def load(path: Optional[str] = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _host(a):
    """(keep-alive object, pointer, dtype code) for a CPU tensor/array."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            if a.is_cuda:
                raise ValueError("oracle inputs must be host tensors")
            a = a.contiguous()
            if a.dtype == torch.bfloat16:
                return a, a.data_ptr(), BF16
            if a.dtype == torch.float32:
                return a, a.data_ptr(), F32
            raise TypeError("oracle inputs are fp32 or bf16, got %s" % a.dtype)
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data, F32


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


# ---------------------------------------------------------------------------
# public API
# ---------------------------------------------------------------------------
def topk_pack(num_experts: int, top_k: int) -> int:
    """(num_experts << 8) | top_k, or 0 when the shape does not fit."""
    return int(load().oracle_topk_pack(num_experts, top_k))


def topk_unpack(word: int):
    """(num_experts, top_k), or None for an invalid word (0 = never set)."""
    e, k = ctypes.c_int32(), ctypes.c_int32()
    rc = load().oracle_topk_unpack(word, ctypes.byref(e), ctypes.byref(k))
    return None if rc != 0 else (e.value, k.value)


def router_logits(x, w_router, tokens=None, nthreads: int = 0) -> np.ndarray:
    """fp64 logits[i, c] = x[tokens[i]] . w_router[c] for every router row c."""
    xk, xp, xdt = _host(x)
    wk, wp, wdt = _host(w_router)
    H = x.shape[1]
    ncols = w_router.shape[0]
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    n = x.shape[0] if tok is None else tok.shape[0]
    out = np.empty((n, ncols), dtype=np.float64)
    load().oracle_router_logits(n, _ptr(tok), H, ncols, xp, xdt, wp, wdt, out.ctypes.data,
                                nthreads)
    return out


def topk_softmax(logits: np.ndarray, num_experts: int, top_k: int, norm_topk: bool,
                 word: Optional[int] = None):
    """(idx [n,k] int32, weights [n,k] f64, gap [n] f64) from fp64 logits whose
    first num_experts columns are the expert logits."""
    lg = np.ascontiguousarray(logits, dtype=np.float64)
    n = lg.shape[0]
    idx = np.empty((n, top_k), dtype=np.int32)
    w = np.empty((n, top_k), dtype=np.float64)
    gap = np.empty((n,), dtype=np.float64)
    if word is None:
        word = topk_pack(num_experts, top_k)
    rc = load().oracle_topk_softmax(n, word, int(bool(norm_topk)), lg.ctypes.data,
                                    lg.shape[1], idx.ctypes.data, w.ctypes.data,
                                    gap.ctypes.data)
    if rc != 0:
        raise ValueError("invalid routing shape word %d" % word)
    return idx, w, gap


def sigmoid(z: np.ndarray) -> np.ndarray:
    zz = np.ascontiguousarray(z, dtype=np.float64)
    out = np.empty(zz.shape[0], dtype=np.float64)
    load().oracle_sigmoid(zz.shape[0], zz.ctypes.data, 1, out.ctypes.data)
    return out


def permute(idx: np.ndarray, num_experts: int):
    """(counts [E], offsets [E+1], scatter_index [T,k], row_token [T*k])."""
    ii = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = ii.shape
    counts = np.empty(num_experts, dtype=np.int32)
    offsets = np.empty(num_experts + 1, dtype=np.int32)
    sidx = np.empty((T, k), dtype=np.int32)
    row_token = np.empty(T * k, dtype=np.int32)
    rc = load().oracle_permute(T, k, num_experts, ii.ctypes.data, counts.ctypes.data,
                               offsets.ctypes.data, sidx.ctypes.data, row_token.ctypes.data)
    if rc != 0:
        raise ValueError("route index outside [0, num_experts)")
    return counts, offsets, sidx, row_token


def moe_ffn(x, idx, weights, gate, w_gate, w_up, w_down, sh_gate=None, sh_up=None,
            sh_down=None, tokens=None, gate_stride=None, up_stride=None,
            down_stride=None, moe_inter=None, nthreads: int = 0) -> np.ndarray:
    """fp64 y[i] = gate[i]*shared(x[tok_i]) + sum_s w[i,s]*expert_{idx[i,s]}(x[tok_i]).

    w_gate/w_up are [E, I, H] (or any buffer with the given expert strides, in
    elements), w_down [E, H, I]; shared weights [I_sh, H], [I_sh, H], [H, I_sh]
    or None.  idx/weights are [n, k] for the listed tokens, gate [n] or None.
    """
    xk, xp, xdt = _host(x)
    gk, gp, wdt = _host(w_gate)
    uk, up_, wdt2 = _host(w_up)
    dk, dp, wdt3 = _host(w_down)
    assert wdt == wdt2 == wdt3
    H = x.shape[1]
    I = int(moe_inter) if moe_inter is not None else int(w_gate.shape[-2])
    gate_stride = I * H if gate_stride is None else gate_stride
    up_stride = I * H if up_stride is None else up_stride
    down_stride = H * I if down_stride is None else down_stride
    if sh_gate is not None:
        sgk, sgp, d1 = _host(sh_gate)
        suk, sup, d2 = _host(sh_up)
        sdk, sdp, d3 = _host(sh_down)
        assert d1 == d2 == d3 == wdt
        I_sh = sh_gate.shape[0]
    else:
        sgp = sup = sdp = None
        I_sh = 0
    ii = np.ascontiguousarray(idx, dtype=np.int32)
    ww = np.ascontiguousarray(weights, dtype=np.float64)
    n, k = ii.shape
    gg = None if gate is None else np.ascontiguousarray(gate, dtype=np.float64)
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    y = np.empty((n, H), dtype=np.float64)
    load().oracle_moe_ffn(n, _ptr(tok), H, I, I_sh, k, xp, xdt, wdt, ii.ctypes.data,
                          ww.ctypes.data, _ptr(gg), gp, gate_stride, up_, up_stride, dp,
                          down_stride, sgp, sup, sdp, y.ctypes.data, nthreads)
    return y


def hash_route(token_ids, table, top_k: int):
    """Hash-MoE routing ("Fused MoE Kernel Notes", Duplicate top-k routes: a
    token-to-expert lookup can give two slots of a token the same expert):
    idx[t, s] = table[token_ids[t], s] for a lookup table [vocab, k]; every
    slot weighs 1/k (the reading taken: the notes' regression pattern uses one
    constant routing weight for all slots), as float64.  A token id outside
    [0, vocab) routes all its slots to -1 (dropped by the permutation)."""
    ids = np.asarray(token_ids, dtype=np.int64)
    tab = np.asarray(table, dtype=np.int64).reshape(-1, top_k)
    idx = np.full((ids.size, top_k), -1, dtype=np.int32)
    for t, tok in enumerate(ids):
        if 0 <= tok < tab.shape[0]:
            for s in range(top_k):
                idx[t, s] = tab[tok, s]
    return idx, np.full((ids.size, top_k), 1.0 / top_k)


def round_act(v: float, dtype: str) -> float:
    """The activation-type value nearest to v (ties to even), as a float."""
    return load().oracle_round_act(float(v), BF16 if dtype == "bf16" else F32)


def rmsnorm(x, w, eps: float):
    """x / sqrt(mean(x^2) + eps) * w per row, in fp64, rounded once to x's
    type; returns a host tensor of that type (the values the layer's router
    and experts see)."""
    import torch
    xk, xp, xdt = _host(x)
    wk, wp, wdt = _host(w)
    assert xdt == wdt
    out = torch.empty(tuple(x.shape), dtype=xk.dtype)
    T, H = x.shape
    load().oracle_rmsnorm(T, H, xp, xdt, wp, float(eps), out.data_ptr())
    return out


def layer_input(wl, inputs):
    """The activations the MoE FFN sees: x, or its input RMSNorm."""
    if getattr(wl, "input_norm", False):
        return rmsnorm(inputs["x"], inputs["norm_weight"], wl.norm_eps)
    return inputs["x"]


def route(wl, inputs, tokens=None, nthreads: int = 0, xin=None):
    """Routing for the listed tokens (all tokens when None): dict with idx,
    weights, gate (or None) and gap.  Direct routes are returned as given.
    xin: the layer input (layer_input), computed here when None."""
    E, k = wl.E, wl.k
    if inputs.get("routes_idx") is not None:
        ridx = inputs["routes_idx"].cpu().numpy()
        rw = inputs["routes_w"].cpu().float().numpy().astype(np.float64)
        if tokens is not None:
            ridx, rw = ridx[tokens], rw[tokens]
        n = ridx.shape[0]
        return dict(idx=ridx.astype(np.int32), weights=rw, gate=None,
                    gap=np.full(n, np.inf), logits=None)
    if xin is None:
        xin = layer_input(wl, inputs)
    lg = router_logits(xin, inputs["w_router"], tokens, nthreads)
    idx, w, gap = topk_softmax(lg, E, k, wl.norm_topk)
    gate = sigmoid(lg[:, E]) if wl.shared_gate else None
    return dict(idx=idx, weights=w, gate=gate, gap=gap, logits=lg)


def forward(wl, inputs, tokens=None, nthreads: int = 0):
    """Whole layer for the listed tokens: input preparation (RMSNorm) when the
    workload has it, routing, expert FFNs + combine, then the residual x."""
    xin = layer_input(wl, inputs)
    r = route(wl, inputs, tokens, nthreads, xin=xin)
    y = moe_ffn(xin, r["idx"], r["weights"], r["gate"], inputs["w_gate"],
                inputs["w_up"], inputs["w_down"], inputs.get("sh_gate"),
                inputs.get("sh_up"), inputs.get("sh_down"), tokens=tokens,
                nthreads=nthreads)
    if getattr(wl, "residual", False):
        x = inputs["x"].cpu().double().numpy()
        y = y + (x if tokens is None else x[np.asarray(tokens)])
    r["y"] = y
    return r
