"""fp64 backward of the routed-expert MoE FFN (the fused scatter / grouped
GEMM / gather op), for checking the CUDA backward.

TEST INFRASTRUCTURE ONLY.  Imported by the test suite and by ``bench.py``'s
CPU-baseline leg -- nowhere else; it imports nothing from the product package
and shares no code with the CUDA path.  Plain numpy in float64: per expert
group one matmul per step (the library primitive), no blocking or fusion.

What it differentiates ("Fused MoE Kernel Notes", Scatter/gather layout and
Backward grouped-GEMM launch bound): with the routes given -- idx [T, k]
(duplicates allowed: "Fused MoE Kernel Notes", Duplicate top-k routes) and
routing weights w [T, k] --

    a_ts = W_gate[e] x_t,  b_ts = W_up[e] x_t,  h_ts = silu(a_ts) * b_ts,
    o_ts = W_down[e] h_ts,  y_t = sum_s w_ts o_ts        (e = idx[t, s])

and, given dy = dL/dy [T, H], the chain rule in reverse order of that
forward (this is the reading of the notes' ``grad_fc2_output =
moe_scatter(grad_output, scatter_index)``: the scattered gradient of row
(t, s) is the gradient of o_ts, so it carries the routing weight):

    do_ts = w_ts dy_t                          (scatter of the output gradient)
    dw_ts = <dy_t, o_ts>                       (routing-weight gradient)
    dh_ts = W_down[e]^T do_ts                  (dgrad through down)
    da_ts = dh_ts * b_ts * silu'(a_ts),  db_ts = dh_ts * silu(a_ts)
    dW_down[e] = sum over rows of e of do_ts h_ts^T          (weight gradients:
    dW_gate[e] = sum da_ts x_t^T,  dW_up[e] = sum db_ts x_t^T  K = group rows)
    dx_t = sum_s (W_gate[e]^T da_ts + W_up[e]^T db_ts)        (gather)

silu(a) = a sigma(a), silu'(a) = sigma(a) (1 + a (1 - sigma(a))).  The
router, a shared expert and the input RMSNorm are ordinary dense layers
around this op and are not part of it.

Pinned in tests/test_backward_oracle.py against central differences of the
C forward oracle, homogeneity identities, a symbolic derivative and the
duplicate-route identity.
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    """Exact float64 copy of a CPU tensor (fp32 / bf16) or array."""
    if hasattr(a, "detach"):
        return a.detach().cpu().double().numpy()
    return np.asarray(a, dtype=np.float64)


def sigmoid(a: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-a))


def group_rows(idx: np.ndarray, num_experts: int):
    """For each expert, its (token, slot) pairs in row-major order -- the order
    of the grouped rows ("Fused MoE Kernel Notes", Scatter/gather layout)."""
    T, k = idx.shape
    flat = idx.reshape(-1)
    out = []
    for e in range(num_experts):
        pairs = np.nonzero(flat == e)[0]
        out.append((pairs // k, pairs % k))
    return out


def forward(x, idx, w, w_gate, w_up, w_down):
    """fp64 routed output y [T, H] and the per-pair intermediates, with the
    same definitions as the backward below (used by the backward and by its
    tests)."""
    X = _f64(x)
    ii = np.asarray(idx, dtype=np.int64)
    W = _f64(w)
    Wg, Wu, Wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    E = Wg.shape[0]
    T, H = X.shape
    y = np.zeros((T, H))
    saved = []
    for e, (tok, slot) in enumerate(group_rows(ii, E)):
        Xe = X[tok]
        A = Xe @ Wg[e].T
        B = Xe @ Wu[e].T
        Hh = A * sigmoid(A) * B
        O = Hh @ Wd[e].T
        np.add.at(y, tok, W[tok, slot][:, None] * O)
        saved.append((tok, slot, Xe, A, B, Hh, O))
    return y, saved


def backward(x, idx, w, w_gate, w_up, w_down, dy):
    """Gradients of sum(dy * y) with respect to x [T, H], w [T, k],
    w_gate / w_up [E, I, H] and w_down [E, H, I], all float64."""
    X = _f64(x)
    W = _f64(w)
    Wg, Wu, Wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    dY = _f64(dy)
    _, saved = forward(x, idx, w, w_gate, w_up, w_down)
    dx = np.zeros_like(X)
    dw = np.zeros_like(W)
    dWg = np.zeros_like(Wg)
    dWu = np.zeros_like(Wu)
    dWd = np.zeros_like(Wd)
    for e, (tok, slot, Xe, A, B, Hh, O) in enumerate(saved):
        if tok.size == 0:
            continue
        dO = W[tok, slot][:, None] * dY[tok]          # scatter of the output gradient
        dw[tok, slot] = np.sum(dY[tok] * O, axis=1)   # routing-weight gradient
        dH = dO @ Wd[e]                                # dgrad through down
        sg = sigmoid(A)
        dA = dH * B * sg * (1.0 + A * (1.0 - sg))
        dB = dH * A * sg
        dWd[e] = dO.T @ Hh                             # weight gradients
        dWg[e] = dA.T @ Xe
        dWu[e] = dB.T @ Xe
        dXe = dA @ Wg[e] + dB @ Wu[e]                  # dgrad through gate/up
        np.add.at(dx, tok, dXe)                        # gather to the tokens
    return dict(dx=dx, dw=dw, dw_gate=dWg, dw_up=dWu, dw_down=dWd)


def group_weight_grads(a, b, offsets) -> np.ndarray:
    """The weight-gradient grouped GEMM on its own ("Fused MoE Kernel Notes",
    group_gemm_same_mn): dW_g = sum over rows r of group g of a[r]^T b[r],
    i.e. a_g^T b_g, for a [rows, M], b [rows, N]; [G, M, N] float64."""
    A, B = _f64(a), _f64(b)
    off = np.asarray(offsets, dtype=np.int64)
    G = off.size - 1
    out = np.zeros((G, A.shape[1], B.shape[1]))
    for g in range(G):
        r0, r1 = off[g], off[g + 1]
        out[g] = A[r0:r1].T @ B[r0:r1]
    return out
