"""Python binding of libmoe, the GB300 (sm_103a) forward pass of a
Mixture-of-Experts FFN layer:

    y = g(x) * shared(x) + sum_k route_weight_k * SwiGLU-expert_k(x)

Every function here marshals torch tensors into the C ABI declared in
``include/moe.h`` (same names, same argument order) and raises ``MoEError``
on a non-OK status.  All arithmetic runs in the library's CUDA kernels;
PyTorch only provides device memory and the current stream.  There is no
fallback: if ``libmoe.so`` is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import workloads  # noqa: F401  (seeded input generators)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_DEVICE_ROUTE, MOE_ERR_TIMEOUT, MOE_ERR_ROWS = 4, 5, 6, 7
MOE_ERR_GATHER = 8
MOE_F32, MOE_BF16 = 0, 1
STAGES = ("residual_setup", "route", "permute", "gate_up", "down", "shared", "combine")


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str, why: str = ""):
        self.status = status
        super().__init__("%s: %s%s" % (where, moe_status_string(status),
                                       (" (" + why + ")") if why else ""))


class MoEShape(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int64), ("hidden", ctypes.c_int32),
                ("moe_inter", ctypes.c_int32), ("shared_inter", ctypes.c_int32),
                ("topk_shape", ctypes.c_uint32), ("shared_gate", ctypes.c_int32),
                ("norm_topk", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("input_norm", ctypes.c_int32), ("residual", ctypes.c_int32),
                ("norm_eps", ctypes.c_double), ("train", ctypes.c_int32),
                ("weight_format", ctypes.c_int32)]


class MoEWeights(ctypes.Structure):
    _fields_ = [("router", ctypes.c_void_p), ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p),
                ("gate_up_stride", ctypes.c_int64), ("down", ctypes.c_void_p),
                ("down_stride", ctypes.c_int64), ("shared_gate_proj", ctypes.c_void_p),
                ("shared_up", ctypes.c_void_p), ("shared_down", ctypes.c_void_p),
                ("norm_weight", ctypes.c_void_p)]


class MoEExpertGrads(ctypes.Structure):
    _fields_ = [("gate", ctypes.c_void_p), ("up", ctypes.c_void_p),
                ("gate_up_stride", ctypes.c_int64), ("down", ctypes.c_void_p),
                ("down_stride", ctypes.c_int64)]


class MoEBackwardInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("fc1", "grad_fc2", "d_fc1", "dx_perm")]


class MoERouteInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "topk_idx", "topk_w", "gate", "counts", "offsets", "scatter_index", "row_token",
        "x_perm", "h", "y_perm", "shared_out")]


_lib = None


def lib():
    """The loaded libmoe (raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libmoe.so is not built (run __graft_entry__.build() or "
                           "python -m mixture_experts_ffn_04_gb300.build)")
    L = ctypes.CDLL(LIB_PATH)
    P, S, i32, i64, u32, sz = (ctypes.c_void_p, ctypes.POINTER(MoEShape), ctypes.c_int32,
                               ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t)
    sig = {
        "moe_topk_pack": (u32, [i32, i32]),
        "moe_topk_unpack": (i32, [u32, ctypes.POINTER(i32), ctypes.POINTER(i32)]),
        "moe_scratch_bytes": (sz, [S]),
        "moe_workspace_bytes": (sz, [S]),
        "moe_workspace_views": (i32, [S, P, ctypes.POINTER(MoERouteInfo)]),
        "moe_workspace_init": (i32, [P, P]),
        "moe_quantize_mxfp8": (i32, [P, i32, i64, i64, i32, i64, i64, P, P]),
        "moe_route": (i32, [S, P, P, P, P, P, P, sz, P]),
        "moe_hash_route": (i32, [S, P, P, i64, P, P, P, sz, P]),
        "moe_permute": (i32, [S, P, P, P, P, P, P, P, P, sz, P]),
        "moe_permute_static": (i32, [S, P, P, P, P, P, P, P, P]),
        "moe_grouped_swiglu": (i32, [S, P, P, P, i64, P, i32, i64, i32, P, P, sz, P]),
        "moe_grouped_swiglu_gather": (i32, [S, P, P, P, P, i64, P, i32, i64, i32, P, P, sz, P]),
        "moe_grouped_down": (i32, [S, P, P, i64, P, i32, i64, i32, P, P, sz, P]),
        "moe_combine": (i32, [S, P, P, P, P, P, P, P, P]),
        "moe_residual_setup": (i32, [S, P, P, P, P]),
        "moe_layer_forward": (i32, [S, ctypes.POINTER(MoEWeights), P, P, P, P, P, sz, P]),
        "moe_layer_forward_traced": (i32, [S, ctypes.POINTER(MoEWeights), P, P, P, P, P, sz, P,
                                           ctypes.POINTER(ctypes.c_void_p)]),
        "moe_get_device_status": (i32, [P, P, ctypes.POINTER(u32)]),
        "moe_status_string": (ctypes.c_char_p, [i32]),
        "moe_last_error": (ctypes.c_char_p, []),
        "moe_stage_name": (ctypes.c_char_p, [i32]),
        "moe_last_launch_count": (i32, []),
        "moe_testing_set_gemm_engine": (i32, [i32]),
        "moe_testing_set_fork_sms": (i32, [i32]),
        "moe_testing_set_zero_pad": (i32, [i32]),
        "moe_get_route_stats": (i32, [P, P, ctypes.POINTER(u32)]),
        "moe_testing_router_logits": (i32, [S, P, P, P, P, sz, P]),
        "moe_testing_wait_probe": (i32, [P, i64, i32, P]),
        # backward (moe_backward.h)
        "moe_backward_views": (i32, [S, P, ctypes.POINTER(MoEBackwardInfo)]),
        "moe_grouped_swiglu_save": (i32, [S, P, P, P, i64, P, i32, i64, i32, P, P, P, sz, P]),
        "moe_scatter_grad": (i32, [S, P, P, P, P, P, P, P]),
        "moe_grouped_down_dgrad": (i32, [S, P, P, i64, P, P, i32, i64, i32, P, P, sz, P]),
        "moe_grouped_gate_up_dgrad": (i32, [S, P, P, P, i64, P, i32, i64, i32, P, P, sz, P]),
        "moe_grouped_wgrad": (i32, [S, P, i64, P, i64, P, i32, i64, i32, i32, P, i64, P, sz, P]),
        "moe_gather_grad": (i32, [S, P, P, P, P, P]),
        "moe_layer_backward": (i32, [S, ctypes.POINTER(MoEWeights), P, P, P,
                                     ctypes.POINTER(MoEExpertGrads), P, sz, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmoe must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return stream


def _check(st: int, where: str):
    if st != MOE_OK:
        why = lib().moe_last_error()
        raise MoEError(st, where, why.decode() if why else "")


def _dtype_code(dt: torch.dtype) -> int:
    return {torch.float32: MOE_F32, torch.bfloat16: MOE_BF16}[dt]


# ---------------------------------------------------------------------------
# the C ABI, name for name
# ---------------------------------------------------------------------------
def moe_topk_pack(num_experts: int, top_k: int) -> int:
    return int(lib().moe_topk_pack(num_experts, top_k))


def moe_topk_unpack(word: int):
    e, k = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().moe_topk_unpack(word, ctypes.byref(e), ctypes.byref(k)), "moe_topk_unpack")
    return e.value, k.value


def moe_scratch_bytes(shape: MoEShape) -> int:
    return int(lib().moe_scratch_bytes(ctypes.byref(shape)))


def moe_workspace_bytes(shape: MoEShape) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(shape)))


def moe_quantize_mxfp8(w, batch, rows, K, src_stride, dst_stride, packed, stream=None):
    """Packed MXFP8 matrices from bf16 / fp32 ones (see include/moe.h)."""
    _check(lib().moe_quantize_mxfp8(_p(w), _dtype_code(w.dtype), batch, rows, K, src_stride,
                                    dst_stride, _p(packed), _stream(stream)),
           "moe_quantize_mxfp8")


def mxfp8_pack(w: torch.Tensor, stream=None) -> torch.Tensor:
    """[..., N, K] weights -> [..., N*K*9/8] uint8 packed MXFP8 matrices (the
    leading dimensions are the batch), on w's device."""
    N, K = w.shape[-2], w.shape[-1]
    batch = w.numel() // (N * K)
    out = torch.empty(tuple(w.shape[:-2]) + (N * K // 8 * 9,), dtype=torch.uint8, device=w.device)
    moe_quantize_mxfp8(w, batch, N, K, N * K, N * K // 8 * 9, out, stream)
    return out


MOE_WEIGHTS_ACT, MOE_WEIGHTS_MXFP8 = 0, 1


def moe_workspace_init(ws: torch.Tensor, stream=None):
    _check(lib().moe_workspace_init(_p(ws), _stream(stream)), "moe_workspace_init")


def moe_workspace_views(shape: MoEShape, ws: torch.Tensor) -> dict:
    """Tensor views of the routing and intermediates inside a layer workspace."""
    info = MoERouteInfo()
    _check(lib().moe_workspace_views(ctypes.byref(shape), _p(ws), ctypes.byref(info)),
           "moe_workspace_views")
    E, k = moe_topk_unpack(shape.topk_shape)
    T, H, I = shape.tokens, shape.hidden, shape.moe_inter
    act = torch.float32 if shape.dtype == MOE_F32 else torch.bfloat16
    base = ws.data_ptr()

    def view(ptr, dt, shp):
        if ptr is None:
            return None
        n = 1
        for d in shp:
            n *= d
        off = ptr - base
        return ws[off: off + n * torch.tensor([], dtype=dt).element_size()].view(dt).view(*shp)

    return dict(topk_idx=view(info.topk_idx, torch.int32, (T, k)),
                topk_w=view(info.topk_w, torch.float32, (T, k)),
                gate=view(info.gate, torch.float32, (T,)),
                counts=view(info.counts, torch.int32, (E,)),
                offsets=view(info.offsets, torch.int32, (E + 1,)),
                scatter_index=view(info.scatter_index, torch.int32, (T, k)),
                row_token=view(info.row_token, torch.int32, (T * k,)),
                x_perm=view(info.x_perm, act, (T * k, H)),
                h=view(info.h, act, (T * k, I)),
                y_perm=view(info.y_perm, act, (T * k, H)),
                shared_out=view(info.shared_out, act, (T, H)))


def moe_route(shape, x, w_router, topk_idx, topk_w, gate, ws, stream=None):
    _check(lib().moe_route(ctypes.byref(shape), _p(x), _p(w_router), _p(topk_idx), _p(topk_w),
                           _p(gate), _p(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_route")


def moe_hash_route(shape, token_ids, table, vocab, topk_idx, topk_w, ws, stream=None):
    _check(lib().moe_hash_route(ctypes.byref(shape), _p(token_ids), _p(table), vocab,
                                _p(topk_idx), _p(topk_w), _p(ws), ws.numel() * ws.element_size(),
                                _stream(stream)), "moe_hash_route")


def moe_permute(shape, x, topk_idx, counts, offsets, scatter_index, row_token, x_perm, ws,
                stream=None):
    _check(lib().moe_permute(ctypes.byref(shape), _p(x), _p(topk_idx), _p(counts), _p(offsets),
                             _p(scatter_index), _p(row_token), _p(x_perm), _p(ws),
                             ws.numel() * ws.element_size(), _stream(stream)), "moe_permute")


def moe_permute_static(shape, x, topk_idx, counts, offsets, scatter_index, row_token, x_perm,
                       stream=None):
    """moe_permute with the library's static scratch instead of a workspace."""
    _check(lib().moe_permute_static(ctypes.byref(shape), _p(x), _p(topk_idx), _p(counts),
                                    _p(offsets), _p(scatter_index), _p(row_token), _p(x_perm),
                                    _stream(stream)), "moe_permute_static")


def moe_grouped_swiglu(shape, x_perm, w_gate, w_up, expert_stride, offsets, num_groups,
                       rows_bound, inter, h, ws, stream=None, w_up_ptr=None):
    up = w_up_ptr if w_up_ptr is not None else _p(w_up)
    _check(lib().moe_grouped_swiglu(ctypes.byref(shape), _p(x_perm), _p(w_gate), up,
                                    expert_stride, _p(offsets), num_groups, rows_bound, inter,
                                    _p(h), _p(ws), ws.numel() * ws.element_size(),
                                    _stream(stream)), "moe_grouped_swiglu")


def moe_grouped_swiglu_gather(shape, x, row_token, w_gate, w_up, expert_stride, offsets,
                              num_groups, rows_bound, inter, h, ws, stream=None, w_up_ptr=None):
    up = w_up_ptr if w_up_ptr is not None else _p(w_up)
    _check(lib().moe_grouped_swiglu_gather(ctypes.byref(shape), _p(x), _p(row_token), _p(w_gate),
                                           up, expert_stride, _p(offsets), num_groups,
                                           rows_bound, inter, _p(h), _p(ws),
                                           ws.numel() * ws.element_size(), _stream(stream)),
           "moe_grouped_swiglu_gather")


def moe_grouped_down(shape, h, w_down, expert_stride, offsets, num_groups, rows_bound, inter,
                     y_perm, ws, stream=None):
    _check(lib().moe_grouped_down(ctypes.byref(shape), _p(h), _p(w_down), expert_stride,
                                  _p(offsets), num_groups, rows_bound, inter, _p(y_perm), _p(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)),
           "moe_grouped_down")


def moe_combine(shape, y_perm, scatter_index, topk_w, shared_out, gate, y, stream=None,
                residual=None):
    _check(lib().moe_combine(ctypes.byref(shape), _p(y_perm), _p(scatter_index), _p(topk_w),
                             _p(shared_out), _p(gate), _p(residual), _p(y), _stream(stream)),
           "moe_combine")


def moe_residual_setup(shape, x, norm_weight, x_norm, stream=None):
    _check(lib().moe_residual_setup(ctypes.byref(shape), _p(x), _p(norm_weight), _p(x_norm),
                                    _stream(stream)), "moe_residual_setup")


def moe_layer_forward(shape, weights: MoEWeights, x, routes_idx, routes_w, y, ws, stream=None):
    _check(lib().moe_layer_forward(ctypes.byref(shape), ctypes.byref(weights), _p(x),
                                   _p(routes_idx), _p(routes_w), _p(y), _p(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)),
           "moe_layer_forward")


def moe_layer_forward_traced(shape, weights: MoEWeights, x, routes_idx, routes_w, y, ws,
                             stage_events, stream=None):
    """stage_events: MOE_NUM_STAGES + 1 torch.cuda.Event objects (recorded once
    beforehand so that their CUDA events exist)."""
    arr = (ctypes.c_void_p * len(stage_events))(*[e.cuda_event for e in stage_events])
    _check(lib().moe_layer_forward_traced(ctypes.byref(shape), ctypes.byref(weights), _p(x),
                                          _p(routes_idx), _p(routes_w), _p(y), _p(ws),
                                          ws.numel() * ws.element_size(), _stream(stream), arr),
           "moe_layer_forward_traced")


def moe_get_device_status(ws, stream=None):
    bits = ctypes.c_uint32(0)
    st = lib().moe_get_device_status(_p(ws), _stream(stream), ctypes.byref(bits))
    return int(st), int(bits.value)


def moe_get_route_stats(ws, stream=None) -> int:
    """Read and clear the count of tokens whose top-k was re-decided exactly."""
    n = ctypes.c_uint32(0)
    _check(lib().moe_get_route_stats(_p(ws), _stream(stream), ctypes.byref(n)),
           "moe_get_route_stats")
    return int(n.value)


def moe_testing_router_logits(shape, x, w_router, logits, ws, stream=None):
    _check(lib().moe_testing_router_logits(ctypes.byref(shape), _p(x), _p(w_router), _p(logits),
                                           _p(ws), ws.numel() * ws.element_size(),
                                           _stream(stream)), "moe_testing_router_logits")


def moe_testing_wait_probe(ws, max_cycles: int, arrive: bool, stream=None):
    _check(lib().moe_testing_wait_probe(_p(ws), max_cycles, int(arrive), _stream(stream)),
           "moe_testing_wait_probe")


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_stage_name(stage: int) -> str:
    return lib().moe_stage_name(stage).decode()


def moe_last_launch_count() -> int:
    return int(lib().moe_last_launch_count())


def moe_last_error() -> str:
    return lib().moe_last_error().decode()


def moe_testing_set_gemm_engine(engine: int) -> int:
    return int(lib().moe_testing_set_gemm_engine(engine))


def moe_testing_set_fork_sms(sms: int) -> int:
    return int(lib().moe_testing_set_fork_sms(sms))


def moe_testing_set_zero_pad(mode: int) -> int:
    return int(lib().moe_testing_set_zero_pad(mode))


# ---------------------------------------------------------------------------
# backward (moe_backward.h), name for name
# ---------------------------------------------------------------------------
def _nbytes(ws):
    return ws.numel() * ws.element_size()


def moe_backward_views(shape, ws) -> dict:
    """Tensor views of the backward's grouped buffers in a train-mode workspace."""
    info = MoEBackwardInfo()
    _check(lib().moe_backward_views(ctypes.byref(shape), _p(ws), ctypes.byref(info)),
           "moe_backward_views")
    _, k = moe_topk_unpack(shape.topk_shape)
    R, H, I = shape.tokens * k, shape.hidden, shape.moe_inter
    act = torch.float32 if shape.dtype == MOE_F32 else torch.bfloat16
    esz = 4 if shape.dtype == MOE_F32 else 2
    base = ws.data_ptr()

    def view(ptr, cols):
        off = ptr - base
        return ws[off: off + R * cols * esz].view(act).view(R, cols)

    return dict(fc1=view(info.fc1, 2 * I), grad_fc2=view(info.grad_fc2, H),
                d_fc1=view(info.d_fc1, 2 * I), dx_perm=view(info.dx_perm, H))


def moe_grouped_swiglu_save(shape, x_perm, w_gate, w_up, expert_stride, offsets, num_groups,
                            rows_bound, inter, h, fc1, ws, stream=None):
    _check(lib().moe_grouped_swiglu_save(ctypes.byref(shape), _p(x_perm), _p(w_gate), _p(w_up),
                                         expert_stride, _p(offsets), num_groups, rows_bound,
                                         inter, _p(h), _p(fc1), _p(ws), _nbytes(ws),
                                         _stream(stream)), "moe_grouped_swiglu_save")


def moe_scatter_grad(shape, dy, scatter_index, topk_w, y_perm, grad_fc2, d_topk_w, stream=None):
    _check(lib().moe_scatter_grad(ctypes.byref(shape), _p(dy), _p(scatter_index), _p(topk_w),
                                  _p(y_perm), _p(grad_fc2), _p(d_topk_w), _stream(stream)),
           "moe_scatter_grad")


def moe_grouped_down_dgrad(shape, grad_fc2, w_down, expert_stride, fc1, offsets, num_groups,
                           rows_bound, inter, d_fc1, ws, stream=None):
    _check(lib().moe_grouped_down_dgrad(ctypes.byref(shape), _p(grad_fc2), _p(w_down),
                                        expert_stride, _p(fc1), _p(offsets), num_groups,
                                        rows_bound, inter, _p(d_fc1), _p(ws), _nbytes(ws),
                                        _stream(stream)), "moe_grouped_down_dgrad")


def moe_grouped_gate_up_dgrad(shape, d_fc1, w_gate, w_up, expert_stride, offsets, num_groups,
                              rows_bound, inter, dx_perm, ws, stream=None):
    _check(lib().moe_grouped_gate_up_dgrad(ctypes.byref(shape), _p(d_fc1), _p(w_gate), _p(w_up),
                                           expert_stride, _p(offsets), num_groups, rows_bound,
                                           inter, _p(dx_perm), _p(ws), _nbytes(ws),
                                           _stream(stream)), "moe_grouped_gate_up_dgrad")


def moe_grouped_wgrad(shape, a, lda, b, ldb, offsets, num_groups, rows_bound, M, N, dw,
                      dw_stride, ws, stream=None, a_ptr=None):
    """a_ptr: a raw device address for a (a column offset into a wider matrix)."""
    ap = a_ptr if a_ptr is not None else _p(a)
    _check(lib().moe_grouped_wgrad(ctypes.byref(shape), ap, lda, _p(b), ldb, _p(offsets),
                                   num_groups, rows_bound, M, N, _p(dw), dw_stride, _p(ws),
                                   _nbytes(ws), _stream(stream)), "moe_grouped_wgrad")


def moe_gather_grad(shape, dx_perm, scatter_index, residual_grad, dx, stream=None):
    _check(lib().moe_gather_grad(ctypes.byref(shape), _p(dx_perm), _p(scatter_index),
                                 _p(residual_grad), _p(dx), _stream(stream)), "moe_gather_grad")


def moe_layer_backward(shape, weights: MoEWeights, dy, dx, d_topk_w, grads: MoEExpertGrads, ws,
                       stream=None):
    _check(lib().moe_layer_backward(ctypes.byref(shape), ctypes.byref(weights), _p(dy), _p(dx),
                                    _p(d_topk_w), ctypes.byref(grads), _p(ws), _nbytes(ws),
                                    _stream(stream)), "moe_layer_backward")


def grads_for(dw_gate, dw_up, dw_down) -> MoEExpertGrads:
    """MoEExpertGrads over [E, I, H], [E, I, H], [E, H, I] tensors."""
    g = MoEExpertGrads()
    g.gate, g.up, g.down = _p(dw_gate), _p(dw_up), _p(dw_down)
    g.gate_up_stride = dw_gate.shape[1] * dw_gate.shape[2]
    g.down_stride = dw_down.shape[1] * dw_down.shape[2]
    return g


# ---------------------------------------------------------------------------
# conveniences over the ABI (allocation through torch, nothing else)
# ---------------------------------------------------------------------------
def shape_for(wl, T: Optional[int] = None) -> MoEShape:
    s = MoEShape()
    s.tokens = wl.T if T is None else T
    s.hidden, s.moe_inter, s.shared_inter = wl.H, wl.I, wl.I_sh
    s.topk_shape = moe_topk_pack(wl.E, wl.k)
    s.shared_gate = int(wl.shared_gate)
    s.norm_topk = int(wl.norm_topk)
    s.dtype = MOE_F32 if wl.dtype == "f32" else MOE_BF16
    s.input_norm = int(getattr(wl, "input_norm", False))
    s.residual = int(getattr(wl, "residual", False))
    s.norm_eps = float(getattr(wl, "norm_eps", 1e-6))
    s.train = int(getattr(wl, "train", False))
    s.weight_format = MOE_WEIGHTS_MXFP8 if getattr(wl, "weights", "act") == "mxfp8" else MOE_WEIGHTS_ACT
    return s


def alloc_workspace(shape: MoEShape, device="cuda", full: bool = True, stream=None):
    n = moe_workspace_bytes(shape) if full else moe_scratch_bytes(shape)
    if n == 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "alloc_workspace", "invalid shape")
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off: off + n]
    moe_workspace_init(ws, stream)
    return ws


def weights_from(inputs: dict) -> MoEWeights:
    """MoEWeights over the tensors of a workloads.make_inputs() dict (split fc1)."""
    w = MoEWeights()
    g, d = inputs["w_gate"], inputs["w_down"]
    w.router = _p(inputs.get("w_router"))
    w.gate, w.up = _p(g), _p(inputs["w_up"])
    w.down = _p(d)
    if g.dtype == torch.uint8:   # packed MXFP8 [E, N*K*9/8]: strides in bytes
        w.gate_up_stride, w.down_stride = g.shape[1], d.shape[1]
    else:
        w.gate_up_stride = g.shape[1] * g.shape[2]
        w.down_stride = d.shape[1] * d.shape[2]
    w.shared_gate_proj = _p(inputs.get("sh_gate"))
    w.shared_up = _p(inputs.get("sh_up"))
    w.shared_down = _p(inputs.get("sh_down"))
    w.norm_weight = _p(inputs.get("norm_weight"))
    return w


class MoELayer:
    """One layer: shape, weight table and a workspace, over caller tensors."""

    def __init__(self, wl, inputs: dict, T: Optional[int] = None, device="cuda",
                 train: bool = False):
        self.wl = wl
        self.inputs = inputs
        self.shape = shape_for(wl, T if T is not None else inputs["x"].shape[0])
        self.shape.train = int(train)
        self.weights = weights_from(inputs)
        self.ws = alloc_workspace(self.shape, device)

    def forward(self, x, y=None, routes_idx=None, routes_w=None, stream=None):
        if y is None:
            y = torch.empty_like(x)
        moe_layer_forward(self.shape, self.weights, x, routes_idx, routes_w, y, self.ws, stream)
        return y

    def backward(self, dy, dx, d_topk_w, grads: MoEExpertGrads, stream=None):
        """Gradients after a train-mode forward on this layer's workspace."""
        moe_layer_backward(self.shape, self.weights, dy, dx, d_topk_w, grads, self.ws, stream)

    def views(self):
        return moe_workspace_views(self.shape, self.ws)

    def device_status(self, stream=None):
        return moe_get_device_status(self.ws, stream)
