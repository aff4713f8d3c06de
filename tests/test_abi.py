"""The C ABI without a GPU: the library loads, exports every symbol the
headers declare, and rejects bad arguments on the host before any CUDA call
(status codes and messages follow include/moe.h)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    import mixture_experts_ffn_04_gb300 as m
    from mixture_experts_ffn_04_gb300 import build
    build.build()
    m.lib()
    return m


def _declared_functions():
    names = []
    for h in ("moe.h", "moe_testing.h", "moe_backward.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(m):
    names = _declared_functions()
    assert len(names) >= 18
    lib = ctypes.CDLL(m.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_pack_unpack_matches_pages_rule(m):
    assert m.moe_topk_pack(256, 8) == (256 << 8) | 8
    assert m.moe_topk_pack(16383, 255) == (1 << 22) - 1
    assert m.moe_topk_pack(16384, 1) == 0 and m.moe_topk_pack(8, 256) == 0
    assert m.moe_topk_unpack(15364) == (60, 4)
    with pytest.raises(m.MoEError) as e:
        m.moe_topk_unpack(0)
    assert e.value.status == m.MOE_ERR_INVALID_ARG


def test_stage_names(m):
    """The stage vocabulary of the header and the binding agree both ways."""
    names = [m.moe_stage_name(i) for i in range(7)]
    assert tuple(names) == m.STAGES
    assert m.moe_stage_name(7) == "" and m.moe_stage_name(-1) == ""


def _shape(m, **kw):
    s = m.MoEShape()
    s.tokens, s.hidden, s.moe_inter, s.shared_inter = 64, 256, 128, 0
    s.topk_shape = m.moe_topk_pack(8, 2)
    s.shared_gate, s.norm_topk, s.dtype = 0, 1, m.MOE_BF16
    for k, v in kw.items():
        setattr(s, k, v)
    return s


def test_validation_rejects_bad_shapes(m):
    lib = m.lib()
    P = ctypes.c_void_p
    w = m.MoEWeights()
    cases = [
        (dict(topk_shape=0), m.MOE_ERR_INVALID_ARG, "never set"),
        (dict(shared_gate=1, shared_inter=0), m.MOE_ERR_INVALID_ARG, "half-specified"),
        (dict(dtype=7), m.MOE_ERR_UNSUPPORTED, "dtype"),
        (dict(hidden=100), m.MOE_ERR_INVALID_ARG, "multiples of 8"),
        (dict(tokens=-1), m.MOE_ERR_INVALID_ARG, "tokens"),
        (dict(input_norm=2), m.MOE_ERR_INVALID_ARG, "input_norm"),
        (dict(norm_eps=-1e-6), m.MOE_ERR_INVALID_ARG, "norm_eps"),
        (dict(norm_eps=float("nan")), m.MOE_ERR_INVALID_ARG, "norm_eps"),
    ]
    for kw, status, frag in cases:
        s = _shape(m, **kw)
        assert m.moe_workspace_bytes(s) == 0
        st = lib.moe_layer_forward(ctypes.byref(s), ctypes.byref(w), P(16), None, None, P(16),
                                   P(256), 1 << 30, None)
        assert st == status, (kw, st)
        assert frag in m.moe_last_error(), m.moe_last_error()


def test_validation_rejects_bad_calls(m):
    lib = m.lib()
    P = ctypes.c_void_p
    s = _shape(m)
    need = m.moe_workspace_bytes(s)
    assert need > m.moe_scratch_bytes(s) > 0
    w = m.MoEWeights()
    w.router = w.gate = w.up = w.down = 4096
    w.gate_up_stride = 128 * 256
    w.down_stride = 256 * 128
    # workspace too small / misaligned / missing
    for ws, n in ((P(4096), need - 1), (P(4096 + 16), need), (None, need)):
        st = lib.moe_layer_forward(ctypes.byref(s), ctypes.byref(w), P(4096), None, None,
                                   P(4096), ws, n, None)
        assert st == m.MOE_ERR_WORKSPACE
    # routes_idx without routes_w
    st = lib.moe_layer_forward(ctypes.byref(s), ctypes.byref(w), P(4096), P(4096), None,
                               P(4096), P(4096), need, None)
    assert st == m.MOE_ERR_INVALID_ARG
    # router with k > E
    s2 = _shape(m, topk_shape=m.moe_topk_pack(4, 8))
    st = lib.moe_route(ctypes.byref(s2), P(4096), P(4096), P(4096), P(4096), None, P(4096),
                       1 << 30, None)
    assert st == m.MOE_ERR_INVALID_ARG and "top_k" in m.moe_last_error()
    # input RMSNorm without its weight, and a weight without input_norm
    sn = _shape(m, input_norm=1)
    st = lib.moe_layer_forward(ctypes.byref(sn), ctypes.byref(w), P(4096), None, None,
                               P(4096), P(4096), m.moe_workspace_bytes(sn), None)
    assert st == m.MOE_ERR_INVALID_ARG and "norm_weight" in m.moe_last_error()
    w.norm_weight = 4096
    st = lib.moe_layer_forward(ctypes.byref(s), ctypes.byref(w), P(4096), None, None,
                               P(4096), P(4096), need, None)
    assert st == m.MOE_ERR_INVALID_ARG and "input_norm" in m.moe_last_error()
    w.norm_weight = None
    # shared weights without shared_inter
    w.shared_up = 4096
    st = lib.moe_layer_forward(ctypes.byref(s), ctypes.byref(w), P(4096), None, None, P(4096),
                               P(4096), need, None)
    assert st == m.MOE_ERR_INVALID_ARG
    # grouped GEMM: zero stride with several groups, misaligned operand
    st = lib.moe_grouped_swiglu(ctypes.byref(s), P(4096), P(4096), P(4096), 0, P(4096), 8, 128,
                                128, P(4096), P(4096), 1 << 30, None)
    assert st == m.MOE_ERR_INVALID_ARG
    st = lib.moe_grouped_down(ctypes.byref(s), P(4098), P(4096), 32768, P(4096), 8, 128, 128,
                              P(4096), P(4096), 1 << 30, None)
    assert st == m.MOE_ERR_INVALID_ARG


def test_workspace_layout_scales(m):
    """Intermediates grow with T*k rows; scratch stays small."""
    from mixture_experts_ffn_04_gb300 import workloads as W
    s = m.shape_for(W.DEEPSEEK_V3)
    T, k, H, I = 8192, 8, 7168, 2048
    inter = 2 * T * k * H * 2 + T * k * I * 2     # x_perm, y_perm and h
    assert inter <= m.moe_workspace_bytes(s) <= inter * 1.2
    assert m.moe_scratch_bytes(s) < 128 << 20   # split-K router partials dominate


def test_backward_validation(m):
    """The backward's host checks (include/moe_backward.h), no GPU needed."""
    lib = m.lib()
    P = ctypes.c_void_p
    w = m.MoEWeights()
    w.gate = w.up = w.down = 4096
    w.gate_up_stride = w.down_stride = 128 * 256
    g = m.MoEExpertGrads()
    g.gate = g.up = g.down = 8192
    g.gate_up_stride = g.down_stride = 128 * 256
    s = _shape(m)
    need = m.moe_workspace_bytes(s)
    # the backward needs a train-mode workspace
    st = lib.moe_layer_backward(ctypes.byref(s), ctypes.byref(w), P(4096), P(4096), P(4096),
                                ctypes.byref(g), P(4096), need, None)
    assert st == m.MOE_ERR_INVALID_ARG and "train" in m.moe_last_error()
    info = m.MoEBackwardInfo()
    assert lib.moe_backward_views(ctypes.byref(s), P(4096), ctypes.byref(info)) == m.MOE_ERR_INVALID_ARG
    st_ = _shape(m, train=1)
    need_t = m.moe_workspace_bytes(st_)
    R, H, I = 64 * 2, 256, 128
    assert need_t - need >= 2 * (R * 2 * I * 2) + 2 * (R * H * 2)   # fc1, d_fc1, grad_fc2, dx_perm
    assert lib.moe_backward_views(ctypes.byref(st_), P(4096), ctypes.byref(info)) == m.MOE_OK
    assert info.fc1 >= 4096 + m.moe_scratch_bytes(st_)
    # shapes whose dense parts the op does not differentiate
    for kw, frag in ((dict(shared_inter=256), "shared"), (dict(input_norm=1), "RMSNorm")):
        sx = _shape(m, train=1, **kw)
        st = lib.moe_layer_backward(ctypes.byref(sx), ctypes.byref(w), P(4096), P(4096), P(4096),
                                    ctypes.byref(g), P(4096), m.moe_workspace_bytes(sx), None)
        assert st == m.MOE_ERR_UNSUPPORTED and frag in m.moe_last_error(), m.moe_last_error()
    # workspace too small; gradient stride smaller than one expert
    st = lib.moe_layer_backward(ctypes.byref(st_), ctypes.byref(w), P(4096), P(4096), P(4096),
                                ctypes.byref(g), P(4096), need_t - 1, None)
    assert st == m.MOE_ERR_WORKSPACE
    g.down_stride = 100
    st = lib.moe_layer_backward(ctypes.byref(st_), ctypes.byref(w), P(4096), P(4096), P(4096),
                                ctypes.byref(g), P(4096), need_t, None)
    assert st == m.MOE_ERR_INVALID_ARG and "stride" in m.moe_last_error()
    # grouped calls: bad sizes and misaligned operands
    st = lib.moe_grouped_wgrad(ctypes.byref(s), P(4096), 100, P(4096), 128, P(4096), 8, 128,
                               128, 128, P(4096), 128 * 128, P(4096), 1 << 30, None)
    assert st == m.MOE_ERR_INVALID_ARG and "lda" in m.moe_last_error()
    st = lib.moe_grouped_down_dgrad(ctypes.byref(s), P(4098), P(4096), 32768, P(4096), P(4096),
                                    8, 128, 128, P(4096), P(4096), 1 << 30, None)
    assert st == m.MOE_ERR_INVALID_ARG
    st = lib.moe_grouped_gate_up_dgrad(ctypes.byref(s), P(4096), P(4096), P(4096), 0, P(4096),
                                       8, 128, 128, P(4096), P(4096), 1 << 30, None)
    assert st == m.MOE_ERR_INVALID_ARG and "expert_stride" in m.moe_last_error()
    st = lib.moe_scatter_grad(ctypes.byref(s), P(4096), None, P(4096), P(4096), P(4096),
                              P(4096), None)
    assert st == m.MOE_ERR_INVALID_ARG
    s_bad = _shape(m, train=2)
    assert m.moe_workspace_bytes(s_bad) == 0


def test_mxfp8_validation(m):
    """MXFP8 expert weights (include/moe.h, moe_weight_format): host checks."""
    lib = m.lib()
    P = ctypes.c_void_p
    assert m.moe_workspace_bytes(_shape(m, weight_format=2)) == 0
    sf = _shape(m, weight_format=m.MOE_WEIGHTS_MXFP8, dtype=m.MOE_F32)
    st = lib.moe_route(ctypes.byref(sf), P(4096), P(4096), P(4096), P(4096), None, P(4096),
                       1 << 30, None)
    assert st == m.MOE_ERR_UNSUPPORTED and "bf16" in m.moe_last_error()
    s = _shape(m, weight_format=m.MOE_WEIGHTS_MXFP8)
    need = m.moe_workspace_bytes(s)
    w = m.MoEWeights()
    w.router = w.gate = w.up = w.down = 4096
    # strides count bytes: one packed [128, 256] matrix is 128*256*9/8 bytes
    w.gate_up_stride = w.down_stride = 128 * 256
    st = lib.moe_layer_forward(ctypes.byref(s), ctypes.byref(w), P(4096), None, None, P(4096),
                               P(4096), need, None)
    assert st == m.MOE_ERR_INVALID_ARG and "stride" in m.moe_last_error()
    # grouped call: a stride below one packed matrix
    st = lib.moe_grouped_swiglu(ctypes.byref(s), P(4096), P(4096), P(4096), 128 * 256, P(4096),
                                8, 128, 128, P(4096), P(4096), 1 << 30, None)
    assert st == m.MOE_ERR_INVALID_ARG and "MXFP8" in m.moe_last_error()
    # the backward refuses MXFP8 weights
    st_ = _shape(m, weight_format=m.MOE_WEIGHTS_MXFP8, train=1)
    g = m.MoEExpertGrads()
    g.gate = g.up = g.down = 8192
    g.gate_up_stride = g.down_stride = 128 * 256
    w.gate_up_stride = w.down_stride = 128 * 256 * 9 // 8
    st = lib.moe_layer_backward(ctypes.byref(st_), ctypes.byref(w), P(4096), P(4096), P(4096),
                                ctypes.byref(g), P(4096), m.moe_workspace_bytes(st_), None)
    assert st == m.MOE_ERR_UNSUPPORTED and "MXFP8" in m.moe_last_error()
    # quantiser: K must be a multiple of 8
    assert lib.moe_quantize_mxfp8(P(4096), m.MOE_BF16, 1, 4, 12, 48, 54, P(4096), None) == m.MOE_ERR_INVALID_ARG


def test_hash_route_validation(m):
    lib = m.lib()
    P = ctypes.c_void_p
    s = _shape(m)
    st = lib.moe_hash_route(ctypes.byref(s), P(4096), P(4096), 0, P(4096), P(4096), P(4096),
                            1 << 30, None)
    assert st == m.MOE_ERR_INVALID_ARG and "vocab" in m.moe_last_error()
    st = lib.moe_hash_route(ctypes.byref(s), None, P(4096), 10, P(4096), P(4096), P(4096),
                            1 << 30, None)
    assert st == m.MOE_ERR_INVALID_ARG


def _declared_arity():
    """{function name: parameter count} from the headers' prototypes."""
    out = {}
    for h in ("moe.h", "moe_testing.h", "moe_backward.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for mm in re.finditer(r"\b(moe_\w+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S):
            params = mm.group(2).strip()
            out[mm.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_arity_matches_headers(m):
    """Every ctypes signature of the binding has as many arguments as the C
    prototype it marshals (a drifted binding would pass garbage silently)."""
    arity = _declared_arity()
    lib = m.lib()
    checked = 0
    for name, n in arity.items():
        f = getattr(lib, name)
        if f.argtypes is None:
            continue
        assert len(f.argtypes) == n, (name, len(f.argtypes), n)
        checked += 1
    assert checked >= 30, checked
