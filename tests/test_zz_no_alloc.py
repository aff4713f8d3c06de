"""moe_permute_static: moe_permute for callers that may not allocate device
memory while they run (a plugin handed only its tensors, a real-time loop that
forbids allocation after start-up).  Its histogram tables live in a static
device array of the library, shared by every call, so each case runs right
after a different shape has used the array.

Checked, bit for bit (indices and copied rows are integer and byte work):
counts, offsets, scatter_index and row_token against the oracle's stable
counting sort of the same routes, x_perm against x gathered through the
oracle's row_token, and all of them against the workspace entry point; both
the multi-chunk path (rank, scan, scatter) and the one-block path (T <= 32)
and T = 0; a route outside [0, E) dropped as documented; the argument errors;
and no device memory taken by a call.  This file is collected last on
purpose."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_04_gb300 as m
from mixture_experts_ffn_04_gb300 import workloads as W
from oracle import oracle as O

pytestmark = pytest.mark.gpu

I32 = dict(dtype=torch.int32, device="cuda")


def _outputs(wl, dtype, with_xperm=True):
    T, k, E, H = wl.T, wl.k, wl.E, wl.H
    return dict(counts=torch.full((E,), -7, **I32), offsets=torch.full((E + 1,), -7, **I32),
                scatter_index=torch.full((T, k), -7, **I32),
                row_token=torch.full((T * k,), -7, **I32),
                x_perm=(torch.full((T * k, H), float("nan"), dtype=dtype, device="cuda")
                        if with_xperm else None))


def _call(fn, s, x, idx, o, *extra):
    fn(s, x, idx, o["counts"], o["offsets"], o["scatter_index"], o["row_token"], o["x_perm"],
       *extra)


def _inputs(wl, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(wl.T, wl.H, generator=g).to(torch.bfloat16)
    if wl.routing == "router":
        idx = torch.randint(0, wl.E, (wl.T, wl.k), generator=g, dtype=torch.int32)
    else:
        idx = W.make_inputs(wl, seed=seed, with_experts=False)["routes_idx"]
    return x, idx


def _check_against_oracle(wl, x, idx, got, dropped=None):
    """dropped: boolean [T, k] of routes outside [0, E) (scatter_index -1,
    not counted).  The oracle groups the valid routes: the dropped ones are
    given to an extra expert E, which sorts after every real group and so
    leaves the real groups' rows as they are."""
    ii = idx.numpy().copy()
    E, T, k = wl.E, wl.T, wl.k
    if dropped is not None:
        ii[dropped] = E
    counts, offsets, sidx, row_token = O.permute(ii, E + 1)
    valid = int(offsets[E])
    assert np.array_equal(got["counts"].cpu().numpy(), counts[:E])
    assert np.array_equal(got["offsets"].cpu().numpy(), offsets[:E + 1])
    gs = got["scatter_index"].cpu().numpy()
    want = sidx.copy()
    if dropped is not None:
        want[dropped] = -1
    assert np.array_equal(gs, want)
    assert np.array_equal(got["row_token"].cpu().numpy()[:valid], row_token[:valid])
    if got["x_perm"] is not None and valid:
        xp = got["x_perm"][:valid].cpu().view(torch.int16)
        assert torch.equal(xp, x.index_select(0, torch.as_tensor(row_token[:valid]).long())
                           .view(torch.int16))
    return valid


CASES = [
    (W.small(W.DEEPSEEK_V3, T=1000, H=512, I=256, I_sh=256), 0),   # E=256, k=8, many chunks
    (W.small(W.ADV_ZIPF, T=300, H=256, I=128, I_sh=256), 1),       # E=64, k=6, duplicates
    (W.small(W.QWEN2_MOE, T=8, H=3584, I=256, I_sh=512), 2),       # T <= 32: one-block path
    (W.small(W.QWEN2_MOE, T=1, H=3584, I=256, I_sh=512), 3),       # one token
    (W.small(W.ADV_E0, T=32, H=256, I=128, I_sh=256), 4),          # one group of T*k rows
]


def test_static_permute_matches_oracle_and_workspace_permute():
    """Every case right after another shape used the static array; each
    compared with the oracle and with moe_permute (workspace)."""
    for wl, seed in CASES + CASES[:2]:
        x, idx = _inputs(wl, seed)
        xd, idd = x.cuda(), idx.cuda()
        s = m.shape_for(wl)
        b = _outputs(wl, xd.dtype)
        _call(m.moe_permute_static, s, xd, idd, b)
        torch.cuda.synchronize()
        assert _check_against_oracle(wl, x, idx, b) == wl.T * wl.k
        ws = m.alloc_workspace(s, full=False)
        a = _outputs(wl, xd.dtype)
        _call(m.moe_permute, s, xd, idd, a, ws)
        torch.cuda.synchronize()
        assert m.moe_get_device_status(ws)[0] == m.MOE_OK
        for key in ("counts", "offsets", "scatter_index", "row_token"):
            assert torch.equal(a[key], b[key]), key
        assert torch.equal(a["x_perm"].view(torch.int16), b["x_perm"].view(torch.int16))


@pytest.mark.parametrize("T", [300, 5])
def test_static_permute_drops_out_of_range_routes(T):
    """A route outside [0, E) is dropped: scatter_index -1, not counted,
    offsets[E] = T*k minus the dropped routes; the other routes are grouped
    exactly as the oracle groups them."""
    wl = W.small(W.DEEPSEEK_V3, T=T, H=256, I=128, I_sh=256)
    x, idx = _inputs(wl, 7)
    idx[0, 1] = wl.E
    idx[T - 1, wl.k - 1] = -1
    idx[T // 2, 0] = 1 << 20
    dropped = (idx.numpy() < 0) | (idx.numpy() >= wl.E)
    b = _outputs(wl, torch.bfloat16)
    _call(m.moe_permute_static, m.shape_for(wl), x.cuda(), idx.cuda(), b)
    torch.cuda.synchronize()
    valid = _check_against_oracle(wl, x, idx, b, dropped=dropped)
    assert valid == T * wl.k - int(dropped.sum())


def test_static_permute_routing_only_and_empty():
    """x_perm NULL (and x NULL): only the routing arrays, as moe_permute.
    T = 0: counts and offsets zero, nothing else touched."""
    wl = W.small(W.DEEPSEEK_V3, T=200, H=256, I=128, I_sh=256)
    x, idx = _inputs(wl, 8)
    b = _outputs(wl, torch.bfloat16, with_xperm=False)
    _call(m.moe_permute_static, m.shape_for(wl), None, idx.cuda(), b)
    torch.cuda.synchronize()
    _check_against_oracle(wl, x, idx, b)

    w0 = W.small(W.DEEPSEEK_V3, T=1, H=256, I=128, I_sh=256)
    s0 = m.shape_for(w0, T=0)
    counts = torch.full((w0.E,), -7, **I32)
    offsets = torch.full((w0.E + 1,), -7, **I32)
    m.moe_permute_static(s0, None, None, counts, offsets, None, None, None)
    torch.cuda.synchronize()
    assert int(counts.abs().sum()) == 0 and int(offsets.abs().sum()) == 0


def test_static_permute_argument_errors():
    wl = W.small(W.DEEPSEEK_V3, T=40, H=256, I=128, I_sh=256)
    s = m.shape_for(wl)
    x, idx = _inputs(wl, 9)
    o = _outputs(wl, torch.bfloat16)
    with pytest.raises(m.MoEError) as e:      # counts missing
        m.moe_permute_static(s, x.cuda(), idx.cuda(), None, o["offsets"], o["scatter_index"],
                             o["row_token"], o["x_perm"])
    assert e.value.status == m.MOE_ERR_INVALID_ARG
    with pytest.raises(m.MoEError) as e:      # x_perm without x
        m.moe_permute_static(s, None, idx.cuda(), o["counts"], o["offsets"],
                             o["scatter_index"], o["row_token"], o["x_perm"])
    assert e.value.status == m.MOE_ERR_INVALID_ARG
    bad = m.shape_for(wl)
    bad.topk_shape = 0                        # routing shape unset
    with pytest.raises(m.MoEError) as e:
        m.moe_permute_static(bad, x.cuda(), idx.cuda(), o["counts"], o["offsets"],
                             o["scatter_index"], o["row_token"], o["x_perm"])
    assert e.value.status == m.MOE_ERR_INVALID_ARG


def test_static_permute_takes_no_device_memory():
    """Free device memory is the same before and after a call (every buffer
    the call touches was made beforehand; the first call on the device has
    already looked the static array up)."""
    wl = W.small(W.DEEPSEEK_V3, T=1000, H=512, I=256, I_sh=256)
    x, idx = _inputs(wl, 10)
    xd, idd = x.cuda(), idx.cuda()
    s = m.shape_for(wl)
    o = _outputs(wl, xd.dtype)
    _call(m.moe_permute_static, s, xd, idd, o)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    _call(m.moe_permute_static, s, xd, idd, o)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    _check_against_oracle(wl, x, idx, o)
