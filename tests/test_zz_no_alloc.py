"""moe_permute_static -- the allocation-free variant of moe_permute, for
callers that may not allocate device memory while they run -- must give the
workspace version's outputs exactly (indices and copied rows are integer and
byte work: bit-exact), on two calls in a row with different shapes, so that
the static scratch left over from the first call cannot leak into the second.
This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_04_gb300 as m
from mixture_experts_ffn_04_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _outputs(wl, x, idx):
    T, k, E, H = wl.T, wl.k, wl.E, wl.H
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(counts=torch.full((E,), -7, **i32), offsets=torch.full((E + 1,), -7, **i32),
                scatter_index=torch.full((T, k), -7, **i32),
                row_token=torch.full((T * k,), -7, **i32),
                x_perm=torch.full((T * k, H), float("nan"), dtype=x.dtype, device="cuda"))


@pytest.mark.parametrize("dummy", [0])
def test_static_permute_matches_workspace_permute(dummy):
    cases = [
        (W.small(W.DEEPSEEK_V3, T=1000, H=512, I=256, I_sh=256), 0),  # E=256, k=8
        (W.small(W.ADV_ZIPF, T=300, H=256, I=128, I_sh=256), 1),      # E=64, k=6, duplicates
    ]
    for wl, seed in cases:
        g = torch.Generator().manual_seed(seed)
        x = torch.randn(wl.T, wl.H, generator=g).to(torch.bfloat16).cuda()
        if wl.routing == "router":
            idx = torch.randint(0, wl.E, (wl.T, wl.k), generator=g, dtype=torch.int32).cuda()
        else:
            idx = W.make_inputs(wl, seed=seed, with_experts=False)["routes_idx"].cuda()
        s = m.shape_for(wl)
        ws = m.alloc_workspace(s, full=False)
        a = _outputs(wl, x, idx)
        m.moe_permute(s, x, idx, a["counts"], a["offsets"], a["scatter_index"], a["row_token"],
                      a["x_perm"], ws)
        b = _outputs(wl, x, idx)
        m.moe_permute_static(s, x, idx, b["counts"], b["offsets"], b["scatter_index"],
                             b["row_token"], b["x_perm"])
        torch.cuda.synchronize()
        assert m.moe_get_device_status(ws)[0] == m.MOE_OK
        for key in ("counts", "offsets", "scatter_index", "row_token"):
            assert torch.equal(a[key], b[key]), key
        assert torch.equal(a["x_perm"].view(torch.int16), b["x_perm"].view(torch.int16))
        assert int(b["offsets"][-1]) == wl.T * wl.k
