"""Failure detection on the GPU without a fault: a bounded mbarrier wait that
nothing completes runs out after its limit, the kernel raises the timeout
bit and returns, the host reads MOE_ERR_TIMEOUT from the status word, and the
context stays usable (a layer forward afterwards matches the oracle)."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_04_gb300 as m
from mixture_experts_ffn_04_gb300 import workloads as W
from oracle import oracle as O

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    wl = W.small(W.QWEN3_30B_A3B, T=64, H=256, I=128, E=8, k=2)
    s = m.shape_for(wl)
    ws = m.alloc_workspace(s, full=False)
    # an arrival completes the phase: no bit
    m.moe_testing_wait_probe(ws, 2_000_000, True)
    st, bits = m.moe_get_device_status(ws)
    assert st == m.MOE_OK and bits == 0
    # nothing arrives: about a millisecond of clocks, then the timeout bit
    m.moe_testing_wait_probe(ws, 2_000_000, False)
    st, bits = m.moe_get_device_status(ws)
    assert st == m.MOE_ERR_TIMEOUT and bits == 4
    assert m.moe_get_device_status(ws)[0] == m.MOE_OK   # read-and-clear
    # the context is still usable
    dev = W.make_inputs(wl, seed=0, device="cuda")
    layer = m.MoELayer(wl, dev)
    y = layer.forward(dev["x"])
    assert layer.device_status()[0] == m.MOE_OK
    ref = O.forward(wl, {k: (v.cpu() if v is not None else None) for k, v in dev.items()})
    ok = ref["gap"] >= 1e-6
    yg = y.double().cpu().numpy()
    err = np.linalg.norm(yg[ok] - ref["y"][ok]) / np.linalg.norm(ref["y"][ok])
    assert err <= 1e-2
