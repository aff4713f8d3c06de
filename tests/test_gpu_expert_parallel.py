"""The expert-parallel layer path (expert_parallel.ep_layer_forward) on one
GPU: with one rank every expert is local and both exchanges are copies, so
route -> permute -> dispatch -> grouped GEMMs over the owned experts ->
return -> combine through the library's entry points must give the layer's
output bit for bit (the two-rank exchanges are checked on the CPU with gloo
in test_expert_parallel.py)."""
import pytest
import torch

import mixture_experts_ffn_04_gb300 as m
from mixture_experts_ffn_04_gb300 import workloads as W
from mixture_experts_ffn_04_gb300.expert_parallel import ExpertParallel, ep_layer_forward

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", [W.small(W.QWEN3_30B_A3B, T=300, H=512, I=256),
                                W.small(W.QWEN3_30B_A3B, T=77, H=392, I=200, E=16, k=3)],
                         ids=["qwen3-reduced", "ragged"])
def test_single_rank_expert_parallel_equals_layer(wl):
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k, v in W.make_inputs(wl, seed=2, device="cpu").items()}
    layer = m.MoELayer(wl, dev)
    y_ref = layer.forward(dev["x"])
    y = ep_layer_forward(m, layer, dev["x"], ExpertParallel(wl.E))
    torch.cuda.synchronize()
    assert layer.device_status()[0] == m.MOE_OK
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
