"""MXFP8 expert weights on the GPU (include/moe.h, moe_weight_format): e4m3
values with one e8m0 scale per block of 8 along the reduced axis ("MoE:
shared experts, arbitrary V_TOPK expert shapes, and an enforced stage-marker
contract").

* moe_quantize_mxfp8 is bit-exact against the oracle's quantiser (bf16 and
  fp32 inputs; zero blocks, tiny and large blocks, blocks holding an
  infinity or a NaN);
* the decode, CUDA-core and tensor-core engines on packed MXFP8 weights give
  bit-identical results to the same engines on the dequantised weights
  stored in bf16 (the dequantisation is exact; the tensor-core engine
  converts the weight tiles into the same shared-memory layout the bf16
  engine loads);
* the whole layer with MXFP8 routed and shared weights (Qwen2-MoE shape with
  its gated shared expert: decode T = 1, 8 on the decode engine, T = 200 on
  the CUDA-core engine) against the oracle on the dequantised weights.
Weights are drawn as packed codes and scales (workloads.py), so the oracle
only decodes them (oracle/mxfp8.py)."""
import dataclasses

import numpy as np
import pytest
import torch

import mixture_experts_ffn_04_gb300 as m
from mixture_experts_ffn_04_gb300 import workloads as W
from oracle import mxfp8 as MX
from oracle import oracle as O

from gpu_util import TOL, TIE_GAP, rel_l2

pytestmark = pytest.mark.gpu


def dequant(packed: torch.Tensor, N: int, K: int) -> torch.Tensor:
    """fp32 [..., N, K] values of packed matrices [..., N*K*9/8] (oracle decode)."""
    p = packed.cpu().numpy().reshape(-1, N * K // 8 * 9)
    out = np.stack([MX.dequantize(*MX.unpack(b, N, K)) for b in p]).astype(np.float32)
    return torch.from_numpy(out.reshape(tuple(packed.shape[:-1]) + (N, K)))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantizer_matches_oracle(dtype):
    g = torch.Generator().manual_seed(3)
    w = torch.randn(3, 40, 64, generator=g) * torch.exp2(torch.randint(-20, 12, (3, 40, 1), generator=g).float())
    w[0, :, :8] = 0.0                      # zero blocks
    w[1, 5, 8:16] = 448.0 * 2.0 ** 3      # exactly at the boundary of a scale
    w[2, 7, :8] = 1.875 * 2.0 ** -4       # the mantissa the floor rule would saturate
    w[0, 3, 16:24] = 1.0
    w[0, 3, 19] = float("inf")             # non-finite blocks are stored as NaN
    w[1, 9, 40] = float("nan")
    w[2, 2, 63] = float("-inf")
    w = w.to(dtype)
    got = m.mxfp8_pack(w.cuda()).cpu().numpy()
    for b in range(3):
        c, s = MX.quantize(w[b].double().numpy(), 64)
        assert np.array_equal(got[b], MX.pack(c, s)), b


# every finite e4m3 code: all bytes but the two NaN codes (S.1111.111)
FINITE_CODES = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def extreme_packed(packed: torch.Tensor, N: int, K: int, seed: int, high: int) -> torch.Tensor:
    """Packed matrices [G, N*K*9/8] rewritten so that each holds every finite
    e4m3 code (both zeros, the subnormals, +-448) at seeded positions, and
    scale bytes at both ends of the range: 10-12 (the smallest codes still
    bf16 normals) and high-4 .. high (values up to 448 * 2^(high-127)), with
    at most one high-scale block per row so the outputs stay finite.  The
    rest keep their drawn codes and scales."""
    rng = np.random.default_rng(seed)
    out = packed.cpu().numpy().copy()
    nk = N * K
    for b in range(out.shape[0]):
        codes = out[b, :nk]
        pos = rng.choice(nk, size=FINITE_CODES.size, replace=False)
        codes[pos] = FINITE_CODES
        scales = out[b, nk:].reshape(N, K // 8)
        for n in range(N):
            lo = rng.choice(K // 8, size=2, replace=False)
            scales[n, lo] = rng.integers(10, 13, size=2)
            if n % 3 == 0:
                scales[n, rng.integers(0, K // 8)] = rng.integers(high - 4, high + 1)
    return torch.from_numpy(out).to(packed.device)


def _grouped_pair(engine, mode, extreme=False):
    E, H, I, T, k = 6, 256, 128, 7, 4
    wl = dataclasses.replace(W.small(W.QWEN2_MOE, T=T, H=H, I=I, I_sh=0, E=E, k=k), weights="mxfp8",
                             shared_gate=False)
    d = W.make_inputs(wl, seed=2, device="cuda")
    if extreme:
        # gate and up share a row's output (silu(g) * u): a lower top scale
        d["w_gate"] = extreme_packed(d["w_gate"], I, H, 11, 175)
        d["w_up"] = extreme_packed(d["w_up"], I, H, 12, 175)
        d["w_down"] = extreme_packed(d["w_down"], H, I, 13, 240)
    idx = torch.randint(0, E, (T, k), generator=torch.Generator().manual_seed(0)).int()
    counts, offsets, sidx, row_token = O.permute(idx.numpy(), E)
    R = T * k
    x_perm = d["x"][torch.from_numpy(row_token).long().cuda()].contiguous()
    off = torch.from_numpy(offsets).cuda()
    out = {}
    for fmt in ("mxfp8", "bf16"):
        s = m.shape_for(dataclasses.replace(wl, weights="mxfp8" if fmt == "mxfp8" else "act"))
        ws = m.alloc_workspace(s, full=False)
        if fmt == "mxfp8":
            wg, wu, wd = d["w_gate"], d["w_up"], d["w_down"]
            gstride, dstride = wg.shape[1], wd.shape[1]
        else:
            wg = dequant(d["w_gate"], I, H).bfloat16().cuda()
            wu = dequant(d["w_up"], I, H).bfloat16().cuda()
            wd = dequant(d["w_down"], H, I).bfloat16().cuda()
            gstride, dstride = I * H, H * I
        prev = m.moe_testing_set_gemm_engine(engine)
        try:
            if mode == "swiglu":
                o = torch.empty(R, I, device="cuda", dtype=torch.bfloat16)
                m.moe_grouped_swiglu(s, x_perm, wg, wu, gstride, off, E, R, I, o, ws)
            else:
                hh = (torch.randn(R, I, generator=torch.Generator().manual_seed(1)) * 0.5).bfloat16().cuda()
                o = torch.empty(R, H, device="cuda", dtype=torch.bfloat16)
                m.moe_grouped_down(s, hh, wd, dstride, off, E, R, I, o, ws)
            assert m.moe_get_device_status(ws)[0] == m.MOE_OK
        finally:
            m.moe_testing_set_gemm_engine(prev)
        out[fmt] = o.cpu()
    return out


@pytest.mark.parametrize("engine", [3, 1, 2], ids=["decode-engine", "cuda-core-engine",
                                                  "tensor-core-engine"])
@pytest.mark.parametrize("mode", ["swiglu", "down"])
@pytest.mark.parametrize("extreme", [False, True], ids=["drawn-codes", "every-code-extreme-scales"])
def test_mxfp8_bitwise_equals_dequantised_bf16(engine, mode, extreme):
    out = _grouped_pair(engine, mode, extreme)
    assert torch.isfinite(out["mxfp8"].float()).all()
    assert torch.equal(out["mxfp8"].view(torch.int16), out["bf16"].view(torch.int16))


def test_extreme_packed_holds_every_code_and_both_scale_ends():
    """The rewritten matrices hold what the bitwise test claims (checked on
    the host before any engine sees them)."""
    E, N, K = 2, 16, 256
    base = torch.zeros(E, N * K // 8 * 9, dtype=torch.uint8)
    base[:, N * K:] = 120
    p = extreme_packed(base, N, K, 0, 240).numpy()
    for b in range(E):
        assert set(FINITE_CODES.tolist()) <= set(np.unique(p[b, :N * K]).tolist())
        sc = p[b, N * K:]
        assert sc.min() <= 12
        assert sc.max() >= 236
        v = MX.dequantize(*MX.unpack(p[b], N, K))
        assert np.isfinite(v).all()
        nz = np.abs(v[v != 0])
        assert nz.min() >= 2.0 ** -126 and nz.max() <= 448.0 * 2.0 ** 113


@pytest.mark.parametrize("T", [1, 3, 8, 200])
def test_layer_forward_with_mxfp8_weights(T):
    wl = dataclasses.replace(W.small(W.QWEN2_MOE, T=T, H=512, I=256, I_sh=512, E=16, k=4),
                             weights="mxfp8")
    dev = W.make_inputs(wl, seed=7, device="cuda")
    layer = m.MoELayer(wl, dev)
    y = layer.forward(dev["x"])
    st, bits = layer.device_status()
    assert st == m.MOE_OK, (st, bits)
    E, I, H, I_sh = wl.E, wl.I, wl.H, wl.I_sh
    host = {"x": dev["x"].cpu(), "w_router": dev["w_router"].cpu(), "routes_idx": None,
            "routes_w": None, "norm_weight": None,
            "w_gate": dequant(dev["w_gate"], I, H), "w_up": dequant(dev["w_up"], I, H),
            "w_down": dequant(dev["w_down"], H, I),
            "sh_gate": dequant(dev["sh_gate"], I_sh, H), "sh_up": dequant(dev["sh_up"], I_sh, H),
            "sh_down": dequant(dev["sh_down"], H, I_sh)}
    ref = O.forward(dataclasses.replace(wl, weights="act"), host)
    ok = ref["gap"] >= TIE_GAP
    gi = layer.views()["topk_idx"].cpu().numpy()
    assert (gi[ok] == ref["idx"][ok]).all()
    yg = y.double().cpu().numpy()
    assert np.isfinite(yg).all()
    assert rel_l2(yg[ok], ref["y"][ok]) <= TOL["bf16"], rel_l2(yg[ok], ref["y"][ok])


@pytest.mark.parametrize("T", [8, 64])
def test_full_size_mxfp8_layer_sampled(T):
    """The Qwen2-MoE-shaped layer at full width (H = 3584, 60 experts of
    2560, gated shared MLP of 20480) with every expert weight in MXFP8, on
    the engines the benchmark uses: sampled tokens against the oracle on the
    dequantised weights (each token's own experts and the shared MLP decoded
    on the host)."""
    wl = dataclasses.replace(W.QWEN2_MOE.with_tokens(T), weights="mxfp8")
    dev = W.make_inputs(wl, seed=0, device="cuda")
    layer = m.MoELayer(wl, dev)
    y = layer.forward(dev["x"])
    st, bits = layer.device_status()
    assert st == m.MOE_OK, (st, bits)
    assert bool(torch.isfinite(y.float()).all())
    H, I, I_sh = wl.H, wl.I, wl.I_sh
    host = {"x": dev["x"].cpu(), "w_router": dev["w_router"].cpu(), "routes_idx": None,
            "routes_w": None, "norm_weight": None}
    r = O.route(dataclasses.replace(wl, weights="act"), host)
    sh = [dequant(dev[k], n, kk) for k, n, kk in (("sh_gate", I_sh, H), ("sh_up", I_sh, H),
                                                  ("sh_down", H, I_sh))]
    gi = layer.views()["topk_idx"].cpu().numpy()
    rng = np.random.default_rng(1)
    for t in np.sort(rng.choice(T, size=min(T, 4), replace=False)):
        if r["gap"][t] < TIE_GAP:
            continue
        assert (gi[t] == r["idx"][t]).all()
        used, inv = np.unique(r["idx"][t], return_inverse=True)
        sel = lambda key, n, kk: torch.stack([dequant(dev[key][e], n, kk) for e in used])
        ref = O.moe_ffn(host["x"][t:t + 1], inv.reshape(1, -1).astype(np.int32),
                        r["weights"][t:t + 1], r["gate"][t:t + 1],
                        sel("w_gate", I, H), sel("w_up", I, H), sel("w_down", H, I),
                        sh[0], sh[1], sh[2])
        yg = y[t:t + 1].double().cpu().numpy()
        assert rel_l2(yg, ref) <= TOL["bf16"], (t, rel_l2(yg, ref))
