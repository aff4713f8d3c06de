"""Expert-parallel exchange (mixture_experts_ffn_04_gb300/expert_parallel.py)
with two gloo ranks on the CPU: each rank routes and groups its own tokens,
the rows of every expert go to the expert's owner and come back, and each
rank's combined output equals the fp64 oracle's forward of its own tokens.
The expert FFNs in the middle are the oracle's (this checks the plan and the
exchanges, not the kernels; the GPU test runs the library's kernels on one
rank).  Uneven expert ranges (E = 7 over 2 ranks), empty experts and
duplicate routes (Zipf) are covered.  Not measured on hardware: every box
here has one GPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mixture_experts_ffn_04_gb300.expert_parallel import ExpertParallel, expert_ranges


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_expert_ranges_cover_every_expert_once():
    for E, world in [(7, 2), (256, 8), (3, 4), (64, 1)]:
        r = expert_ranges(E, world)
        assert r[0][0] == 0 and r[-1][1] == E and len(r) == world
        assert all(a[1] == b[0] for a, b in zip(r, r[1:]))
        sizes = [e1 - e0 for e0, e1 in r]
        assert max(sizes) - min(sizes) <= 1


CASES = {
    "router-E7": dict(base="QWEN3_30B_A3B", T=40, H=64, I=32, E=7, k=2),
    "zipf-duplicates-E8": dict(base="ADV_ZIPF", T=50, H=64, I=32, E=8, k=3, I_sh=0),
}


def _rank_inputs(name, rank):
    from mixture_experts_ffn_04_gb300 import workloads as W
    c = dict(CASES[name])
    base = getattr(W, c.pop("base"))
    wl = W.small(base, **c)
    inp = W.make_inputs(wl, seed=11, device="cpu")          # the same weights on every rank
    tok = W.make_inputs(wl, seed=100 + rank, device="cpu", with_experts=False)
    inp["x"] = tok["x"]                                     # each rank's own tokens
    if wl.routing != "router":
        inp["routes_idx"], inp["routes_w"] = tok["routes_idx"], tok["routes_w"]
    return wl, inp


def _worker(rank, world, port, name, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        _check_rank(rank, name, q)
    except Exception as exc:   # report instead of leaving the parent waiting
        q.put((rank, "error: %r" % (exc,), 0, 0))
        raise
    finally:
        dist.destroy_process_group()


def _check_rank(rank, name, q):
    from oracle import oracle as O
    wl, inp = _rank_inputs(name, rank)
    T, H, E, k = wl.T, wl.H, wl.E, wl.k
    r = O.route(wl, inp)
    idx, w = r["idx"], r["weights"]
    counts, offsets, sidx, row_token = O.permute(idx, E)
    x = inp["x"].double()
    x_perm = x[torch.as_tensor(row_token, dtype=torch.long)]
    ep = ExpertParallel(E)
    lc, loff = ep.plan(torch.as_tensor(counts))
    x_loc = ep.dispatch(x_perm)
    assert x_loc.shape[0] == int(loff[-1])
    # every row the owner received belongs to one of its experts: compute
    # it with the oracle, one expert a row
    y_loc = torch.zeros_like(x_loc)
    for j, e in enumerate(range(ep.e0, ep.e1)):
        a, b = int(loff[j]), int(loff[j + 1])
        if b > a:
            n = b - a
            y_loc[a:b] = torch.from_numpy(O.moe_ffn(
                x_loc[a:b].float().to(torch.float32), np.full((n, 1), 0, np.int32),
                np.ones((n, 1)), None, inp["w_gate"][e:e + 1], inp["w_up"][e:e + 1],
                inp["w_down"][e:e + 1]))
    y_perm = torch.zeros(T * k, H, dtype=torch.float64)
    ep.combine_back(y_loc, y_perm)
    y = np.zeros((T, H))
    yp = y_perm.numpy()
    for t in range(T):
        for s in range(k):
            y[t] += w[t, s] * yp[sidx[t, s]]
    ref = O.forward(wl, inp)["y"]
    err = float(np.abs(y - ref).max() / max(np.abs(ref).max(), 1e-300))
    q.put((rank, err, int(loff[-1]), int(counts.sum())))
    dist.barrier()


@pytest.mark.parametrize("name", sorted(CASES))
def test_two_rank_expert_parallel_equals_the_oracle(name):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, name, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in procs), key=lambda r: r[0])
    for rank, err, _, _ in res:
        assert not isinstance(err, str), (rank, err)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every routed row of both ranks was computed by exactly one owner
    assert sum(r[2] for r in res) == sum(r[3] for r in res)
    for rank, err, _, _ in res:
        assert err < 1e-12, (rank, err)
