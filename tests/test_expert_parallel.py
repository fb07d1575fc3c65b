"""Expert parallelism (serving_router_gate_gb300.expert_parallel) on the CPU:
the slot ranges and shared-expert shards partition the layer, and with gloo
ranks (world sizes 2 and 4) the one SUM reduction of the ranks' partial
outputs -- each computed by the fp64 oracle on that rank's slot range (SKIP)
and shared shard -- equals the oracle's full layer.  The GPU side of each rank
runs the same library calls as a one-GPU layer with a local range; its partials
are checked on a GPU in tests/test_gpu_expert_parallel.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import moe_inputs as mi
import oracle
from serving_router_gate_gb300.expert_parallel import (ep_reduce_output, ep_shared_range, ep_shared_shard,
                                                       ep_slot_range)


@pytest.mark.parametrize("S,world", [(60, 2), (64, 4), (288, 8), (13, 4), (8, 8), (5, 3)])
def test_slot_ranges_are_contiguous_and_cover_every_slot(S, world):
    seen = []
    prev_end = 0
    for r in range(world):
        lo, n = ep_slot_range(S, world, r)
        assert lo == prev_end and n >= 1
        prev_end = lo + n
        seen.extend(range(lo, lo + n))
    assert seen == list(range(S))
    sizes = [ep_slot_range(S, world, r)[1] for r in range(world)]
    assert max(sizes) - min(sizes) <= 1
    if S % world == 0:
        assert set(sizes) == {S // world}  # E / ep_size slots per rank


def test_slot_range_rejects_more_ranks_than_slots():
    with pytest.raises(ValueError):
        ep_slot_range(4, 8, 0)


@pytest.mark.parametrize("I_sh,world", [(5632, 2), (5632, 8), (256, 4), (192, 4)])
def test_shared_shards_concatenate_to_the_shared_mlp(I_sh, world):
    H = 128
    g = torch.Generator().manual_seed(I_sh + world)
    W1s = torch.randn(2 * I_sh, H, generator=g).to(torch.bfloat16)
    W2s = torch.randn(H, I_sh, generator=g).to(torch.bfloat16)
    gate, up, cols = [], [], []
    for r in range(world):
        a, w = ep_shared_range(I_sh, world, r)
        assert w % 64 == 0
        s1, s2 = ep_shared_shard(W1s, W2s, world, r)
        if w == 0:
            assert s1 is None and s2 is None
            continue
        assert s1.shape == (2 * w, H) and s2.shape == (H, w)
        gate.append(s1[:w])
        up.append(s1[w:])
        cols.append(s2)
    assert torch.equal(torch.cat(gate + up), W1s)
    assert torch.equal(torch.cat(cols, 1), W2s)


CFG = mi.MoEConfig("ep_cpu", T=24, H=128, I=128, E=8, k=3, renorm=True, n_shared=2, I_shared=128,
                   shared_gate=True)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _partial_oracle(inp, world, rank):
    """The oracle's partial output of one rank: its slot range (SKIP) and its shard of the
    shared experts (concatenated as the GPU runs them), gated by the same sigmoid."""
    cfg = inp["cfg"]
    lo, n = ep_slot_range(cfg.E, world, rank)
    c1, c2 = mi.shared_concat(inp["W1s"], inp["W2s"])
    s1, s2 = ep_shared_shard(c1, c2, world, rank)
    kw = dict(local_start=lo, local_count=n, mode=oracle.NONLOCAL_SKIP)
    if s1 is not None:
        kw.update(W1s=s1[None], W2s=s2[None], shared_gate_w=inp["w_s"])
    res = oracle.moe_layer(inp["x"], inp["Wg"], None, cfg.k, cfg.renorm, inp["W1"][lo:lo + n],
                           inp["W2"][lo:lo + n], **kw)
    return res["out"]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = mi.make_inputs(CFG)
        part = torch.from_numpy(_partial_oracle(inp, world, rank))
        out = ep_reduce_output(part.to(torch.float64))  # fp32 reduction, back to the partial's dtype
        q.put((rank, out.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_partials_reduced_over_gloo_ranks_equal_the_full_layer(world):
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    inp = mi.make_inputs(CFG)
    c1, c2 = mi.shared_concat(inp["W1s"], inp["W2s"])
    full = oracle.moe_layer(inp["x"], inp["Wg"], None, CFG.k, CFG.renorm, inp["W1"], inp["W2"], W1s=c1[None],
                            W2s=c2[None], shared_gate_w=inp["w_s"])["out"]
    for r in range(world):
        # every rank holds the same sum; the fp32 reduction rounds each partial once
        np.testing.assert_allclose(res[r], full, rtol=0, atol=1e-6 * np.abs(full).max())
        assert np.array_equal(res[r], res[0])
