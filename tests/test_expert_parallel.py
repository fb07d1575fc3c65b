"""Expert parallelism (serving_router_gate_gb300.expert_parallel) on the CPU.

Reduction mode: the slot ranges and shared-expert shards partition the layer,
and with gloo ranks (world sizes 2 and 4) the one SUM reduction of the ranks'
partial outputs -- each computed by the fp64 oracle on that rank's slot range
(SKIP) and shared shard -- equals the oracle's full layer.

All-to-all mode: with gloo ranks that each hold their own tokens, the
package's split sizes and exchanges (DistExchange over gloo) carry every
pair's row to the rank owning its slot and the expert outputs back; with the
oracle standing in for the kernels on each rank (routing and permutation,
the receive-side order, the expert MLPs, the combine), every rank's output
equals the oracle's layer on its own tokens.

The GPU side of both modes runs the library's calls; it is checked on a GPU
in tests/test_gpu_expert_parallel.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import moe_inputs as mi
import oracle
from serving_router_gate_gb300.expert_parallel import (DistExchange, a2a_count_splits, a2a_recv_splits,
                                                       a2a_send_splits, ep_reduce_output, ep_row_range,
                                                       ep_shared_range, ep_shared_shard, ep_slot_range, wrap_int32)


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


@pytest.mark.parametrize("T,world", [(300, 2), (300, 4), (7, 8), (1, 3), (4096, 8), (0, 2)])
def test_reduce_scatter_row_ranges_cover_every_row_once(T, world):
    seen = []
    for r in range(world):
        lo, hi = ep_row_range(T, world, r)
        assert lo == (seen[-1] + 1 if seen else 0) or lo == hi
        seen.extend(range(lo, hi))
    assert seen == list(range(T))
    sizes = [ep_row_range(T, world, r)[1] - ep_row_range(T, world, r)[0] for r in range(world)]
    assert max(sizes) - min(sizes) <= 1


def test_epochs_wrap_to_int32_keeping_order_and_parity():
    assert wrap_int32(1) == 1 and wrap_int32(2 ** 31 - 1) == 2 ** 31 - 1
    assert wrap_int32(2 ** 31) == -2 ** 31 and wrap_int32(2 ** 32 + 5) == 5
    for e in (1, 2 ** 31 - 2, 2 ** 31 - 1, 2 ** 31, 2 ** 32 - 1, 2 ** 32 + 7):
        # the kernels compare int32 differences: the next epoch is ahead, the last one behind
        nxt = wrap_int32(wrap_int32(e + 1) - wrap_int32(e))
        prv = wrap_int32(wrap_int32(e - 1) - wrap_int32(e))
        assert nxt == 1 and prv == -1
        assert wrap_int32(e) % 2 == e % 2  # the slot parity survives the wrap


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


# --------------------------------------------------------------------------- all-to-all mode

def test_a2a_split_sizes():
    S, world = 13, 4
    assert a2a_count_splits(S, world) == [ep_slot_range(S, world, d)[1] for d in range(world)]
    assert sum(a2a_count_splits(S, world)) == S
    offsets = np.array([0, 2, 2, 5, 6, 6, 6, 9, 10, 10, 12, 15, 15, 20])  # S + 1 = 14 entries
    sp = a2a_send_splits(offsets, S, world)
    # ranges (0, 3), (3, 3), (6, 3), (9, 4): rows offsets[hi] - offsets[lo]
    assert sp == [5, 1, 4, 10] and sum(sp) == offsets[-1]
    rc = torch.tensor([[1, 0, 2], [0, 0, 0], [4, 1, 1]], dtype=torch.int32)
    assert a2a_recv_splits(rc) == [3, 0, 6]


A2A_CFG = mi.MoEConfig("a2a_cpu", T=24, H=128, I=128, E=8, k=3, renorm=True, n_shared=1, I_shared=128,
                       shared_gate=True)
A2A_TOKENS = {2: [24, 9], 4: [24, 0, 17, 5]}  # each rank's own batch (one rank without tokens)


def _a2a_rank_output(inp, x, world, rank, ex):
    """One rank of the all-to-all layer with the oracle in place of the kernels."""
    cfg = inp["cfg"]
    S, k, H = cfg.E, cfg.k, cfg.H
    lo, S_l = ep_slot_range(S, world, rank)
    T = x.shape[0]
    # dispatch: route, slot map, group the pairs by slot (all S slots)
    if T:
        ids, w, _ = oracle.route(x, inp["Wg"], None, k, cfg.renorm)
        counts, offsets, perm_src, pair_row = oracle.permute(oracle.slot_map(ids), S)
        send = x[torch.from_numpy(perm_src.astype(np.int64) // k)]
    else:
        w = np.zeros((0, k))
        counts, offsets, pair_row = np.zeros(S, np.int32), np.zeros(S + 1, np.int32), np.zeros(0, np.int32)
        send = torch.empty((0, H), dtype=torch.bfloat16)
    recv_counts = torch.empty((world, S_l), dtype=torch.int32)
    ex.all_to_all(recv_counts.view(-1), torch.from_numpy(counts), [S_l] * world, a2a_count_splits(S, world))
    send_splits = a2a_send_splits(offsets, S, world)
    recv_splits = a2a_recv_splits(recv_counts)
    recv = torch.empty((sum(recv_splits), H), dtype=torch.bfloat16)
    ex.all_to_all(recv, send.contiguous(), recv_splits, send_splits)
    # experts: the received rows in slot order, each through its slot's expert
    off_l, gemm_row, exch_row = oracle.a2a_regroup(recv_counts.numpy())
    y_loc = np.zeros((recv.shape[0], H))
    for c in range(S_l):
        for r in range(off_l[c], off_l[c + 1]):
            y_loc[r] = oracle.expert_mlp(recv[int(exch_row[r])], inp["W1"][lo + c], inp["W2"][lo + c])[0]
    y_ret = torch.empty((send.shape[0], H), dtype=torch.float64)
    ex.all_to_all(y_ret, torch.from_numpy(y_loc[gemm_row]).contiguous(), send_splits, recv_splits)
    # combine: fixed j order, then the gated shared expert on the rank's own tokens
    out = np.zeros((T, H))
    W1c, W2c = mi.shared_concat(inp["W1s"], inp["W2s"])
    ws = inp["w_s"].to(torch.float64).numpy()
    y_ret = y_ret.numpy()
    for t in range(T):
        for j in range(k):
            out[t] += w[t, j] * y_ret[pair_row[t * k + j]]
        g = 1.0 / (1.0 + np.exp(-float(x[t].to(torch.float64).numpy() @ ws)))
        out[t] += g * oracle.expert_mlp(x[t], W1c, W2c)[0]
    return out


def _a2a_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = mi.make_inputs(A2A_CFG)
        x = mi.rank_tokens(A2A_CFG, rank, A2A_TOKENS[world][rank])
        q.put((rank, _a2a_rank_output(inp, x, world, rank, DistExchange())))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_a2a_exchange_over_gloo_ranks_gives_each_rank_its_layer(world):
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_a2a_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    inp = mi.make_inputs(A2A_CFG)
    c1, c2 = mi.shared_concat(inp["W1s"], inp["W2s"])
    for r in range(world):
        x = mi.rank_tokens(A2A_CFG, r, A2A_TOKENS[world][r])
        assert res[r].shape == (x.shape[0], A2A_CFG.H)
        if x.shape[0] == 0:
            continue
        ref = oracle.moe_layer(x, inp["Wg"], None, A2A_CFG.k, A2A_CFG.renorm, inp["W1"], inp["W2"], W1s=c1[None],
                               W2s=c2[None], shared_gate_w=inp["w_s"])["out"]
        np.testing.assert_allclose(res[r], ref, rtol=0, atol=1e-12 * np.abs(ref).max())
