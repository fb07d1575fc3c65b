"""The GPU side of expert parallelism on one GPU.

Reduction mode: each rank's partial output (its slot range under SKIP and its
shard of the shared experts, through the same library calls a rank runs) is
computed in turn, and the partials summed on the host equal the full layer --
against the fp64 oracle and against the one-GPU layer, within the output
tolerance.

All-to-all mode: moe_a2a_regroup moves rows into the oracle's receive-side
order and back, bit for bit; and N ranks held by one process
(a2a_forward_local: the ranks' steps one after another, the exchanges as
device copies) give every rank the one-GPU layer's output on its own tokens,
bit for bit, and the oracle's within the output tolerance -- on mid-size
cases with ragged and empty batches, replica slots, group-limited top-k and
routing on the input, and with the Qwen2-like and redundant-slot workloads'
batches split over 4 and 8 ranks.

Peer reduction (moe_ep_signal / moe_ep_reduce): ranks held by one process
write their partials and flags, then each forms its rows of the sum --
bitwise the rank-order fp32 sum of the partials, two steps in a row (both
slots), as an all-reduce and as a reduce-scatter; a flag nothing raises makes
the bounded wait give up with MOE_ERR_TIMEOUT; and two processes on the GPU
map each other's buffers by CUDA IPC (flags raised and the host synchronised
before any reduce starts, so no kernel waits on the other process).

Ranks run one after another on one GPU: nothing waits on another rank."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import serving_router_gate_gb300 as moe
from serving_router_gate_gb300.expert_parallel import (EPAllToAllLayer, EPMoELayer, PeerReduction, a2a_forward_local,
                                                       ep_row_range)
from serving_router_gate_gb300.layer import layer_from_inputs

from parity_util import check_out, oracle_layer, oracle_threads, sample_tokens, to_cpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _threads():
    oracle_threads()


def _ep_partials(inp, world):
    cfg = inp["cfg"]
    d = lambda t: None if t is None else t.cuda().contiguous()  # noqa: E731
    W1s = W2s = None
    if inp["W1s"] is not None:
        W1s, W2s = mi.shared_concat(inp["W1s"], inp["W2s"])
    x = inp["x"].cuda()
    acc = torch.zeros(cfg.T, cfg.H, dtype=torch.float32, device="cuda")
    for r in range(world):
        ep = EPMoELayer(d(inp["Wg"]), d(inp["W1"]), d(inp["W2"]), cfg.k, cfg.renorm, cfg.T, world, r,
                        logit_bias=d(inp["bias"]), rep_offset=d(inp["rep_offset"]), rep_slots=d(inp["rep_slots"]),
                        W1s=d(W1s), W2s=d(W2s), shared_gate_w=d(inp["w_s"]))
        part = ep.forward(x)  # no process group: the reduction is this rank's partial alone
        acc += part.float()
        assert moe.moe_get_device_status(ep.layer.ws) == 0
    torch.cuda.synchronize()
    return acc.to(torch.bfloat16)


@pytest.mark.parametrize("world", [2, 4])
def test_ep_partials_sum_to_the_full_layer(world):
    cfg = mi.MoEConfig("ep_gpu", T=300, H=256, I=256, E=16, k=4, renorm=True, n_shared=2, I_shared=256,
                       shared_gate=True)
    inp = mi.make_inputs(cfg)
    out = _ep_partials(inp, world)
    ref = oracle_layer(to_cpu(inp))
    check_out(out, ref["out"], f"sum of {world} expert-parallel partials")
    full = layer_from_inputs(inp, "cuda").forward(inp["x"].cuda())
    check_out(out, full.double().cpu().numpy(), "against the one-GPU layer")


def test_ep_with_replica_slots_and_uneven_ranges():
    # 13 slots over 4 ranks (3, 3, 3, 4) with replicas and a Zipf bias; no shared experts
    cfg = mi.MoEConfig("ep_rep", T=200, H=256, I=128, E=10, S=13, n_hot=3, zipf_s=1.1, k=3, renorm=True)
    inp = mi.make_inputs(cfg)
    out = _ep_partials(inp, 4)
    check_out(out, oracle_layer(to_cpu(inp))["out"], "sum of partials with replica slots")


# --------------------------------------------------------------------------- all-to-all mode

def _bits(t):
    return t.view(torch.int16).cpu()


@pytest.mark.parametrize("N,S_l,H,seed", [(2, 5, 64, 0), (4, 3, 192, 1), (8, 36, 2048, 2), (1, 7, 256, 3),
                                          (64, 64, 64, 4), (3, 1, 7168, 5)])
def test_a2a_regroup_matches_the_oracle_order(N, S_l, H, seed):
    g = torch.Generator().manual_seed(seed)
    counts = torch.randint(0, 5, (N, S_l), generator=g, dtype=torch.int32)
    counts[0, 0] = 0       # an empty block
    if N > 2:
        counts[N - 2] = 0  # a source that sent nothing
    R = int(counts.sum())
    cap = R + 3            # rows past the total are neither read nor written
    src = torch.randn(cap, H, generator=g).to(torch.bfloat16).cuda()
    nan = torch.full((cap, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(moe.MOE_WS_HEADER_BYTES, dtype=torch.uint8, device="cuda")
    rc = counts.cuda()
    off = torch.full((S_l + 1,), -7, dtype=torch.int32, device="cuda")
    dst = nan.clone()
    row_map = torch.full((cap,), -5, dtype=torch.int32, device="cuda")
    before = moe.moe_get_launch_count()
    moe.moe_a2a_regroup(rc, src, dst, moe.MOE_A2A_TO_GEMM, off, ws, row_map=row_map)
    assert moe.moe_get_launch_count() == before + 1
    ref_off, gemm_row, exch_row = oracle.a2a_regroup(counts.numpy())
    assert off.cpu().tolist() == ref_off.tolist()
    assert row_map[:R].cpu().tolist() == exch_row.tolist()
    assert row_map[R:].cpu().tolist() == [-5] * (cap - R)
    exch = torch.from_numpy(exch_row.astype(np.int64))
    assert torch.equal(_bits(dst[:R]), _bits(src[:R])[exch])
    assert torch.equal(_bits(dst[R:]), _bits(nan[R:]))
    back = nan.clone()
    moe.moe_a2a_regroup(rc, dst, back, moe.MOE_A2A_TO_EXCHANGE, None, ws)
    assert torch.equal(_bits(back[:R]), _bits(src[:R]))
    assert torch.equal(_bits(back[R:]), _bits(nan[R:]))
    assert moe.moe_get_device_status(ws) == 0


@pytest.mark.parametrize("bad", ["total", "negative"])
def test_a2a_regroup_flags_bad_counts_and_moves_nothing(bad):
    counts = torch.tensor([[3, 2], [1, 4]], dtype=torch.int32)
    cap = 10
    if bad == "total":
        cap = 9            # 10 rows announced, room for 9
    else:
        counts[1, 0] = -1
    src = torch.randn(cap, 64).to(torch.bfloat16).cuda()
    dst = torch.zeros(cap, 64, dtype=torch.bfloat16, device="cuda")
    off = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(moe.MOE_WS_HEADER_BYTES, dtype=torch.uint8, device="cuda")
    moe.moe_a2a_regroup(counts.cuda(), src, dst, moe.MOE_A2A_TO_GEMM, off, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_DEVICE_BOUNDS
    assert int(dst.view(torch.int16).abs().sum()) == 0
    assert off.cpu().tolist() == [-7, -7, -7]


@pytest.mark.parametrize("shared", [False, True])
def test_grouped_fc2_scatter_equals_fc2_with_rows_moved(shared):
    # 7 groups with ragged counts (an empty one, a partial last tile), a shared problem
    g = torch.Generator().manual_seed(11)
    H, I, G, T = 256, 192, 7, 40
    counts = [130, 0, 5, 64, 257, 1, 33]
    rows = sum(counts)
    cap = rows + 9
    offsets = torch.tensor([0] + list(np.cumsum(counts)), dtype=torch.int32, device="cuda")
    h = (torch.randn(cap, I, generator=g) * 0.5).to(torch.bfloat16).cuda()
    W2 = (torch.randn(G, H, I, generator=g) * 0.05).to(torch.bfloat16).cuda()
    h_sh = W2s = None
    if shared:
        h_sh = (torch.randn(T, 128, generator=g) * 0.5).to(torch.bfloat16).cuda()
        W2s = (torch.randn(H, 128, generator=g) * 0.05).to(torch.bfloat16).cuda()
    ws = torch.zeros(moe.MOE_WS_HEADER_BYTES, dtype=torch.uint8, device="cuda")
    y = torch.empty(cap, H, dtype=torch.bfloat16, device="cuda")
    ysh = torch.empty(T, H, dtype=torch.bfloat16, device="cuda") if shared else None
    moe.moe_grouped_fc2(h, offsets, W2, h_sh, W2s, y, ysh, ws)
    perm = torch.randperm(rows, generator=g)
    y_row = torch.full((cap,), -1, dtype=torch.int32)
    y_row[:rows] = perm.to(torch.int32)
    y2 = torch.full((cap, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    ysh2 = torch.empty(T, H, dtype=torch.bfloat16, device="cuda") if shared else None
    moe.moe_grouped_fc2_scatter(h, offsets, W2, h_sh, W2s, y_row.cuda(), y2, ysh2, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    assert torch.equal(_bits(y2)[perm], _bits(y[:rows]))
    assert torch.equal(_bits(y2[rows:]), _bits(torch.full((cap - rows, H), float("nan"), dtype=torch.bfloat16)))
    if shared:
        assert torch.equal(_bits(ysh2), _bits(ysh))


def _a2a_layers(inp, world, max_T, recv_cap=None):
    cfg = inp["cfg"]
    d = lambda t: None if t is None else t.cuda().contiguous()  # noqa: E731
    W1s = W2s = None
    if inp["W1s"] is not None:
        W1s, W2s = mi.shared_concat(inp["W1s"], inp["W2s"])
    Wg, W1, W2, bias, ro, rs, W1s, W2s, ws_ = (d(inp["Wg"]), d(inp["W1"]), d(inp["W2"]), d(inp["bias"]),
                                               d(inp["rep_offset"]), d(inp["rep_slots"]), d(W1s), d(W2s),
                                               d(inp["w_s"]))
    return [EPAllToAllLayer(Wg, W1, W2, cfg.k, cfg.renorm, max_T, world, r, logit_bias=bias, rep_offset=ro,
                            rep_slots=rs, W1s=W1s, W2s=W2s, shared_gate_w=ws_, n_group=cfg.n_group,
                            topk_group=cfg.topk_group, on_input=cfg.on_input, recv_cap=recv_cap)
            for r in range(world)]


def _check_a2a(inp, xs, recv_cap=None, n_oracle=None, bitwise=True):
    """Every rank's output: bitwise the one-GPU layer's on its tokens (unless the one-GPU
    layer splits the shared FC2 over K at small batches, which the all-to-all layer's stage
    calls do not), and the oracle's within the output tolerance (on n_oracle sampled tokens,
    or all)."""
    cfg = inp["cfg"]
    world = len(xs)
    max_T = max(1, max(x.shape[0] for x in xs))
    layers = _a2a_layers(inp, world, max_T, recv_cap)
    outs = a2a_forward_local(layers, [x.cuda() for x in xs])
    torch.cuda.synchronize()
    for L in layers:
        assert moe.moe_get_device_status(L.ws) == 0
    one = layer_from_inputs(inp, "cuda", max_T=max_T)
    inp_cpu = to_cpu(inp)
    for r, (x, out) in enumerate(zip(xs, outs)):
        T = x.shape[0]
        assert out.shape == (T, cfg.H)
        if T == 0:
            continue
        if bitwise:
            ref = one.forward(x.cuda())
            assert torch.equal(_bits(out), _bits(ref)), f"rank {r}: differs from the one-GPU layer"
        tok = None if n_oracle is None else sample_tokens(T, n_oracle, seed=r)
        part = oracle_layer(dict(inp_cpu, x=x.cpu()), tokens=tok)
        check_out(out if tok is None else out[torch.from_numpy(tok).cuda()], part["out"], f"rank {r}")
    # every pair went to exactly one rank: the rows received sum to the pairs sent
    assert sum(L.rows_in for L in layers) == sum(L.rows_out for L in layers) == cfg.k * sum(x.shape[0] for x in xs)
    return layers


@pytest.mark.parametrize("tokens", [[129, 64], [300, 0, 77, 513]])
def test_a2a_layer_gives_each_rank_its_layer(tokens):
    cfg = mi.MoEConfig("a2a_gpu", T=16, H=256, I=256, E=16, k=4, renorm=True, n_shared=2, I_shared=128,
                       shared_gate=True)
    inp = mi.make_inputs(cfg)
    xs = [mi.rank_tokens(cfg, r, T) for r, T in enumerate(tokens)]
    _check_a2a(inp, xs)


@pytest.mark.parametrize("variant", ["replicas", "grouped", "on_input"])
def test_a2a_layer_routing_variants(variant):
    if variant == "replicas":  # 13 slots over 4 ranks (3, 3, 3, 4), Zipf bias, no shared experts
        cfg = mi.MoEConfig("a2a_rep", T=8, H=256, I=128, E=10, S=13, n_hot=3, zipf_s=1.1, k=3, renorm=True)
    elif variant == "grouped":
        cfg = mi.MoEConfig("a2a_grp", T=8, H=256, I=128, E=16, k=4, renorm=True, n_group=4, topk_group=2,
                           n_shared=1, I_shared=128)
    else:
        cfg = mi.MoEConfig("a2a_oni", T=8, H=256, I=128, E=12, k=2, renorm=False, on_input=True)
    inp = mi.make_inputs(cfg)
    xs = [mi.rank_tokens(cfg, r, T) for r, T in enumerate([200, 33, 0, 150])]
    _check_a2a(inp, xs)


def test_a2a_layer_at_decode_sizes():
    # DeepSeek-V2-Lite-like shapes (64 experts, k = 6, two shared experts of 2816): ranks with
    # 1, 8, 0 and 32 tokens -- the tiny permutation over all slots, short GEMM tiles and FC2
    # storing short tiles through its row map
    cfg = mi.CONFIGS["dsv2_lite_like_decode_t32"]
    inp = mi.make_inputs(cfg, device="cpu", weights_device="cuda")
    xs = [mi.rank_tokens(cfg, r, T) for r, T in enumerate([1, 8, 0, 32])]
    _check_a2a(inp, xs, bitwise=False)


def test_a2a_regroup_edge_cases():
    ws = torch.zeros(moe.MOE_WS_HEADER_BYTES, dtype=torch.uint8, device="cuda")
    # nothing received: offsets all zero, no row touched
    counts = torch.zeros(3, 5, dtype=torch.int32)
    src = torch.randn(4, 64).to(torch.bfloat16).cuda()
    dst = torch.full((4, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    off = torch.full((6,), -1, dtype=torch.int32, device="cuda")
    moe.moe_a2a_regroup(counts.cuda(), src, dst, moe.MOE_A2A_TO_GEMM, off, ws)
    torch.cuda.synchronize()
    assert off.cpu().tolist() == [0] * 6 and bool((dst == 7.0).all())
    # a total equal to the buffers' rows exactly
    counts = torch.tensor([[2, 1], [0, 3]], dtype=torch.int32)
    src = torch.randn(6, 128).to(torch.bfloat16).cuda()
    dst = torch.empty_like(src)
    off = torch.empty(3, dtype=torch.int32, device="cuda")
    moe.moe_a2a_regroup(counts.cuda(), src, dst, moe.MOE_A2A_TO_GEMM, off, ws)
    torch.cuda.synchronize()
    ref_off, _, exch_row = oracle.a2a_regroup(counts.numpy())
    assert off.cpu().tolist() == ref_off.tolist()
    assert torch.equal(_bits(dst), _bits(src)[torch.from_numpy(exch_row.astype(np.int64))])
    assert moe.moe_get_device_status(ws) == 0


def test_a2a_qwen2_moe_like_batch_over_4_ranks():
    # the workload's 4096 tokens as four ranks' batches of 1024
    inp = mi.make_inputs(mi.CONFIGS["qwen2_moe_like_prefill"], device="cpu", weights_device="cuda")
    xs = list(inp["x"].split(1024))
    _check_a2a(inp, xs, n_oracle=12)


def test_a2a_redundant_slots_batch_over_8_ranks():
    # the workload's 16384 tokens as eight ranks' batches of 2048; 288 slots, 36 per rank
    inp = mi.make_inputs(mi.CONFIGS["redundant_slots_prefill"], device="cpu", weights_device="cuda")
    xs = list(inp["x"].split(2048))
    layers = _check_a2a(inp, xs, recv_cap=3 * 2048 * 8, n_oracle=6)
    assert max(L.rows_in for L in layers) <= 3 * 2048 * 8


# --------------------------------------------------------------------------- peer reduction

def _rank_order_sum(parts):
    acc = parts[0].float()
    for p in parts[1:]:
        acc = acc + p.float()
    return acc.to(torch.bfloat16)


def _peer_case(world, scatter, steps=((300, 0), (177, 1))):
    cfg = mi.MoEConfig("ep_peer", T=300, H=256, I=256, E=16, k=4, renorm=True, n_shared=2, I_shared=256,
                       shared_gate=True)
    inp = mi.make_inputs(cfg)
    d = lambda t: None if t is None else t.cuda().contiguous()  # noqa: E731
    W1s, W2s = mi.shared_concat(inp["W1s"], inp["W2s"])
    reds = PeerReduction.local_set(cfg.T, cfg.H, world, "cuda", scatter=scatter)
    eps = [EPMoELayer(d(inp["Wg"]), d(inp["W1"]), d(inp["W2"]), cfg.k, cfg.renorm, cfg.T, world, r,
                      W1s=d(W1s), W2s=d(W2s), shared_gate_w=d(inp["w_s"]), peer=reds[r]) for r in range(world)]
    inp_cpu = to_cpu(inp)
    for T, seed in steps:  # two steps: slots 1 and 0
        x = inp["x"][:T] if seed == 0 else mi.rank_tokens(cfg, seed, T)
        xd = x.cuda()
        for e in eps:
            e.write_partial(xd)
        outs = [e.peer.reduce().clone() for e in eps]
        torch.cuda.synchronize()
        for e in eps:
            assert moe.moe_get_device_status(e.peer.ws) == 0
            assert moe.moe_get_device_status(e.layer.ws) == 0
        ep0 = eps[0].peer.epoch
        parts = [r.slots[ep0 % 2, :T] for r in reds]
        ref = _rank_order_sum(parts)
        for r, out in enumerate(outs):
            lo, hi = ep_row_range(T, world, r) if scatter else (0, T)
            assert torch.equal(_bits(out[lo:hi]), _bits(ref[lo:hi])), f"rank {r}, T={T}"
        full = torch.cat([outs[r][slice(*ep_row_range(T, world, r))] for r in range(world)]) if scatter else outs[0]
        check_out(full, oracle_layer(dict(inp_cpu, x=x.cpu()))["out"], f"peer reduction of {world} ranks, T={T}")


@pytest.mark.parametrize("world,scatter", [(2, False), (4, False), (3, True), (4, True)])
def test_peer_reduction_of_local_ranks(world, scatter):
    _peer_case(world, scatter)


def test_peer_reduction_wait_times_out_on_a_missing_flag():
    H, T = 256, 64
    reds = PeerReduction.local_set(T, H, 2, "cuda")
    for r in reds:
        r.begin(T).fill_(1.0)
    reds[0].signal()  # rank 1 never raises its flag
    out = reds[0].out
    out.fill_(3.0)
    moe.moe_set_wait_timeout_ns(2_000_000)
    try:
        reds[0].reduce()
        torch.cuda.synchronize()
    finally:
        moe.moe_set_wait_timeout_ns(4_000_000_000)
    assert moe.moe_get_device_status(reds[0].ws) == moe.MOE_ERR_TIMEOUT
    assert bool((out == 3.0).all())  # nothing written
    reds[1].signal()  # now both flags are up: the same epoch reduces
    res = reds[0].reduce()
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(reds[0].ws) == 0
    assert bool((res == 2.0).all())


def _ipc_worker(rank, port, q):
    import os
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        moe.moe_set_wait_timeout_ns(1_000_000_000)  # any wait ends within a second
        cfg = mi.MoEConfig("ep_ipc", T=200, H=256, I=128, E=8, k=2, renorm=True)
        inp = mi.make_inputs(cfg)
        d = lambda t: None if t is None else t.cuda().contiguous()  # noqa: E731
        red = PeerReduction(cfg.T, cfg.H, 2, rank, "cuda")
        ep = EPMoELayer(d(inp["Wg"]), d(inp["W1"]), d(inp["W2"]), cfg.k, cfg.renorm, cfg.T, 2, rank, peer=red)
        res = []
        for T in (200, 131):
            x = inp["x"][:T].cuda()
            ep.write_partial(x)          # partial, then this rank's flag in both ranks' arrays
            torch.cuda.synchronize()
            dist.barrier()               # both flags are up before either reduce starts
            out = red.reduce().clone()
            torch.cuda.synchronize()
            res.append((out.cpu(), red.slots[red.epoch % 2, :T].cpu(), moe.moe_get_device_status(red.ws)))
            dist.barrier()               # both reduces done before the next step's partials
        red.close()
        dist.barrier()                   # no mapping left before either process frees its buffers
        q.put((rank, res))
    finally:
        dist.destroy_process_group()


def test_peer_reduction_across_two_processes_by_ipc():
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ipc_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=600) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for step in range(2):
        (o0, p0, s0), (o1, p1, s1) = res[0][step], res[1][step]
        assert s0 == 0 and s1 == 0
        ref = _rank_order_sum([p0, p1])
        assert torch.equal(_bits(o0), _bits(ref)) and torch.equal(_bits(o1), _bits(ref))


# --------------------------------------------------------------------------- poisoned buffers

_A2A_BUFS = ("topk_ids", "topk_w", "slot_ids", "counts", "offsets", "perm_src", "pair_row", "send", "recv_counts",
             "local_offsets", "recv", "x_loc", "row_map", "h", "h_sh", "y_sh", "out")


def _a2a_poisoned_run(layers, xs, byte):
    for L in layers:
        for name in _A2A_BUFS:
            t = getattr(L, name)
            if t is not None:
                t.view(torch.uint8).fill_(byte)
        L.ws[moe.MOE_WS_HEADER_BYTES:].fill_(byte)  # the header (status word, counters) stays
    torch.cuda.synchronize()
    outs = [o.clone() for o in a2a_forward_local(layers, [x.cuda() for x in xs])]
    torch.cuda.synchronize()
    return outs


def test_a2a_layer_reads_no_unwritten_memory():
    # every buffer of every rank filled with all-ones bytes (NaN in bf16 / fp32, -1 in int32)
    # before a forward: the outputs must equal those of a forward on zero-filled buffers
    cfg = mi.MoEConfig("a2a_poison", T=16, H=256, I=256, E=16, k=4, renorm=True, n_shared=1, I_shared=256,
                       shared_gate=True)
    inp = mi.make_inputs(cfg)
    xs = [mi.rank_tokens(cfg, r, T) for r, T in enumerate([300, 0, 77, 513])]
    layers = _a2a_layers(inp, 4, 513)
    clean = _a2a_poisoned_run(layers, xs, 0x00)
    poisoned = _a2a_poisoned_run(layers, xs, 0xFF)
    for r, (a, b) in enumerate(zip(clean, poisoned)):
        assert torch.equal(_bits(a), _bits(b)), f"rank {r} depends on unwritten memory"
        assert torch.isfinite(b.float()).all()
    for L in layers:
        assert moe.moe_get_device_status(L.ws) == 0


def test_peer_reduction_reads_no_unwritten_memory():
    # the partial slots and outputs poisoned before a step (the flags are state and stay)
    H, T, world = 256, 100, 3
    g = torch.Generator().manual_seed(5)
    parts = [(torch.randn(T, H, generator=g)).to(torch.bfloat16).cuda() for _ in range(world)]
    results = []
    for byte in (0x00, 0xFF):
        reds = PeerReduction.local_set(128, H, world, "cuda", scatter=True)
        for r in reds:
            r.slots.view(torch.uint8).fill_(byte)
            r.out.view(torch.uint8).fill_(byte)
        for r, p in zip(reds, parts):
            r.begin(T).copy_(p)
            r.signal()
        outs = [r.reduce().clone() for r in reds]
        torch.cuda.synchronize()
        full = torch.cat([outs[r][slice(*ep_row_range(T, world, r))] for r in range(world)])
        results.append(full)
        for r in reds:
            assert moe.moe_get_device_status(r.ws) == 0
    assert torch.equal(_bits(results[0]), _bits(results[1]))
    assert torch.equal(_bits(results[0]), _bits(_rank_order_sum(parts)))
