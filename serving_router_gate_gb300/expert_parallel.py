"""Expert parallelism across GPUs: each rank owns a contiguous range of expert
slots and a shard of the shared experts, computes a partial layer output, and
one SUM reduction over the ranks gives the layer output.

Method (vLLM EP-aware FusedMoE override, ep_fused_moe_patch.py):
  * module docstring "EP expert dispatch": top-k routing gives global expert
    ids, identical on every rank; each rank masks the experts outside its range
    (weight 0) and remaps its own to local ids -- moe_permute with a local range
    and MOE_NONLOCAL_SKIP;
  * the patched __init__: E_local = E / ep_size experts per rank, contiguous
    ranges, renormalisation over all k before the mask;
  * ep_reduce_output: the routed partial plus the shared experts' partial (a
    row-parallel shard: each rank holds a slice of their intermediate size),
    then one all-reduce -- DeepSpeed PR #6964 likewise forms the layer's
    reduction once, after the weighted sum of the selected experts' outputs.

Readings taken here: slot ranges split S as evenly as contiguous ranges allow
(rank r owns [r S / N, (r + 1) S / N)), which is E / N when N divides S; the
shared experts' intermediate is split the same way in units of 64 (the
library's row granularity); the reduction runs in fp32 (the pages do not fix
its precision) and the result is rounded to bf16 once.

Every rank calls the same three library calls as a one-GPU layer (moe_route,
moe_permute with its range, moe_forward with its shard); only the reduction is
a collective -- torch.distributed's all-reduce, or (PeerReduction) the
library's own kernels reading every rank's partial in rank order through
mapped memory, with bounded flag waits.

The all-to-all mode (EPAllToAllLayer, below) follows TensorRT-LLM PR #10985's
other path: every rank holds its own tokens, dispatches each pair's row to
the rank owning its slot and gets the expert outputs back.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from . import MOE_NONLOCAL_SKIP
from .layer import MoELayer


def ep_slot_range(S: int, world: int, rank: int) -> Tuple[int, int]:
    """(first slot, slot count) of rank `rank` among `world` ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if world > S:
        raise ValueError(f"{world} ranks for {S} slots")
    lo, hi = rank * S // world, (rank + 1) * S // world
    return lo, hi - lo


def ep_shared_range(I_shared: int, world: int, rank: int, unit: int = 64) -> Tuple[int, int]:
    """(first column, width) of rank `rank`'s slice of the shared experts' intermediate
    size, in whole units of `unit` columns (a rank may get none)."""
    if I_shared % unit:
        raise ValueError(f"shared intermediate {I_shared} is not a multiple of {unit}")
    n = I_shared // unit
    lo, hi = rank * n // world, (rank + 1) * n // world
    return lo * unit, (hi - lo) * unit


def ep_shared_shard(W1s: torch.Tensor, W2s: torch.Tensor, world: int, rank: int):
    """The row-parallel shard of the shared experts (as one concatenated MLP:
    W1s [2 I_sh, H] gate rows then up rows, W2s [H, I_sh]) that rank `rank` holds:
    gate rows [a, a + w), up rows [I_sh + a, I_sh + a + w), W2s columns [a, a + w).
    Returns (W1 shard [2 w, H], W2 shard [H, w]) or (None, None) for w = 0."""
    I_sh = W2s.shape[1]
    a, w = ep_shared_range(I_sh, world, rank)
    if w == 0:
        return None, None
    W1 = torch.cat([W1s[a:a + w], W1s[I_sh + a:I_sh + a + w]], 0).contiguous()
    W2 = W2s[:, a:a + w].contiguous()
    return W1, W2


def ep_reduce_output(partial: torch.Tensor, group=None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Sum of the ranks' partial outputs [T, H] (routed + shared on each rank), in fp32,
    rounded once to the partial's dtype: the layer output on every rank."""
    import torch.distributed as dist
    acc = partial.float()
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    res = acc.to(partial.dtype)
    if out is not None:
        out.copy_(res)
        return out
    return res


def wrap_int32(v: int) -> int:
    """v as the signed 32-bit integer it wraps to (the flags' representation of an epoch)."""
    return ((int(v) + 2 ** 31) % 2 ** 32) - 2 ** 31


def ep_row_range(T: int, world: int, rank: int) -> Tuple[int, int]:
    """Rows [lo, hi) of a [T, H] output that rank `rank` keeps in the reduce-scatter (the
    vLLM EP patch's ep_reduce_scatter_output): contiguous, as even as T allows."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    return rank * T // world, (rank + 1) * T // world


class PeerReduction:
    """The one SUM of expert parallelism by plain loads of every rank's partial
    (moe_ep_signal / moe_ep_reduce) instead of a collective library.

    Each rank holds two bf16 partial slots [max_T, H] and an int32 flag per rank, all in
    its own GPU's memory; the other ranks' slots and flags are mapped into this process
    (CUDA IPC, handles exchanged over the process group), or -- for ranks held by one
    process on one device (local_set) -- are plain device addresses.  Per step:
    begin(T) advances the epoch e and returns slot e % 2 to write the partial into;
    signal() raises this rank's flag to e in every rank's array once the partial is
    written; reduce() waits for every rank's flag e and forms this rank's rows of the
    sum (all rows, or its slice with scatter=True) in rank order.  The flags hold e as a
    32-bit integer that wraps around (the kernels compare differences)."""

    def __init__(self, max_T: int, H: int, world: int, rank: int, device, group=None, scatter: bool = False,
                 _exchange: bool = True):
        from . import MOE_WS_HEADER_BYTES, moe_workspace_init
        if not 1 <= world <= 16:
            raise ValueError("1 to 16 ranks")
        self.max_T, self.H, self.world, self.rank = int(max_T), int(H), int(world), int(rank)
        self.group, self.scatter = group, bool(scatter)
        self.slots = torch.empty((2, self.max_T, self.H), dtype=torch.bfloat16, device=device)
        self.flags = torch.zeros((self.world,), dtype=torch.int32, device=device)
        self.ws = torch.empty((MOE_WS_HEADER_BYTES,), dtype=torch.uint8, device=device)
        moe_workspace_init(self.ws)
        self.out = torch.empty((self.max_T, self.H), dtype=torch.bfloat16, device=device)
        self.epoch = 0
        self._imported = []
        self.peer_slots = self.peer_flags = None
        if _exchange:
            self._map_peers()

    def _map_peers(self):
        """Exchange IPC handles of the slots and flags over the process group and map the
        other ranks' buffers."""
        import torch.distributed as dist
        from . import moe_ipc_export, moe_ipc_import
        mine = (moe_ipc_export(self.slots), moe_ipc_export(self.flags))
        allh = [None] * self.world
        dist.all_gather_object(allh, mine, group=self.group)
        self.peer_slots, self.peer_flags = [], []
        for n, ((hs, os_), (hf, of)) in enumerate(allh):
            if n == self.rank:
                self.peer_slots.append(self.slots.data_ptr())
                self.peer_flags.append(self.flags.data_ptr())
                continue
            a, b = moe_ipc_import(hs, os_), moe_ipc_import(hf, of)
            self._imported += [(a, os_), (b, of)]
            self.peer_slots.append(a)
            self.peer_flags.append(b)

    @classmethod
    def local_set(cls, max_T: int, H: int, world: int, device, scatter: bool = False):
        """The reductions of `world` ranks held by one process on one device, wired to
        each other's buffers directly."""
        reds = [cls(max_T, H, world, r, device, scatter=scatter, _exchange=False) for r in range(world)]
        for r in reds:
            r.peer_slots = [o.slots.data_ptr() for o in reds]
            r.peer_flags = [o.flags.data_ptr() for o in reds]
        return reds

    def begin(self, T: int) -> torch.Tensor:
        """The slot [T, H] this step's partial goes into (the epoch advances)."""
        assert 0 < T <= self.max_T
        self.epoch += 1
        self.T = int(T)
        return self.slots[self.epoch % 2, :T]

    def _epoch32(self) -> int:
        return wrap_int32(self.epoch)

    def signal(self, stream=None) -> None:
        from . import moe_ep_signal
        moe_ep_signal(self.peer_flags, self.rank, self._epoch32(), stream)

    def rows(self):
        return ep_row_range(self.T, self.world, self.rank) if self.scatter else (0, self.T)

    def reduce(self, stream=None) -> torch.Tensor:
        """This rank's rows of the sum over the ranks, bf16 [T, H] (rows outside its slice
        unwritten with scatter=True)."""
        from . import moe_ep_reduce
        slot_bytes = self.max_T * self.H * 2 * (self.epoch % 2)
        lo, hi = self.rows()
        out = self.out[:self.T]
        moe_ep_reduce([p + slot_bytes for p in self.peer_slots], self.flags, self._epoch32(), lo, hi, out,
                      self.ws, stream)
        return out

    def close(self) -> None:
        from . import moe_ipc_close
        for a, off in self._imported:
            moe_ipc_close(a, off)
        self._imported = []


class EPMoELayer:
    """One rank's share of an expert-parallel MoE layer.

    Wg [E, H] (replicated), W1 [S, 2I, H], W2 [S, H, I] (all slots; only this
    rank's range is kept), optional shared experts W1s [2 I_sh, H], W2s [H, I_sh]
    (concatenated; only this rank's shard is kept) and their gate vector; further
    keyword options (routing variant, weight format) go to MoELayer as they are.
    forward(x) returns the full layer output [T, H] after the reduction."""

    def __init__(self, Wg, W1, W2, k, renorm, max_T, world: int, rank: int, logit_bias=None, rep_offset=None,
                 rep_slots=None, W1s=None, W2s=None, shared_gate_w=None, group=None,
                 peer: Optional[PeerReduction] = None, **layer_options):
        S = W1.shape[0]
        self.world, self.rank, self.group = world, rank, group
        # peer: the reduction by plain loads of the ranks' partials (moe_ep_reduce) instead of
        # the all-reduce of a collective library
        self.peer = peer
        self.start, self.count = ep_slot_range(S, world, rank)
        W1l = W1[self.start:self.start + self.count].contiguous()
        W2l = W2[self.start:self.start + self.count].contiguous()
        W1sh = W2sh = None
        gate = None
        if W1s is not None:
            W1sh, W2sh = ep_shared_shard(W1s, W2s, world, rank)
            gate = shared_gate_w if W1sh is not None else None
        self.layer = MoELayer(Wg, W1l, W2l, k, renorm, max_T, logit_bias=logit_bias, rep_offset=rep_offset,
                              rep_slots=rep_slots, S=S, local_start=self.start, local_count=self.count,
                              W1s=W1sh, W2s=W2sh, shared_gate_w=gate, **layer_options)

    def partial(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        """This rank's partial output (its slots' experts and its shared shard), bf16 [T, H]."""
        return self.layer.forward(x, stream)

    def forward(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        if self.peer is not None:
            if x.shape[0] == 0:
                return self.layer.out[:0]
            self.write_partial(x, stream)
            return self.peer.reduce(stream)
        return ep_reduce_output(self.partial(x, stream), self.group)

    def write_partial(self, x: torch.Tensor, stream=None) -> None:
        """Peer reduction, first half: this rank's partial into its slot, then its flag."""
        self.layer.forward(x, stream, out=self.peer.begin(x.shape[0]))
        self.peer.signal(stream)


# ----------------------------------------------------------------------------- all-to-all dispatch and combine

def a2a_count_splits(S: int, world: int):
    """Per-slot counts a rank sends to each rank: the counts of that rank's slot range,
    so the splits are the ranges' sizes (every rank receives S_local counts per source)."""
    return [ep_slot_range(S, world, d)[1] for d in range(world)]


def a2a_send_splits(offsets, S: int, world: int):
    """Rows a rank sends to each rank: its permuted rows of that rank's slot range, from
    the offsets [S + 1] of its own permutation (host values)."""
    res = []
    for d in range(world):
        lo, n = ep_slot_range(S, world, d)
        res.append(int(offsets[lo + n]) - int(offsets[lo]))
    return res


def a2a_recv_splits(recv_counts):
    """Rows a rank receives from each source rank: the row sums of recv_counts
    [N, S_local] (host values)."""
    return [int(sum(int(v) for v in row)) for row in recv_counts.tolist()]


def _words(t: torch.Tensor) -> torch.Tensor:
    """Rows of 2-byte elements travel as 32-bit words (element pairs; the rows' widths are
    even): a bit copy that NCCL and gloo both move."""
    return t.view(torch.int32) if t.element_size() == 2 else t


class DistExchange:
    """The all-to-all exchanges of EPAllToAllLayer over a torch.distributed process group
    (NCCL between GPUs, gloo between CPU processes)."""

    def __init__(self, group=None):
        self.group = group

    def all_to_all(self, out: torch.Tensor, inp: torch.Tensor, out_splits, in_splits) -> None:
        """out = the rows every rank sent to this one, in rank order; inp = the rows this
        rank sends, in_splits[d] of them (consecutive, in rank order) to rank d."""
        import torch.distributed as dist
        dist.all_to_all_single(_words(out), _words(inp), list(out_splits), list(in_splits), group=self.group)


class EPAllToAllLayer:
    """One rank of the all-to-all expert-parallel layer (TensorRT-LLM PR #10985, "MoE
    all-to-all paradigm", sequence diagram, all-to-all path: the tokens are dispatched to
    the ranks responsible for their experts, each rank computes the MoE on its local
    experts, and the results are gathered back to the tokens' ranks).

    Each rank holds its own batch of tokens (attention data parallelism), the whole router,
    the whole shared experts (with attention data parallelism nothing is split by tensor
    parallelism) and the experts of its contiguous slot range [r S / N, (r + 1) S / N).
    One forward, all on the current stream:
      1. dispatch: route the rank's tokens and group their pairs by slot over all S slots
         (moe_route, moe_permute); the rows bound for one rank are one contiguous run;
      2. the per-slot counts are exchanged (every rank receives, from every source, the
         counts of its own slots), copied to the host with the row offsets (the one host
         synchronisation: the row exchange needs its split sizes), then the rows;
      3. experts: the received rows are put in slot order (moe_a2a_regroup, which also
         records each row's arrival position), FC1+SwiGLU and FC2 of the rank's slots run
         over them in the same launches as the shared experts over the rank's own tokens
         (moe_grouped_fc1 / moe_grouped_fc2_scatter), FC2 storing each output row at its
         input's arrival position;
      4. combine: the reverse exchange returns every output row to its token's rank, into
         the place its input row left from, and moe_finalize forms the weighted sum of each
         token's k rows in fixed j order plus the shared output.
    Every kept pair's output row is the one the one-GPU layer computes for it (the GEMMs
    treat each row alone), so each rank's output equals the one-GPU layer's on its tokens.

    recv_cap: rows a rank can receive (default world * max_T * k, every pair of every rank);
    a forward that would receive more raises before the row exchange.  bf16 weights only."""

    def __init__(self, Wg, W1, W2, k, renorm, max_T, world: int, rank: int, logit_bias=None, rep_offset=None,
                 rep_slots=None, W1s=None, W2s=None, shared_gate_w=None, n_group: int = 1, topk_group: int = 1,
                 on_input: bool = False, recv_cap: Optional[int] = None, exchange=None):
        from . import moe_workspace_init, moe_workspace_size
        self.world, self.rank = int(world), int(rank)
        self.exchange = exchange if exchange is not None else DistExchange()
        self.Wg, self.bias = Wg, logit_bias
        self.E, self.H = Wg.shape
        self.S = int(W1.shape[0])
        self.I = int(W2.shape[2])
        self.k, self.renorm = int(k), bool(renorm)
        self.n_group, self.topk_group, self.on_input = int(n_group), int(topk_group), bool(on_input)
        self.rep_offset, self.rep_slots = rep_offset, rep_slots
        self.start, self.count = ep_slot_range(self.S, self.world, self.rank)
        self.W1 = W1[self.start:self.start + self.count].contiguous()
        self.W2 = W2[self.start:self.start + self.count].contiguous()
        self.W1s, self.W2s, self.gate = W1s, W2s, shared_gate_w
        self.I_sh = 0 if W2s is None else int(W2s.shape[1])
        self.max_T = int(max_T)
        self.recv_cap = int(recv_cap if recv_cap is not None else self.world * self.max_T * self.k)
        dev = Wg.device
        T, k, H, S, S_l = self.max_T, self.k, self.H, self.S, self.count
        i32 = dict(dtype=torch.int32, device=dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.topk_ids = torch.empty((T, k), **i32)
        self.topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.slot_ids = torch.empty((T, k), **i32)
        self.counts = torch.empty((S,), **i32)
        self.offsets = torch.empty((S + 1,), **i32)
        self.perm_src = torch.empty((T * k,), **i32)
        self.pair_row = torch.empty((T, k), **i32)
        self.send = torch.empty((T * k, H), **bf)     # rows out; then the returned output rows
        self.recv_counts = torch.empty((self.world, S_l), **i32)
        self.local_offsets = torch.empty((S_l + 1,), **i32)
        self.recv = torch.empty((self.recv_cap, H), **bf)   # arrival order: rows in, then outputs out
        self.x_loc = torch.empty((self.recv_cap, H), **bf)  # slot order
        self.row_map = torch.empty((self.recv_cap,), **i32)  # arrival row of each slot-order row
        self.h = torch.empty((self.recv_cap, self.I), **bf)
        self.h_sh = torch.empty((T, self.I_sh), **bf) if self.I_sh else None
        self.y_sh = torch.empty((T, H), **bf) if self.I_sh else None
        self.out = torch.empty((T, H), **bf)
        pin = dev.type == "cuda"
        self.offsets_host = torch.empty((S + 1,), dtype=torch.int32, pin_memory=pin)
        self.recv_counts_host = torch.empty((self.world, S_l), dtype=torch.int32, pin_memory=pin)
        nbytes = moe_workspace_size(T, H, self.I, self.E, S, k, self.I_sh)
        self.ws = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
        moe_workspace_init(self.ws)
        self.T = 0
        self.send_splits = self.recv_splits = None

    # ---- the four steps (forward runs them in order; a2a_forward_local interleaves the
    # ---- steps of several ranks held by one process)

    def dispatch(self, x: torch.Tensor) -> None:
        """Route x [T, H] and group its pairs by slot into self.send (rows) and self.counts."""
        from . import moe_permute, moe_route, moe_route_grouped
        T = x.shape[0]
        assert T <= self.max_T and x.shape[1] == self.H and x.dtype == torch.bfloat16
        self.T, self.x = T, x
        if T == 0:  # nothing to route: the rank still takes part in every exchange
            self.counts.zero_()
            self.offsets.zero_()
            return
        ids, w = self.topk_ids[:T], self.topk_w[:T]
        if self.n_group > 1:
            moe_route_grouped(x, self.Wg, self.bias, self.k, self.renorm, self.n_group, self.topk_group, ids, w,
                              self.ws)
        else:
            moe_route(x, self.Wg, self.bias, self.k, self.renorm, ids, w, self.ws)
        moe_permute(ids, w, self.E, self.rep_offset, self.rep_slots, self.S, 0, -1, MOE_NONLOCAL_SKIP, x,
                    self.slot_ids[:T], self.counts, self.offsets, self.perm_src[:T * self.k], self.pair_row[:T],
                    self.send[:T * self.k], self.ws, on_input=self.on_input)

    def plan(self) -> None:
        """After the count exchange: the split sizes of the row exchanges, on the host."""
        self.offsets_host.copy_(self.offsets, non_blocking=True)
        self.recv_counts_host.copy_(self.recv_counts, non_blocking=True)
        if self.offsets.is_cuda:
            torch.cuda.current_stream().synchronize()
        self.send_splits = a2a_send_splits(self.offsets_host, self.S, self.world)
        self.recv_splits = a2a_recv_splits(self.recv_counts_host)
        self.rows_out, self.rows_in = sum(self.send_splits), sum(self.recv_splits)
        if self.rows_in > self.recv_cap:
            raise RuntimeError(f"rank {self.rank} receives {self.rows_in} rows, more than recv_cap={self.recv_cap}")

    def experts(self) -> None:
        """The rank's slots over the received rows, and the shared experts over its own tokens."""
        from . import MOE_A2A_TO_GEMM, moe_a2a_regroup, moe_grouped_fc1, moe_grouped_fc2_scatter
        T = self.T
        moe_a2a_regroup(self.recv_counts, self.recv, self.x_loc, MOE_A2A_TO_GEMM, self.local_offsets, self.ws,
                        row_map=self.row_map)
        sh = self.I_sh > 0 and T > 0
        moe_grouped_fc1(self.x_loc, self.local_offsets, self.W1, self.x if sh else None, self.W1s if sh else None,
                        self.h, self.h_sh[:T] if sh else None, self.ws)
        # FC2 stores each output row at its input's arrival row (the received rows are
        # no longer needed): the outputs are in exchange order for the return trip
        moe_grouped_fc2_scatter(self.h, self.local_offsets, self.W2, self.h_sh[:T] if sh else None,
                                self.W2s if sh else None, self.row_map, self.recv, self.y_sh[:T] if sh else None,
                                self.ws)

    def combine(self) -> torch.Tensor:
        """After the reverse exchange: each token's weighted sum (plus the shared output)."""
        from . import moe_finalize
        T = self.T
        if T == 0:
            return self.out[:0]
        sh = self.I_sh > 0
        moe_finalize(self.send, self.pair_row[:T], None if self.on_input else self.topk_w[:T],
                     self.y_sh[:T] if sh else None, self.x if (sh and self.gate is not None) else None,
                     self.gate if sh else None, self.out[:T], self.ws)
        return self.out[:T]

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        """out [T, H] bf16 for this rank's tokens x [T, H]; every rank calls it (T may differ
        between ranks, and may be 0)."""
        ex = self.exchange
        self.dispatch(x)
        ex.all_to_all(self.recv_counts.view(-1), self.counts, [self.count] * self.world,
                      a2a_count_splits(self.S, self.world))
        self.plan()
        ex.all_to_all(self.recv[:self.rows_in], self.send[:self.rows_out], self.recv_splits, self.send_splits)
        self.experts()
        ex.all_to_all(self.send[:self.rows_out], self.recv[:self.rows_in], self.send_splits, self.recv_splits)
        return self.combine()


def a2a_forward_local(layers, xs, after_phase=None):
    """All ranks of an all-to-all layer held by one process on one device (a stand-in for N
    GPUs): the ranks' steps run one after another, and each exchange is a set of device
    copies between the ranks' buffers in the order an all-to-all delivers them.  Returns
    each rank's output.  after_phase(name), if given, is called after each phase (the
    ranks' dispatches, the count exchange, the plans, the row exchange, the experts, the
    reverse exchange, the combines), e.g. to separate their kernels in a timeline."""
    N = len(layers)
    assert all(L.world == N and L.rank == r for r, L in enumerate(layers)) and len(xs) == N
    note = after_phase or (lambda name: None)
    for L, x in zip(layers, xs):
        L.dispatch(x)
    note("dispatch")
    for d, Ld in enumerate(layers):
        for s, Ls in enumerate(layers):
            Ld.recv_counts[s].copy_(Ls.counts[Ld.start:Ld.start + Ld.count])
    note("count exchange")
    for L in layers:
        L.plan()
    note("plan")

    def blocks(splits):
        at = [0]
        for v in splits:
            at.append(at[-1] + v)
        return at

    send_at = [blocks(L.send_splits) for L in layers]
    recv_at = [blocks(L.recv_splits) for L in layers]
    for d, Ld in enumerate(layers):
        for s, Ls in enumerate(layers):
            n = Ls.send_splits[d]
            assert n == Ld.recv_splits[s]
            if n:
                Ld.recv[recv_at[d][s]:recv_at[d][s] + n].copy_(Ls.send[send_at[s][d]:send_at[s][d] + n])
    note("row exchange")
    for L in layers:
        L.experts()
    note("experts")
    for d, Ld in enumerate(layers):
        for s, Ls in enumerate(layers):
            n = Ls.send_splits[d]
            if n:
                Ls.send[send_at[s][d]:send_at[s][d] + n].copy_(Ld.recv[recv_at[d][s]:recv_at[d][s] + n])
    note("reverse exchange")
    outs = [L.combine() for L in layers]
    note("combine")
    return outs
