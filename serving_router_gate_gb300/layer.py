"""One MoE layer on one GPU: buffers for up to max_T tokens and the three
stream-ordered library calls (moe_route -> moe_permute -> moe_forward).

Weights are handed over per expert slot, as the fused op of the TensorRT-LLM
redundant-expert refactor (PR #4495) computes on slots: W1 [S_local, 2I, H]
(gate rows then up rows), W2 [S_local, H, I].  With a local expert range only
the local slots' weights are passed (the vLLM EP weight loader keeps only the
local experts).  All tensors live on the current CUDA device; nothing is
allocated per call and no call synchronises the host.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (MOE_NONLOCAL_SKIP, moe_forward, moe_forward_fp8, moe_forward_nvfp4, moe_forward_w8a8, moe_permute,
               moe_quantize_fp8_rows, moe_quantize_nvfp4_rows, moe_route, moe_route_grouped, moe_workspace_init,
               moe_workspace_size, nvfp4_sf_row_bytes)


class MoELayer:
    def __init__(self, Wg: torch.Tensor, W1: torch.Tensor, W2: torch.Tensor, k: int, renorm: bool,
                 max_T: int, logit_bias: Optional[torch.Tensor] = None,
                 rep_offset: Optional[torch.Tensor] = None, rep_slots: Optional[torch.Tensor] = None,
                 S: Optional[int] = None, local_start: int = 0, local_count: int = -1,
                 nonlocal_mode: int = MOE_NONLOCAL_SKIP, W1s: Optional[torch.Tensor] = None,
                 W2s: Optional[torch.Tensor] = None, shared_gate_w: Optional[torch.Tensor] = None,
                 on_input: bool = False, n_group: int = 1, topk_group: int = 1, fp8: bool = False,
                 act8: bool = False, fp4: bool = False):
        self.Wg, self.W1, self.W2 = Wg, W1, W2
        # routing applied on the input: rows scaled by the weights, outputs summed unweighted
        self.on_input = bool(on_input)
        # group-limited top-k (n_group <= 1: plain top-k)
        self.n_group, self.topk_group = int(n_group), int(topk_group)
        self.E, self.H = Wg.shape
        self.I = W2.shape[2]
        self.k, self.renorm = int(k), bool(renorm)
        self.bias = logit_bias
        self.rep_offset, self.rep_slots = rep_offset, rep_slots
        self.S = int(S if S is not None else (self.E if rep_offset is None else rep_slots.shape[0]))
        self.local_start, self.local_count, self.mode = int(local_start), int(local_count), int(nonlocal_mode)
        self.S_local = self.local_count if self.local_count >= 0 else self.S
        assert W1.shape == (self.S_local, 2 * self.I, self.H), W1.shape
        self.W1s, self.W2s, self.gate = W1s, W2s, shared_gate_w
        self.I_sh = 0 if W2s is None else W2s.shape[1]
        self.max_T = int(max_T)
        dev = Wg.device
        T, k, H = self.max_T, self.k, self.H
        i32 = dict(dtype=torch.int32, device=dev)
        self.topk_ids = torch.empty((T, k), **i32)
        self.topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.slot_ids = torch.empty((T, k), **i32)
        self.counts = torch.empty((self.S_local,), **i32)
        self.offsets = torch.empty((self.S_local + 1,), **i32)
        self.perm_src = torch.empty((T * k,), **i32)
        self.pair_row = torch.empty((T, k), **i32)
        self.x_perm = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        nbytes = moe_workspace_size(T, H, self.I, self.E, max(self.S, self.S_local), k, self.I_sh)
        self.ws = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
        moe_workspace_init(self.ws)
        # E4M3 expert weights with one fp32 scale per row, quantised once here
        self.fp8 = bool(fp8)
        # E4M3 activations as well (per row, power-of-two scales, inside moe_forward_w8a8)
        self.act8 = bool(act8)
        if self.act8 and not self.fp8:
            raise ValueError("E4M3 activations need E4M3 weights (fp8=True)")
        self.W1q = self.s1 = self.W2q = self.s2 = self.W1sq = self.s1s = self.W2sq = self.s2s = None
        if self.fp8:
            def quant(w):
                q = torch.empty(w.shape, dtype=torch.uint8, device=dev)
                sc = torch.empty(w.shape[:-1], dtype=torch.float32, device=dev)
                moe_quantize_fp8_rows(w, q, sc)
                return q, sc
            self.W1q, self.s1 = quant(W1)
            self.W2q, self.s2 = quant(W2)
            if W1s is not None:
                self.W1sq, self.s1s = quant(W1s)
                self.W2sq, self.s2s = quant(W2s)
        # NVFP4 experts (E2M1 codes, E4M3 block scales, fp32 row scales), quantised once here;
        # the activations are quantised inside moe_forward_nvfp4
        self.fp4 = bool(fp4)
        if self.fp4 and self.fp8:
            raise ValueError("one weight format at a time")
        self.W1f = self.W2f = self.W1sf = self.W2sf = None
        if self.fp4:
            def quant4(w):
                K = w.shape[-1]
                q = torch.empty(w.shape[:-1] + (K // 2,), dtype=torch.uint8, device=dev)
                sb = torch.empty(w.shape[:-1] + (nvfp4_sf_row_bytes(K),), dtype=torch.uint8, device=dev)
                sc = torch.empty(w.shape[:-1], dtype=torch.float32, device=dev)
                moe_quantize_nvfp4_rows(w, q, sb, sc, pow2=False)
                return q, sb, sc
            self.W1f = quant4(W1)
            self.W2f = quant4(W2)
            if W1s is not None:
                self.W1sf = quant4(W1s)
                self.W2sf = quant4(W2s)

    def views(self, T: int) -> dict:
        k = self.k
        return dict(topk_ids=self.topk_ids[:T], topk_w=self.topk_w[:T], slot_ids=self.slot_ids[:T],
                    counts=self.counts, offsets=self.offsets, perm_src=self.perm_src[:T * k],
                    pair_row=self.pair_row[:T], x_perm=self.x_perm[:T * k], out=self.out[:T])

    def route(self, x: torch.Tensor, stream=None) -> dict:
        v = self.views(x.shape[0])
        if self.n_group > 1:
            moe_route_grouped(x, self.Wg, self.bias, self.k, self.renorm, self.n_group, self.topk_group,
                              v["topk_ids"], v["topk_w"], self.ws, stream)
        else:
            moe_route(x, self.Wg, self.bias, self.k, self.renorm, v["topk_ids"], v["topk_w"], self.ws, stream)
        return v

    def rows_from_tokens(self, T: int) -> bool:
        """Whether the expert input rows are read from the token rows through pair_row, with
        the weights applied at the output: quantised activations (NVFP4, or E4M3 with E4M3
        weights) are made once per token row and placed at its pairs' rows, so moe_permute
        copies no rows into x_perm (at every batch size this saves more in the permute than
        the token-row quantiser gives up in parallelism)."""
        if self.on_input:
            return False
        return self.fp4 or self.act8

    def permute(self, x: torch.Tensor, stream=None) -> dict:
        v = self.views(x.shape[0])
        xp = None if self.rows_from_tokens(x.shape[0]) else v["x_perm"]
        moe_permute(v["topk_ids"], v["topk_w"], self.E, self.rep_offset, self.rep_slots, self.S,
                    self.local_start, self.local_count, self.mode, x, v["slot_ids"], v["counts"], v["offsets"],
                    v["perm_src"], v["pair_row"], xp, self.ws, stream, on_input=self.on_input)
        return v

    def expert_forward(self, x: torch.Tensor, stream=None, out: Optional[torch.Tensor] = None) -> dict:
        v = self.views(x.shape[0])
        if out is not None:
            v["out"] = out
        w = None if self.on_input else v["topk_w"]
        xs = x if (self.I_sh > 0) else None
        if self.fp4:
            (q1, f1, s1), (q2, f2, s2) = self.W1f, self.W2f
            q1s = f1s = s1s = q2s = f2s = s2s = None
            if self.W1sf is not None:
                (q1s, f1s, s1s), (q2s, f2s, s2s) = self.W1sf, self.W2sf
            if self.rows_from_tokens(x.shape[0]):
                moe_forward_nvfp4(None, v["offsets"], q1, f1, s1, q2, f2, s2, v["pair_row"], w, x, q1s, f1s, s1s,
                                  q2s, f2s, s2s, self.gate, v["out"], self.ws, stream)
            else:
                moe_forward_nvfp4(v["x_perm"], v["offsets"], q1, f1, s1, q2, f2, s2, v["pair_row"], w, xs, q1s, f1s,
                                  s1s, q2s, f2s, s2s, self.gate, v["out"], self.ws, stream)
        elif self.fp8:
            fwd = moe_forward_w8a8 if self.act8 else moe_forward_fp8
            # E4M3 activations: x also lets large batches quantise each token row once
            xa = x if self.act8 else xs
            xp = None if self.rows_from_tokens(x.shape[0]) else v["x_perm"]
            fwd(xp, v["offsets"], self.W1q, self.s1, self.W2q, self.s2, v["pair_row"], w, xa,
                self.W1sq, self.s1s, self.W2sq, self.s2s, self.gate, v["out"], self.ws, stream)
        else:
            moe_forward(v["x_perm"], v["offsets"], self.W1, self.W2, v["pair_row"], w, xs, self.W1s, self.W2s,
                        self.gate, v["out"], self.ws, stream)
        return v

    def capture(self, x: torch.Tensor, pre=None, post=None, out: Optional[torch.Tensor] = None) -> "torch.cuda.CUDAGraph":
        """Record one forward (optionally wrapped by pre()/post() stream work, e.g.
        host<->device copies) into a CUDA graph; replaying it re-runs the same
        kernels with the same pointers.  Every library call is capturable: none
        synchronises or allocates, and tensor maps are built on the host when the
        call is recorded.  Run one forward outside capture first, so per-device
        one-time set-up happens before recording."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            if pre:
                pre()
            self.forward(x, out=out)
            if post:
                post()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            if pre:
                pre()
            self.forward(x, out=out)
            if post:
                post()
        return g

    def forward(self, x: torch.Tensor, stream=None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """out [T, H] bf16 for x [T, H] bf16, T <= max_T: the given device tensor, or a view
        of the layer's own output buffer."""
        assert x.shape[0] <= self.max_T and x.shape[1] == self.H
        if out is not None:
            assert out.shape == x.shape and out.dtype == torch.bfloat16 and out.device == x.device
        if x.shape[0] == 0:
            return self.out[:0] if out is None else out
        self.route(x, stream)
        self.permute(x, stream)
        return self.expert_forward(x, stream, out)["out"]


class HostPipeline:
    """Forward a sequence of host batches through one layer with the host<->device copies
    overlapping the compute: while batch i runs on the compute stream, batch i+1's input is
    copied to the device on one copy stream and batch i-1's output to the host on another.
    Two device input buffers and two device output buffers alternate between batches;
    events order every buffer's copies against the forwards that use it (an input buffer
    is refilled only after the forward two batches back has read it, an output buffer is
    rewritten only after its previous copy to the host).  Each forward is a replay of a
    CUDA graph captured on its buffer pair.  Host tensors must be pinned for the copies to
    run asynchronously.  Nothing is allocated per batch and the host never waits: read the
    outputs after the device (or the output stream) is synchronised."""

    def __init__(self, layer: MoELayer, example: torch.Tensor):
        """example: one batch [T, H] bf16 (host or device); it fixes T and is the input of
        the forwards run while the two graphs are captured."""
        T = example.shape[0]
        assert 0 < T <= layer.max_T and example.shape[1] == layer.H and example.dtype == torch.bfloat16
        dev = layer.Wg.device
        self.layer, self.T = layer, int(T)
        shape = (self.T, layer.H)
        self.x_dev = [example.to(dev).clone() for _ in range(2)]
        self.out_dev = [torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.s_in, self.s_cmp, self.s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        self.ev_in = [torch.cuda.Event() for _ in range(2)]   # input buffer b filled
        self.ev_fwd = [torch.cuda.Event() for _ in range(2)]  # forward on buffers b done
        self.ev_out = [torch.cuda.Event() for _ in range(2)]  # output buffer b copied to the host
        self.graphs = [layer.capture(self.x_dev[b], out=self.out_dev[b]) for b in range(2)]
        self.n = 0  # batches issued so far (the buffer parity carries over between calls)

    def run(self, xs_host, outs_host, before_forward=None):
        """Issue the batches: xs_host[i] ([T, H] bf16, pinned) in, outs_host[i] out.
        before_forward(i), if given, is called on the compute stream right before
        forward i (e.g. to flush L2 for a measurement)."""
        assert len(xs_host) == len(outs_host)
        for i, (xh, oh) in enumerate(zip(xs_host, outs_host)):
            assert xh.shape == (self.T, self.layer.H) and oh.shape == (self.T, self.layer.H)
            b = self.n & 1
            self.n += 1
            self.s_in.wait_event(self.ev_fwd[b])
            with torch.cuda.stream(self.s_in):
                self.x_dev[b].copy_(xh, non_blocking=True)
            self.ev_in[b].record(self.s_in)
            self.s_cmp.wait_event(self.ev_in[b])
            self.s_cmp.wait_event(self.ev_out[b])
            with torch.cuda.stream(self.s_cmp):
                if before_forward is not None:
                    before_forward(i)
                self.graphs[b].replay()
            self.ev_fwd[b].record(self.s_cmp)
            self.s_out.wait_event(self.ev_fwd[b])
            with torch.cuda.stream(self.s_out):
                oh.copy_(self.out_dev[b], non_blocking=True)
            self.ev_out[b].record(self.s_out)


def layer_from_inputs(inp: dict, device="cuda", max_T: Optional[int] = None, local_start: int = 0,
                      local_count: int = -1, nonlocal_mode: int = MOE_NONLOCAL_SKIP,
                      on_input: Optional[bool] = None) -> MoELayer:
    """A MoELayer over the tensors of moe_inputs.make_inputs() (moved to `device`); the
    routing variant (groups, routing on the input) follows the workload unless given."""
    from moe_inputs import shared_concat
    cfg = inp["cfg"]
    if on_input is None:
        on_input = cfg.on_input

    def d(t):
        return None if t is None else t.to(device).contiguous()

    W1, W2 = inp["W1"], inp["W2"]
    if local_count >= 0:
        W1 = W1[local_start:local_start + local_count]
        W2 = W2[local_start:local_start + local_count]
    W1s = W2s = None
    if inp["W1s"] is not None:
        W1s, W2s = shared_concat(inp["W1s"], inp["W2s"])
    return MoELayer(d(inp["Wg"]), d(W1), d(W2), cfg.k, cfg.renorm, max_T or cfg.T, logit_bias=d(inp["bias"]),
                    rep_offset=d(inp["rep_offset"]), rep_slots=d(inp["rep_slots"]), S=cfg.slots,
                    local_start=local_start, local_count=local_count, nonlocal_mode=nonlocal_mode,
                    W1s=d(W1s), W2s=d(W2s), shared_gate_w=d(inp["w_s"]), on_input=on_input,
                    n_group=cfg.n_group, topk_group=cfg.topk_group, fp8=cfg.fp8, act8=cfg.act8, fp4=cfg.fp4)
