"""Seeded synthetic inputs for the MoE layer forward.

This module only draws random tensors and lays them out; it holds none of the
layer's arithmetic (no routing, masking, permutation, MLP or combine), so the
CUDA path and the CPU oracle can both be fed from it without sharing code.

Workloads (shapes and value distributions of the layer configurations the
library is measured and checked on):

  tiny                      T=64, H=256, I=512, E=8, k=2, renorm on
  qwen2_moe_like_prefill    T=4096, H=2048, I=1408, E=60, k=4, renorm off,
                            1 shared expert (I=5632) scaled by sigmoid(x . w_s)
  dsv2_lite_like_decode_tN  T=N in {1, 8, 32, 128}, H=2048, I=1408, E=64, k=6,
                            renorm off, 2 shared experts of I=2816 (unscaled)
  large_expert_prefill      T=8192, H=7168, I=2048, E=256, k=8, renorm on,
                            expert weights N(0, 0.01); optional local range
  redundant_slots_prefill   T=16384, H=7168, I=2048, E=256 experts in S=288
                            slots (32 hottest experts get 2 slots), Zipf(1.1)
                            logit bias, k=8, renorm on, expert weights N(0, 0.01)

Value distributions: x ~ N(0, 1) rounded to bf16; gate weights Wg ~ N(0, 0.02)
in fp32; expert and shared-expert weights ~ N(0, w_std) rounded to bf16; the
shared gate vector w_s ~ N(0, 0.02) in bf16.

Seeding: tensor number i of a workload draws from its own torch.Generator
seeded with seed * 1000 + i, in the order x (0), Wg (1), W1 (2), W2 (3), W1s
(4), W2s (5), w_s (6), expert hotness order (7), slot shuffle (8); the own
batch of expert-parallel rank r (all-to-all layer) is tensor 100 + r.  Tensors
drawn on a CUDA device use a CUDA generator and so differ from CPU draws with
the same seed; within one run both sides of every check read the same bytes.

Redundant slots: a seeded permutation ranks the experts by hotness (rank 1 is
the hottest); the logit bias of expert e is -s * ln(rank_e) (the log of Zipf(s)
probabilities; the normaliser cancels in a softmax).  The n_hot hottest experts
get two slots, the rest one; the slot ids of all (expert, replica) pairs are a
seeded shuffle of 0..S-1.  Replica slots hold copies of the expert's weights.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    renorm: bool
    S: Optional[int] = None          # expert slots (None: S = E, identity map)
    n_hot: int = 0                   # experts that get a second slot
    zipf_s: float = 0.0              # Zipf exponent of the logit bias (0: no bias)
    n_shared: int = 0                # shared experts
    I_shared: int = 0                # intermediate size of each shared expert
    shared_gate: bool = False        # scale the shared output by sigmoid(x . w_s)
    n_group: int = 1                 # group-limited top-k: expert groups (1: plain top-k)
    topk_group: int = 1              # groups kept per token
    on_input: bool = False           # routing weight applied to the expert input, outputs summed unweighted
    fp8: bool = False                # E4M3 expert weights with one fp32 scale per row
    act8: bool = False               # and E4M3 activations, one power-of-two scale per row
    fp4: bool = False                # NVFP4 expert weights and activations (E2M1, E4M3 block scales)
    w_std: float = 0.02              # expert weight std
    gate_std: float = 0.02           # router weight std
    seed: int = 0

    @property
    def slots(self) -> int:
        return self.E if self.S is None else self.S

    def with_(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": MoEConfig("tiny", T=64, H=256, I=512, E=8, k=2, renorm=True),
    "qwen2_moe_like_prefill": MoEConfig("qwen2_moe_like_prefill", T=4096, H=2048, I=1408, E=60, k=4,
                                        renorm=False, n_shared=1, I_shared=5632, shared_gate=True),
    "large_expert_prefill": MoEConfig("large_expert_prefill", T=8192, H=7168, I=2048, E=256, k=8,
                                      renorm=True, w_std=0.01),
    "redundant_slots_prefill": MoEConfig("redundant_slots_prefill", T=16384, H=7168, I=2048, E=256,
                                         k=8, renorm=True, S=288, n_hot=32, zipf_s=1.1, w_std=0.01),
}
# a cut-down redundant-slot layer (same H and I, 16 slots of about 512 rows, a few GB on the
# device) on which the FC1 DRAM traffic of the full workload is captured and scaled per slot
CONFIGS["redundant_slots_cut16"] = MoEConfig("redundant_slots_cut16", T=1024, H=7168, I=2048, E=16, k=8,
                                             renorm=True, w_std=0.01)
# the router of the large-expert and redundant-slot layers (H = 7168, E = 256, Zipf bias) on
# 8192 tokens with small experts: about 2 GB on the device, for router captures
CONFIGS["router_h7168_e256_cut"] = MoEConfig("router_h7168_e256_cut", T=8192, H=7168, I=64, E=256, k=8,
                                             renorm=True, zipf_s=1.1, w_std=0.01)
# the router variants of the next steps, on the Qwen2-like and DeepSeek-V2-Lite-like shapes:
# group-limited top-k (DeepSeek-V2-style: 8 groups, 3 kept, k = 6 of 64 experts) and the
# routing weight applied on the expert input
CONFIGS["grouped_topk_prefill"] = MoEConfig("grouped_topk_prefill", T=4096, H=2048, I=1408, E=64, k=6,
                                            renorm=False, n_shared=2, I_shared=2816, n_group=8, topk_group=3)
CONFIGS["routing_on_input_prefill"] = CONFIGS["qwen2_moe_like_prefill"].with_(name="routing_on_input_prefill",
                                                                              on_input=True)
for _t in (1, 8, 32, 128):
    CONFIGS[f"dsv2_lite_like_decode_t{_t}"] = MoEConfig(
        f"dsv2_lite_like_decode_t{_t}", T=_t, H=2048, I=1408, E=64, k=6, renorm=False,
        n_shared=2, I_shared=2816)
# E4M3 expert weights (one fp32 scale per row) on the decode and Qwen2-like shapes
for _name in ["dsv2_lite_like_decode_t1", "dsv2_lite_like_decode_t8", "dsv2_lite_like_decode_t32",
              "dsv2_lite_like_decode_t128", "qwen2_moe_like_prefill"]:
    CONFIGS[_name + "_fp8"] = CONFIGS[_name].with_(name=_name + "_fp8", fp8=True)
    # E4M3 weights and activations (tcgen05 kind::f8f6f4)
    CONFIGS[_name + "_w8a8"] = CONFIGS[_name].with_(name=_name + "_w8a8", fp8=True, act8=True)
    # NVFP4 weights and activations (tcgen05 kind::mxf4nvf4)
    CONFIGS[_name + "_nvfp4"] = CONFIGS[_name].with_(name=_name + "_nvfp4", fp4=True)


def _gen(device, seed: int, idx: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + idx)
    return g


def _normal(shape, std, gen, device, dtype) -> torch.Tensor:
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _expert_stack(n: int, rows: int, cols: int, std: float, gen, device) -> torch.Tensor:
    """n matrices [rows, cols] in bf16, drawn one after another from one generator."""
    out = torch.empty((n, rows, cols), dtype=torch.bfloat16, device=device)
    for e in range(n):
        out[e] = _normal((rows, cols), std, gen, device, torch.bfloat16)
    return out


def slot_table(cfg: MoEConfig):
    """Hotness order, logit bias and the expert -> slot table of a workload.

    Returns dict(rank [E] (1 = hottest), bias [E] fp32 or None, rep_offset [E+1],
    rep_slots [S], expert_of_slot [S]) as CPU int32/float32 tensors; rep_offset /
    rep_slots are None for the identity map (S == E and no replicas).
    """
    E, S = cfg.E, cfg.slots
    g7 = _gen("cpu", cfg.seed, 7)
    order = torch.randperm(E, generator=g7)          # order[0] is the hottest expert
    rank = torch.empty(E, dtype=torch.int64)
    rank[order] = torch.arange(1, E + 1)
    bias = None
    if cfg.zipf_s:
        bias = (-cfg.zipf_s * torch.log(rank.to(torch.float64))).to(torch.float32)
    if S == E and cfg.n_hot == 0:
        return dict(rank=rank, bias=bias, rep_offset=None, rep_slots=None,
                    expert_of_slot=torch.arange(E, dtype=torch.int32))
    assert S == E + cfg.n_hot, "each hot expert gets exactly one extra slot"
    rep_count = torch.ones(E, dtype=torch.int64)
    rep_count[rank <= cfg.n_hot] = 2
    rep_offset = torch.zeros(E + 1, dtype=torch.int64)
    rep_offset[1:] = torch.cumsum(rep_count, 0)
    g8 = _gen("cpu", cfg.seed, 8)
    slot_of_pair = torch.randperm(S, generator=g8)   # (expert, replica) pair i -> slot
    rep_slots = slot_of_pair.to(torch.int32)
    expert_of_slot = torch.empty(S, dtype=torch.int32)
    for e in range(E):
        for r in range(int(rep_count[e])):
            expert_of_slot[int(slot_of_pair[int(rep_offset[e]) + r])] = e
    return dict(rank=rank, bias=bias, rep_offset=rep_offset.to(torch.int32), rep_slots=rep_slots,
                expert_of_slot=expert_of_slot)


def make_inputs(cfg: MoEConfig, device="cpu", weights_device=None) -> dict:
    """All inputs of one workload, seeded.

    x [T, H] bf16; Wg [E, H] fp32; bias [E] fp32 or None; W1 [S, 2I, H] bf16
    (gate rows then up rows, indexed by slot); W2 [S, H, I] bf16; W1s
    [n_shared, 2*I_sh, H] / W2s [n_shared, H, I_sh] bf16 or None; w_s [H] bf16 or
    None; rep_offset [E+1] / rep_slots [S] int32 or None; expert_of_slot [S].
    """
    wdev = device if weights_device is None else weights_device
    T, H, I, E = cfg.T, cfg.H, cfg.I, cfg.E
    tab = slot_table(cfg)
    x = _normal((T, H), 1.0, _gen(device, cfg.seed, 0), device, torch.bfloat16)
    Wg = _normal((E, H), cfg.gate_std, _gen(device, cfg.seed, 1), device, torch.float32)
    W1e = _expert_stack(E, 2 * I, H, cfg.w_std, _gen(wdev, cfg.seed, 2), wdev)
    W2e = _expert_stack(E, H, I, cfg.w_std, _gen(wdev, cfg.seed, 3), wdev)
    if tab["rep_offset"] is None:
        W1, W2 = W1e, W2e
    else:
        idx = tab["expert_of_slot"].to(torch.int64).to(wdev)
        W1 = W1e.index_select(0, idx)
        W2 = W2e.index_select(0, idx)
        del W1e, W2e
    W1s = W2s = w_s = None
    if cfg.n_shared:
        W1s = _expert_stack(cfg.n_shared, 2 * cfg.I_shared, H, cfg.w_std, _gen(wdev, cfg.seed, 4), wdev)
        W2s = _expert_stack(cfg.n_shared, H, cfg.I_shared, cfg.w_std, _gen(wdev, cfg.seed, 5), wdev)
        if cfg.shared_gate:
            w_s = _normal((H,), 0.02, _gen(device, cfg.seed, 6), device, torch.bfloat16)
    bias = tab["bias"]
    if bias is not None:
        bias = bias.to(device)

    def _dev(t):
        return None if t is None else t.to(device)

    return dict(cfg=cfg, x=x, Wg=Wg, bias=bias, W1=W1, W2=W2, W1s=W1s, W2s=W2s, w_s=w_s,
                rep_offset=_dev(tab["rep_offset"]), rep_slots=_dev(tab["rep_slots"]),
                expert_of_slot=tab["expert_of_slot"], rank=tab["rank"])


def rank_tokens(cfg: MoEConfig, rank: int, T: int, device="cpu") -> torch.Tensor:
    """Token rows [T, H] bf16 of one rank's own batch (expert parallelism with attention
    data parallelism: every rank holds different tokens), N(0, 1) like x, drawn from the
    generator seeded with seed * 1000 + 100 + rank."""
    return _normal((T, cfg.H), 1.0, _gen(device, cfg.seed, 100 + rank), device, torch.bfloat16)


def shared_concat(W1s: torch.Tensor, W2s: torch.Tensor):
    """Lay n shared experts out as one gated MLP of intermediate n*I_sh.

    W1s [n, 2*I_sh, H] -> [2*n*I_sh, H] as (gate_0..gate_{n-1}; up_0..up_{n-1});
    W2s [n, H, I_sh] -> [H, n*I_sh] as [W2_0 | ... | W2_{n-1}].  A pure layout
    change: the sum of the n experts' outputs equals this MLP's output.
    """
    n, two_i, H = W1s.shape
    I_sh = two_i // 2
    gate = W1s[:, :I_sh, :].reshape(n * I_sh, H)
    up = W1s[:, I_sh:, :].reshape(n * I_sh, H)
    W1c = torch.cat([gate, up], 0).contiguous()
    W2c = W2s.permute(1, 0, 2).reshape(H, n * I_sh).contiguous()
    return W1c, W2c


def zipf_bias_for(rank: torch.Tensor, s: float) -> torch.Tensor:
    """Logit bias -s * ln(rank) for a given hotness ranking (1 = hottest)."""
    return (-s * torch.log(rank.to(torch.float64))).to(torch.float32)


def describe(cfg: MoEConfig) -> str:
    parts = [f"T={cfg.T}", f"H={cfg.H}", f"I={cfg.I}", f"E={cfg.E}", f"S={cfg.slots}", f"k={cfg.k}",
             f"renorm={'on' if cfg.renorm else 'off'}"]
    if cfg.n_shared:
        parts.append(f"shared={cfg.n_shared}x{cfg.I_shared}" + ("+sigmoid gate" if cfg.shared_gate else ""))
    if cfg.zipf_s:
        parts.append(f"zipf={cfg.zipf_s}")
    if cfg.n_group > 1:
        parts.append(f"grouped top-k {cfg.topk_group} of {cfg.n_group} groups")
    if cfg.on_input:
        parts.append("routing on input")
    if cfg.fp8:
        parts.append("E4M3 weights, row scales" + (" + E4M3 activations, power-of-two row scales"
                                                   if cfg.act8 else ""))
    if cfg.fp4:
        parts.append("NVFP4 weights and activations (E2M1, E4M3 scale per 16 elements, fp32 row scale)")
    return ", ".join(parts)


def flops_per_token(cfg: MoEConfig) -> dict:
    """Algorithmic flop counts per token (multiply-add = 2 flops)."""
    routed = 6.0 * cfg.k * cfg.H * cfg.I
    shared = 6.0 * cfg.n_shared * cfg.H * cfg.I_shared
    gate = 2.0 * cfg.H * cfg.E
    return dict(routed=routed, shared=shared, gate=gate, total=routed + shared + gate)

