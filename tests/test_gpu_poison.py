"""Reads of memory no kernel wrote, exposed by poisoning (a stand-in for a race
and initialisation checker).

Every buffer of a layer that a forward writes before it reads -- routing
outputs, permutation outputs, x_perm, out, and the workspace body behind its
header (router partials, permutation scratch, h, h_shared, y, y_shared, the
split shared FC2's fp32 partials, the E4M3 rows and scales) -- is filled with
all-ones bytes (a NaN in bf16 and fp32, -1 in int32) before a forward, and the
forward must reproduce bitwise what it gives on zero-filled buffers.  A kernel
that read a row, a partial or a scale nobody wrote would carry the NaN (or a
-1 index) into its result.
"""
import pytest
import torch

import moe_inputs as mi
import serving_router_gate_gb300 as moe
from serving_router_gate_gb300.layer import layer_from_inputs

pytestmark = pytest.mark.gpu

_BUFS = ("topk_ids", "topk_w", "slot_ids", "counts", "offsets", "perm_src", "pair_row", "x_perm", "out")


def _fill(layer, byte):
    for name in _BUFS:
        getattr(layer, name).view(torch.uint8).fill_(byte)
    layer.ws[moe.MOE_WS_HEADER_BYTES:].fill_(byte)  # the header (status word, counters) stays


def _forward(layer, x, byte):
    _fill(layer, byte)
    torch.cuda.synchronize()
    layer.forward(x)
    torch.cuda.synchronize()
    T = x.shape[0]
    got = {n: getattr(layer, n)[:T].clone() for n in ("topk_ids", "topk_w", "slot_ids", "pair_row", "out")}
    got["counts"] = layer.counts.clone()
    got["offsets"] = layer.offsets.clone()
    rows = int(layer.offsets[-1])
    got["perm_src"] = layer.perm_src[:rows].clone()
    if not layer.rows_from_tokens(T):  # else the experts read the token rows and x_perm stays unwritten
        got["x_perm"] = layer.x_perm[:rows].clone()
    return got


CASES = {
    # bf16 experts, a gated shared expert, several tiles per slot
    "bf16": mi.MoEConfig("poison_bf16", T=1000, H=512, I=384, E=12, k=3, renorm=True, n_shared=1,
                         I_shared=256, shared_gate=True),
    # a small batch: the shared FC2 runs split over K into fp32 partials summed by the combine
    "split_shared_fc2": mi.MoEConfig("poison_split", T=40, H=512, I=256, E=8, k=2, renorm=False, n_shared=2,
                                     I_shared=512),
    # E4M3 weights and activations: quantised rows and scales in the workspace
    "w8a8": mi.MoEConfig("poison_w8a8", T=1000, H=512, I=384, E=12, k=3, renorm=True, n_shared=1,
                         I_shared=256, shared_gate=True, fp8=True, act8=True),
    "w8a8_small": mi.MoEConfig("poison_w8a8_small", T=40, H=512, I=256, E=8, k=2, renorm=False, n_shared=2,
                               I_shared=512, fp8=True, act8=True),
    # E4M3 weights, bf16 activations
    "w8": mi.MoEConfig("poison_w8", T=300, H=256, I=256, E=6, k=2, renorm=True, fp8=True),
    # a local expert range (fewer rows than the buffers hold)
    "local_range": mi.MoEConfig("poison_local", T=600, H=256, I=256, E=16, k=4, renorm=True),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_poisoned_buffers_give_the_clean_result(case):
    cfg = CASES[case]
    inp = mi.make_inputs(cfg)
    kw = dict(local_start=4, local_count=8) if case == "local_range" else {}
    layer = layer_from_inputs(inp, "cuda", **kw)
    x = inp["x"].cuda()
    clean = _forward(layer, x, 0x00)
    poisoned = _forward(layer, x, 0xFF)
    for name, a in clean.items():
        b = poisoned[name]
        assert a.shape == b.shape, name
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"{case}: {name} depends on unwritten memory"
    assert torch.isfinite(poisoned["out"].float()).all()
    assert moe.moe_get_device_status(layer.ws) == 0
