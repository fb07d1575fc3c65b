"""moe_route_noalloc -- the router for callers that cannot allocate device
memory (a plugin handed only its input/output buffers, a runtime whose memory
belongs to a pool the library cannot reach, a service that forbids allocation
once running).  It must give what moe_route gives: the same ids bit for bit
and the same weights within the router's certified fp32 bound, on two calls
in a row (the second call sees the first call's leftovers in the shared
scratch array), and refuse sizes beyond its fixed scratch.

This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import serving_router_gate_gb300 as moe

from parity_util import router_bound

pytestmark = pytest.mark.gpu


def _route_both(cfg, bias=None):
    inp = mi.make_inputs(cfg)
    x, Wg = inp["x"].cuda(), inp["Wg"].cuda()
    b = None if bias is None else bias.cuda()
    T, k = cfg.T, cfg.k
    ids_a = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w_a = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.moe_workspace_size(T, cfg.H, cfg.I, cfg.E, cfg.E, k, 0), dtype=torch.uint8,
                     device="cuda")
    moe.moe_workspace_init(ws)
    moe.moe_route(x, Wg, b, k, cfg.renorm, ids_a, w_a, ws)
    ids_b = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w_b = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_route_noalloc(x, Wg, b, k, cfg.renorm, ids_b, w_b)
    torch.cuda.synchronize()
    assert torch.equal(ids_a, ids_b)
    B = router_bound(inp["x"], inp["Wg"], bias, cfg.H)
    rel = np.expm1(4.0 * B)[:, None] + 128 * 2.0 ** -24  # both sides within the bound of the exact value
    wa, wb = w_a.cpu().double().numpy(), w_b.cpu().double().numpy()
    assert np.all(np.abs(wa - wb) <= rel * np.abs(wa) + 1e-7)


def test_noalloc_route_matches_route_on_two_calls_in_a_row():
    # first call: a larger batch that fills more of the scratch array
    cfg1 = mi.MoEConfig("na1", T=3000, H=2048, I=64, E=60, k=4, renorm=False)
    _route_both(cfg1, bias=torch.linspace(-1.0, 1.0, 60))
    # second call: different sizes over the first call's leftovers
    cfg2 = mi.MoEConfig("na2", T=64, H=256, I=64, E=8, k=2, renorm=True)
    _route_both(cfg2)


def _router_plan_splits(T, H, E, sms):
    """The number of K ranges moe_route's split plan picks (its cost model: CTAs of
    128 tokens x 64 experts run in waves of two per SM; a CTA costs its range plus
    about three 32-wide chunks)."""
    tiles = -(-T // 128) * -(-E // 64)
    slots = max(1, min(2 * sms, 2048))
    best, best_ns = None, 1
    for kc in range(32, H + 1, 32):
        ns = -(-H // kc)
        if ns > 32 or (ns - 1) * kc >= H or tiles * ns > 2048 + tiles:
            continue
        cost = -(-(tiles * ns) // slots) * (kc + 96)
        if best is None or cost < best:
            best, best_ns = cost, ns
    return best_ns


def test_noalloc_route_lowers_the_split_to_fit_and_still_matches_route():
    # 153 x 4 token/expert tiles: moe_route splits H = 7168 into several K ranges whose
    # partial logits (nsplit * T * E fp32) outgrow the 16 MiB array; the no-alloc call
    # lowers the split until one fits (here down to a single range) and must still give
    # moe_route's ids bit for bit and its weights within the certified bound
    T, H, E, k = 153 * 64, 7168, 256, 8
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ns = _router_plan_splits(T, H, E, sms)
    assert ns > 1 and ns * T * E * 4 > 16 << 20, (ns, sms)
    g = torch.Generator().manual_seed(11)
    x = torch.randn((T, H), generator=g).to(torch.bfloat16)
    Wg = torch.randn((E, H), generator=g) * 0.02
    ids_a = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w_a = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.moe_workspace_size(T, H, 64, E, E, k, 0), dtype=torch.uint8, device="cuda")
    moe.moe_workspace_init(ws)
    xd, Wd = x.cuda(), Wg.cuda()
    moe.moe_route(xd, Wd, None, k, True, ids_a, w_a, ws)
    for _ in range(2):
        ids_b = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
        w_b = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
        moe.moe_route_noalloc(xd, Wd, None, k, True, ids_b, w_b)
        torch.cuda.synchronize()
        assert torch.equal(ids_a, ids_b)
        B = router_bound(x, Wg, None, H)
        rel = np.expm1(4.0 * B)[:, None] + 128 * 2.0 ** -24
        wa, wb = w_a.cpu().double().numpy(), w_b.cpu().double().numpy()
        assert np.all(np.abs(wa - wb) <= rel * np.abs(wa) + 1e-7)


def test_noalloc_route_rejects_sizes_beyond_its_scratch():
    T, H, E = 20000, 64, 256  # T*(E+1) floats > 16 MiB even with a single K range
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    Wg = torch.zeros((E, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.moe_route_noalloc(x, Wg, None, 2, True, ids, w)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
