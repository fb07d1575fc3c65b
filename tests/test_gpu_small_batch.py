"""GPU parity of the small-batch paths (decode sizes) against the fp64 oracle.

Batches of at most 16 tokens route in one launch (logits over many CTAs, the
selection by the CTA that finishes last), and batches of at most 256 pairs
permute in one CTA entirely in shared memory.  Every routing variant those
paths serve is compared here in full:
plain and renormalised top-k, replica slots with a Zipf bias, local ranges
(SKIP and MOD, summing to the full layer), routing on the input, group-limited
top-k, 512 experts with k = 32, exact logit ties, E4M3 weights and activations,
and the shared expert with and without its gate.  Tolerances: tests/parity_util.py.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import serving_router_gate_gb300 as moe

from parity_util import check_out, check_routing, check_x_perm, oracle_layer, oracle_threads, run_gpu, to_cpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _threads():
    oracle_threads()


def _check(inp, local_start=0, local_count=-1, mode=0, on_input=None):
    g = run_gpu(inp, local_start, local_count, mode, on_input=on_input)
    ref = oracle_layer(to_cpu(inp), local_start, local_count, mode, on_input=on_input)
    check_routing(g, dict(ids=ref["ids"], w=ref["w"], w_masked=ref["w_masked"], slots=ref["slots"],
                          counts=ref["counts"], offsets=ref["offsets"], perm_src=ref["perm_src"],
                          pair_row=ref["pair_row"]), to_cpu(inp), masked=local_count >= 0)
    if not (on_input if on_input is not None else inp["cfg"].on_input):
        check_x_perm(g, inp["x"].cuda(), inp["cfg"].k)
    check_out(g["out"], ref["out"])
    st = moe.moe_get_device_status(g["layer"].ws)
    assert st == 0, f"device status {st}"
    return g, ref


@pytest.mark.parametrize("T", [1, 2, 5, 8, 16])
@pytest.mark.parametrize("renorm", [False, True])
def test_small_batches_with_two_shared_experts(T, renorm):
    cfg = mi.MoEConfig(f"sb{T}", T=T, H=512, I=256, E=64, k=6, renorm=renorm, n_shared=2, I_shared=512)
    _check(mi.make_inputs(cfg))


@pytest.mark.parametrize("T", [1, 7])
def test_small_batch_gated_shared_expert_and_wide_hidden(T):
    # H = 7168 splits each expert's row into parts over four warps (npl = 7 pieces per lane)
    cfg = mi.MoEConfig(f"sbw{T}", T=T, H=7168, I=128, E=32, k=4, renorm=True, n_shared=1, I_shared=128,
                       shared_gate=True)
    _check(mi.make_inputs(cfg))


def test_small_batch_replica_slots_and_zipf_bias():
    cfg = mi.MoEConfig("sb_rep", T=13, H=256, I=128, E=10, S=13, n_hot=3, zipf_s=1.1, k=4, renorm=True)
    _check(mi.make_inputs(cfg))


def test_small_batch_local_ranges_skip_mod_and_sum():
    cfg = mi.MoEConfig("sb_ranges", T=11, H=256, I=256, E=16, k=4, renorm=True)
    inp = mi.make_inputs(cfg)
    full, _ = _check(inp)
    acc = torch.zeros(cfg.T, cfg.H, dtype=torch.float64)
    for start in (0, 4, 8, 12):
        gs, _ = _check(inp, start, 4, moe.MOE_NONLOCAL_SKIP)
        gm, _ = _check(inp, start, 4, moe.MOE_NONLOCAL_MOD)
        assert torch.equal(gs["out"].view(torch.int16), gm["out"].view(torch.int16))
        acc += gs["out"].double()
    check_out(acc.to(torch.bfloat16), full["out"].double().numpy(), "sum of local ranges")


def test_small_batch_routing_on_input():
    cfg = mi.MoEConfig("sb_oi", T=9, H=256, I=256, E=12, k=3, renorm=True, n_shared=1, I_shared=256,
                       shared_gate=True, on_input=True)
    g = run_gpu(mi.make_inputs(cfg), on_input=True)
    inp = mi.make_inputs(cfg)
    ref = oracle_layer(to_cpu(inp), on_input=True)
    check_routing(g, dict(ids=ref["ids"], w=ref["w"], w_masked=ref["w_masked"], slots=ref["slots"],
                          counts=ref["counts"], offsets=ref["offsets"], perm_src=ref["perm_src"],
                          pair_row=ref["pair_row"]), to_cpu(inp), masked=False)
    rows = g["rows"]
    perm = g["perm_src"].numpy()[:rows]
    wm = ref["w_masked"].reshape(-1)[perm]
    x64 = inp["x"].double().numpy()[perm // cfg.k]
    xp = g["x_perm"][:rows].double().cpu().numpy()
    exp_rows = wm[:, None] * x64
    assert np.all(np.abs(xp - exp_rows) <= 2.0 ** -8 * np.abs(exp_rows) + 1e-6 * np.abs(x64) + 1e-30)
    check_out(g["out"], ref["out"])


def test_small_batch_grouped_topk_and_group_tie():
    cfg = mi.MoEConfig("sb_grp", T=6, H=256, I=128, E=64, k=6, renorm=False, n_group=8, topk_group=3,
                       n_shared=1, I_shared=128)
    _check(mi.make_inputs(cfg))
    # group 1 a copy of group 0: the exact tie goes to the lower group after the rechecks
    tie = mi.MoEConfig("sb_gtie", T=10, H=256, I=128, E=16, k=2, renorm=True, n_group=4, topk_group=1)
    inp = mi.make_inputs(tie)
    Wg = inp["Wg"].clone()
    Wg[4:8] = Wg[0:4]
    inp["Wg"] = Wg
    g, _ = _check(inp)
    ids = g["topk_ids"].numpy()
    assert not (ids // 4 == 1).any()


def test_small_batch_exact_expert_ties_go_to_lower_id():
    # experts 2k+1 copy experts 2k: every candidate cluster is an exact tie, decided by the
    # compensated and fp64 rechecks in favour of the lower id
    cfg = mi.MoEConfig("sb_tie", T=12, H=256, I=128, E=16, k=3, renorm=True)
    inp = mi.make_inputs(cfg)
    Wg = inp["Wg"].clone()
    Wg[1::2] = Wg[0::2]
    inp["Wg"] = Wg
    g, _ = _check(inp)
    ids = g["topk_ids"].numpy()
    assert (ids[:, 0] % 2 == 0).all()
    layer = g["layer"]
    assert moe.moe_get_route_stats(layer.ws) >= cfg.T


def test_small_batch_envelope_extremes():
    # 512 experts (16 logits per lane), k = 32: 16 tokens x 32 = 512 pairs take the larger
    # permutation path, 8 tokens x 32 = 256 pairs the one-CTA one
    for T in (8, 16):
        _check(mi.make_inputs(mi.MoEConfig(f"sb_e512_{T}", T=T, H=64, I=64, E=512, k=32, renorm=True)))
    # 1024 slots
    _check(mi.make_inputs(mi.MoEConfig("sb_s1024", T=16, H=128, I=64, E=512, S=1024, n_hot=512, k=8,
                                       renorm=False)))


@pytest.mark.parametrize("T", [1, 8])
def test_small_batch_e4m3_weights_and_activations(T):
    cfg = mi.MoEConfig(f"sb_w8a8_{T}", T=T, H=512, I=256, E=16, k=4, renorm=True, n_shared=2, I_shared=256,
                       fp8=True, act8=True)
    _check(mi.make_inputs(cfg))
    _check(mi.make_inputs(cfg.with_(name=f"sb_w8_{T}", act8=False)))


def test_small_batch_back_to_back_calls_reuse_the_ticket():
    # the router's ticket returns to 0 after every launch: many launches in a row, in one
    # CUDA graph and eagerly, give the same ids as the first
    cfg = mi.MoEConfig("sb_rep_calls", T=3, H=256, I=128, E=24, k=4, renorm=True)
    inp = mi.make_inputs(cfg)
    g, _ = _check(inp)
    layer = g["layer"]
    x = inp["x"].cuda()
    first = layer.topk_ids[:cfg.T].clone()
    for _ in range(5):
        layer.route(x)
    graph = layer.capture(x)
    for _ in range(5):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(layer.topk_ids[:cfg.T], first)
    assert moe.moe_get_device_status(layer.ws) == 0
