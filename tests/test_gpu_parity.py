"""GPU parity of the CUDA layer against the fp64 oracle, through the C ABI.

Small and mid-size workloads are compared in full (several M/N/K tiles, ragged
per-slot tails, partial N tiles); the full-size workloads compare routing and
permutation bit-exactly on every token and the layer output on sampled tokens.
Tolerances: see tests/parity_util.py.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import serving_router_gate_gb300 as moe
from serving_router_gate_gb300.layer import layer_from_inputs

from parity_util import (check_out, check_routing, check_x_perm, make, oracle_layer, oracle_routing, permute_with_rows,
                         oracle_threads, run_gpu, sample_tokens, to_cpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _threads():
    oracle_threads()


def _full_check(inp, local_start=0, local_count=-1, mode=0):
    g = run_gpu(inp, local_start, local_count, mode)
    ref = oracle_layer(to_cpu(inp), local_start, local_count, mode)
    check_routing(g, dict(ids=ref["ids"], w=ref["w"], w_masked=ref["w_masked"], slots=ref["slots"],
                          counts=ref["counts"], offsets=ref["offsets"], perm_src=ref["perm_src"],
                          pair_row=ref["pair_row"]), to_cpu(inp), masked=local_count >= 0)
    check_x_perm(g, inp["x"].cuda(), inp["cfg"].k)
    check_out(g["out"], ref["out"])
    st = moe.moe_get_device_status(g["layer"].ws)
    assert st == 0, f"device status {st}"
    return g, ref


# --------------------------------------------------------------------------- small / mid sizes, full compare

@pytest.mark.parametrize("renorm", [True, False])
def test_tiny_layer(renorm):
    _full_check(make("tiny", renorm=renorm))


MID = mi.MoEConfig("mid", T=1000, H=512, I=384, E=12, k=3, renorm=True, n_shared=1, I_shared=256,
                   shared_gate=True)


def test_mid_layer_with_gated_shared_expert():
    _full_check(mi.make_inputs(MID))


def test_partial_n_tiles_and_two_shared_experts():
    cfg = mi.MoEConfig("odd", T=200, H=320, I=320, E=5, k=2, renorm=False, n_shared=2, I_shared=192)
    _full_check(mi.make_inputs(cfg))


def test_replica_slots_with_zipf_bias():
    cfg = mi.MoEConfig("rep", T=700, H=256, I=256, E=10, S=13, n_hot=3, zipf_s=1.1, k=4, renorm=True)
    _full_check(mi.make_inputs(cfg))


def test_local_ranges_sum_to_full_and_mod_equals_skip():
    cfg = mi.MoEConfig("ranges", T=600, H=256, I=256, E=16, k=4, renorm=True)
    inp = mi.make_inputs(cfg)
    full, _ = _full_check(inp)
    acc = torch.zeros(cfg.T, cfg.H, dtype=torch.float64)
    for start in (0, 4, 8, 12):
        g_skip, ref = _full_check(inp, start, 4, moe.MOE_NONLOCAL_SKIP)
        g_mod, _ = _full_check(inp, start, 4, moe.MOE_NONLOCAL_MOD)
        # MOD computes the non-local pairs with weight 0: bitwise the same output
        assert torch.equal(g_skip["out"].view(torch.int16), g_mod["out"].view(torch.int16))
        assert int(g_mod["counts"].sum()) == cfg.T * cfg.k
        acc += g_skip["out"].double()
    check_out(acc.to(torch.bfloat16), full["out"].double().numpy(), "sum of local ranges")


def test_all_experts_selected_and_single_expert():
    _full_check(mi.make_inputs(mi.MoEConfig("kE", T=130, H=256, I=256, E=8, k=8, renorm=True)))
    _full_check(mi.make_inputs(mi.MoEConfig("k1", T=130, H=256, I=256, E=8, k=1, renorm=True)))


def test_one_hot_expert_gets_every_token():
    cfg = mi.MoEConfig("hot", T=900, H=256, I=256, E=8, k=2, renorm=False)
    inp = mi.make_inputs(cfg)
    inp["bias"] = torch.zeros(cfg.E)
    inp["bias"][5] = 50.0  # every token picks expert 5 first: one group of 900 rows (8 m-tiles)
    g, ref = _full_check(inp)
    assert int(g["counts"][5]) == cfg.T


def test_supported_envelope_extremes():
    # 512 experts (16 logits per lane in the select kernel, its shared memory above 48 KB),
    # k = 32, and the smallest hidden and intermediate sizes (one K step per GEMM)
    _full_check(mi.make_inputs(mi.MoEConfig("e512k32", T=150, H=64, I=64, E=512, k=32, renorm=True)))
    # 1024 slots (each of 512 experts replicated): 1024 GEMM groups, most of them with rows
    g, _ = _full_check(mi.make_inputs(mi.MoEConfig("s1024", T=400, H=128, I=64, E=512, S=1024, n_hot=512, k=8,
                                                   renorm=False)))
    assert int((g["counts"] > 0).sum()) > 900
    # 128 experts (4 logits per lane) with a gated shared expert
    _full_check(mi.make_inputs(mi.MoEConfig("e128", T=300, H=192, I=128, E=128, k=6, renorm=True, n_shared=1,
                                            I_shared=64, shared_gate=True)))


def test_local_range_without_pairs_gives_zero():
    cfg = mi.MoEConfig("empty", T=64, H=256, I=256, E=8, k=2, renorm=True)
    inp = mi.make_inputs(cfg)
    inp["bias"] = torch.zeros(cfg.E)
    inp["bias"][:4] = 60.0  # experts 4..7 are never chosen
    g, _ = _full_check(inp, 4, 4, moe.MOE_NONLOCAL_SKIP)
    assert g["rows"] == 0
    assert torch.count_nonzero(g["out"].float()) == 0


def test_zero_tokens_is_a_noop():
    inp = make("tiny")
    layer = layer_from_inputs(inp, "cuda")
    out = layer.forward(inp["x"][:0].cuda())
    assert out.shape == (0, 256)
    torch.cuda.synchronize()


def test_two_runs_are_bitwise_identical():
    inp = mi.make_inputs(MID)
    layer = layer_from_inputs(inp, "cuda")
    x = inp["x"].cuda()
    a = layer.forward(x).clone()
    b = layer.forward(x).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("mode", [0, 2])
def test_gemm_tile_modes_single_and_pairs(mode):
    # CTA pairs running 2-SM MMAs, each CTA loading its own half of the weight
    # tile (mode 2 forces them on a mid-size layer: groups with odd and even
    # m-tile counts, shared problem with an odd count), and single CTAs must
    # give the same results
    cfg = mi.MoEConfig("pairs", T=1400, H=512, I=384, E=6, k=3, renorm=True, n_shared=1, I_shared=384,
                       shared_gate=True)
    inp = mi.make_inputs(cfg)
    try:
        moe.moe_set_gemm_pair_mode(mode)
        g, _ = _full_check(inp)
        ref0 = g["out"]
        moe.moe_set_gemm_pair_mode(0 if mode else 2)
        g2 = run_gpu(inp)
        assert torch.equal(g2["out"].view(torch.int16), ref0.view(torch.int16))
    finally:
        moe.moe_set_gemm_pair_mode(1)


def test_programmatic_dependent_launch_on_and_off_agree():
    inp = mi.make_inputs(MID)
    layer = layer_from_inputs(inp, "cuda")
    x = inp["x"].cuda()
    try:
        moe.moe_set_pdl(False)
        a = layer.forward(x).clone()
        moe.moe_set_pdl(True)
        b = layer.forward(x).clone()
    finally:
        moe.moe_set_pdl(True)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert moe.moe_get_device_status(layer.ws) == 0


def test_cuda_graph_replay_matches_eager_launches():
    inp = mi.make_inputs(MID)
    layer = layer_from_inputs(inp, "cuda")
    x = inp["x"].cuda()
    c0 = moe.moe_get_launch_count()
    eager = layer.forward(x).clone()
    per_forward = moe.moe_get_launch_count() - c0
    assert per_forward >= 5  # router, permute, FC1, FC2, finalize at least
    g = layer.capture(x)
    # capture runs one forward on a side stream, then records one: both count
    assert moe.moe_get_launch_count() - c0 == 3 * per_forward
    layer.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(layer.out.view(torch.int16), eager.view(torch.int16))
    assert moe.moe_get_device_status(layer.ws) == 0


def test_replica_table_equals_identity_map():
    cfg = mi.MoEConfig("rep2", T=500, H=256, I=256, E=10, S=13, n_hot=3, k=3, renorm=True)
    inp = mi.make_inputs(cfg)
    g_rep = run_gpu(inp)
    ident = dict(inp)
    W1e = torch.empty((cfg.E,) + tuple(inp["W1"].shape[1:]), dtype=torch.bfloat16)
    W2e = torch.empty((cfg.E,) + tuple(inp["W2"].shape[1:]), dtype=torch.bfloat16)
    for s, e in enumerate(inp["expert_of_slot"].tolist()):
        W1e[e], W2e[e] = inp["W1"][s], inp["W2"][s]
    ident.update(W1=W1e, W2=W2e, rep_offset=None, rep_slots=None, cfg=cfg.with_(S=None, n_hot=0))
    g_id = run_gpu(ident)
    assert torch.equal(g_rep["topk_ids"], g_id["topk_ids"])
    np.testing.assert_allclose(g_rep["out"].float().numpy(), g_id["out"].float().numpy(), rtol=0, atol=2e-3)


# --------------------------------------------------------------------------- stages on their own

def test_stages_fc1_fc2_finalize_against_oracle_rows():
    cfg = MID
    inp = mi.make_inputs(cfg)
    g = run_gpu(inp)
    layer = g["layer"]
    rows = g["rows"]
    ref = oracle_layer(to_cpu(inp))
    dev = torch.device("cuda")
    h = torch.empty((cfg.T * cfg.k, cfg.I), dtype=torch.bfloat16, device=dev)
    y = torch.empty((cfg.T * cfg.k, cfg.H), dtype=torch.bfloat16, device=dev)
    moe.moe_grouped_fc1(layer.x_perm, layer.offsets, layer.W1, None, None, h, None, layer.ws)
    moe.moe_grouped_fc2(h, layer.offsets, layer.W2, None, None, y, None, layer.ws)
    torch.cuda.synchronize()
    # a sample of rows: h and y of row r equal the oracle's expert MLP of its (token, slot)
    perm = g["perm_src"].numpy()
    slots = ref["slots"].reshape(-1)
    xs = inp["x"]
    for r in sample_tokens(rows, 24, seed=1):
        p = int(perm[r])
        t, s = p // cfg.k, int(slots[p])
        y_ref, h_ref = oracle.expert_mlp(xs[t], inp["W1"][s], inp["W2"][s])
        h_ref_f = torch.from_numpy(h_ref.view(np.int16)).view(torch.bfloat16).double().numpy()
        hg = h[r].double().cpu().numpy()
        assert np.abs(hg - h_ref_f).max() <= 2.0 ** -7 * np.abs(h_ref_f).max() + 1e-6
        check_out(y[r:r + 1], y_ref[None, :], f"y row {r}")
    # finalize alone on the oracle-free GPU y reproduces moe_forward's output bitwise
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    W1s, W2s = mi.shared_concat(inp["W1s"], inp["W2s"])
    h_sh = torch.empty((cfg.T, cfg.I_shared), dtype=torch.bfloat16, device=dev)
    y_sh = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    x = xs.cuda()
    moe.moe_grouped_fc1(layer.x_perm, layer.offsets, layer.W1, x, W1s.cuda(), h, h_sh, layer.ws)
    moe.moe_grouped_fc2(h, layer.offsets, layer.W2, h_sh, W2s.cuda(), y, y_sh, layer.ws)
    moe.moe_finalize(y, layer.pair_row, layer.topk_w, y_sh, x, inp["w_s"].cuda(), out, layer.ws)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), layer.out.view(torch.int16))
    check_out(out, ref["out"])


def test_small_batch_splits_shared_fc2_and_matches_unsplit_stages():
    """At most 128 tokens: moe_forward splits the shared expert's FC2 over K into
    fp32 partials (I_sh / I ranges, here 4) summed by the combine.  The result
    agrees with the unsplit stage-by-stage path (bf16 shared output) to within
    one bf16 rounding of the shared term, and with the oracle."""
    cfg = mi.MoEConfig("split", T=37, H=256, I=128, E=9, k=3, renorm=False, n_shared=2, I_shared=256,
                       shared_gate=True)
    inp = mi.make_inputs(cfg)
    g = run_gpu(inp)
    layer = g["layer"]
    check_out(g["out"], oracle_layer(to_cpu(inp))["out"])
    dev = torch.device("cuda")
    P = cfg.T * cfg.k
    Ish = cfg.n_shared * cfg.I_shared
    h = torch.empty((P, cfg.I), dtype=torch.bfloat16, device=dev)
    y = torch.empty((P, cfg.H), dtype=torch.bfloat16, device=dev)
    h_sh = torch.empty((cfg.T, Ish), dtype=torch.bfloat16, device=dev)
    y_sh = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    W1s, W2s = mi.shared_concat(inp["W1s"], inp["W2s"])
    x = inp["x"].cuda()
    moe.moe_grouped_fc1(layer.x_perm, layer.offsets, layer.W1, x, W1s.cuda(), h, h_sh, layer.ws)
    moe.moe_grouped_fc2(h, layer.offsets, layer.W2, h_sh, W2s.cuda(), y, y_sh, layer.ws)
    moe.moe_finalize(y, layer.pair_row, layer.topk_w, y_sh, x, inp["w_s"].cuda(), out, layer.ws)
    torch.cuda.synchronize()
    a, b = out.float(), g["out"].float().to(dev)
    # the two differ by the bf16 rounding of y_shared (and the output rounding)
    tol = 2.0 ** -7 * (y_sh.float().abs() + a.abs()) + 1e-6
    assert bool(((a - b).abs() <= tol).all())
    assert moe.moe_get_device_status(layer.ws) == 0


# --------------------------------------------------------------------------- group-limited top-k

def test_grouped_topk_layer_full_compare():
    """moe_route_grouped: ids, weights, permutation and outputs against the oracle's
    group-limited top-k (8 groups of 4 experts, 3 groups kept)."""
    cfg = mi.MoEConfig("grouped", T=700, H=512, I=256, E=32, k=4, renorm=True, n_group=8, topk_group=3,
                       n_shared=1, I_shared=256)
    inp = mi.make_inputs(cfg)
    g, ref = _full_check(inp)
    ids = g["topk_ids"].numpy()
    assert max(len({int(e) // 4 for e in row}) for row in ids) <= 3
    # the restriction matters: plain top-k picks other experts for some tokens
    plain, _, _ = oracle.route(inp["x"], inp["Wg"], None, 4, True)
    assert not np.array_equal(plain, ids)


def test_grouped_topk_exact_group_tie_goes_to_lower_group():
    """Group 1 is a copy of group 0, so their scores tie exactly for every token: the
    fp32 gap is zero, the compensated and fp64 rechecks tie too, and the lower group
    must win (as in the oracle)."""
    cfg = mi.MoEConfig("gtie", T=300, H=256, I=128, E=16, k=2, renorm=True, n_group=4, topk_group=1)
    inp = mi.make_inputs(cfg)
    Wg = inp["Wg"].clone()
    Wg[4:8] = Wg[0:4]
    inp["Wg"] = Wg
    g, ref = _full_check(inp)
    ids = g["topk_ids"].numpy()
    assert not (ids // 4 == 1).any()  # group 1 never wins over its copy
    # group 0 wins for some tokens, and those needed the recheck
    assert (ids // 4 == 0).any()


# --------------------------------------------------------------------------- routing applied on the input

def _on_input_check(inp, local_start=0, local_count=-1, mode=0):
    g = run_gpu(inp, local_start, local_count, mode, on_input=True)
    ref = oracle_layer(to_cpu(inp), local_start, local_count, mode, on_input=True)
    check_routing(g, dict(ids=ref["ids"], w=ref["w"], w_masked=ref["w_masked"], slots=ref["slots"],
                          counts=ref["counts"], offsets=ref["offsets"], perm_src=ref["perm_src"],
                          pair_row=ref["pair_row"]), to_cpu(inp), masked=local_count >= 0)
    # x_perm rows are the routing weight times the token's row, rounded once to bf16:
    # against the oracle's weight (fp64), so within one bf16 rounding plus the weight error
    rows = g["rows"]
    perm = g["perm_src"].numpy()[:rows]
    k = inp["cfg"].k
    wm = ref["w_masked"].reshape(-1)[perm]
    x64 = inp["x"].double().numpy()[perm // k]
    xp = g["x_perm"][:rows].double().cpu().numpy()
    exp_rows = wm[:, None] * x64
    assert np.all(np.abs(xp - exp_rows) <= 2.0 ** -8 * np.abs(exp_rows) + 1e-6 * np.abs(x64) + 1e-30)
    check_out(g["out"], ref["out"])
    assert moe.moe_get_device_status(g["layer"].ws) == 0
    return g, ref


def test_routing_on_input_mid_layer():
    _on_input_check(mi.make_inputs(MID))


def test_routing_on_input_local_ranges_skip_mod_and_sum():
    cfg = mi.MoEConfig("oi_ranges", T=600, H=256, I=256, E=16, k=4, renorm=True)
    inp = mi.make_inputs(cfg)
    full, _ = _on_input_check(inp)
    acc = torch.zeros_like(full["out"], dtype=torch.float64)
    for start in (0, 8):
        gs, _ = _on_input_check(inp, start, 8, moe.MOE_NONLOCAL_SKIP)
        gm, _ = _on_input_check(inp, start, 8, moe.MOE_NONLOCAL_MOD)
        assert torch.equal(gs["out"].view(torch.int16), gm["out"].view(torch.int16))  # zero rows add nothing
        acc += gs["out"].double()
    a, b = acc.numpy(), full["out"].double().numpy()
    assert np.abs(a - b).max() <= 2.0 ** -7 * np.abs(b).max() + 1e-3


# --------------------------------------------------------------------------- E4M3 expert weights

def test_quantize_fp8_rows_bit_exact():
    g = torch.Generator().manual_seed(11)
    w = (torch.randn(300, 192, generator=g) * 0.02).to(torch.bfloat16)
    w[7] = 0.0
    w[9, 5] = 3.0  # a row with one large value: most others become subnormal E4M3
    q_ref, s_ref = oracle.quantize_fp8_rows(w)
    q = torch.empty((300, 192), dtype=torch.uint8, device="cuda")
    sc = torch.empty(300, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_rows(w.cuda(), q, sc)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


FP8_MID = MID.with_(name="mid_fp8", fp8=True)


def test_fp8_weights_mid_layer():
    _full_check(mi.make_inputs(FP8_MID))


def test_fp8_weights_with_subnormal_and_zero_values():
    """One large entry per row of slot 0's W1 pushes that row's other values into the
    E4M3 subnormal range (and some to zero): the widening to bf16 must stay exact."""
    inp = mi.make_inputs(FP8_MID)
    W1 = inp["W1"].clone()
    W1[0, :, 0] = 1000.0
    W1[1, :5] = 0.0  # all-zero rows: scale 0
    inp["W1"] = W1
    q, _ = oracle.quantize_fp8_rows(W1[0])
    assert ((q & 0x78) == 0).mean() > 0.3  # many subnormal or zero codes
    _full_check(inp)


def test_fp8_weights_partial_tiles_two_shared_and_short_batch():
    cfg = mi.MoEConfig("odd_fp8", T=200, H=320, I=320, E=5, k=2, renorm=False, n_shared=2, I_shared=192, fp8=True)
    _full_check(mi.make_inputs(cfg))
    # at most 32 tokens: the short-tile variant, and the split shared FC2
    cfg = mi.MoEConfig("short_fp8", T=24, H=256, I=128, E=9, k=3, renorm=True, n_shared=2, I_shared=256,
                       shared_gate=True, fp8=True)
    _full_check(mi.make_inputs(cfg))


def test_fp8_weights_with_routing_on_input():
    # the quantised expert paths keep apply_routing_on_input (the TensorRT-LLM PR #10985
    # review notes quantised MoE ops that drop it): rows scaled before FC1, outputs summed
    # with weight 1
    _on_input_check(mi.make_inputs(FP8_MID.with_(on_input=True)))


def test_fp8_stage_gemms_against_oracle_rows():
    inp = mi.make_inputs(FP8_MID)
    g = run_gpu(inp)
    layer = g["layer"]
    cfg = FP8_MID
    dev = torch.device("cuda")
    P = cfg.T * cfg.k
    h = torch.empty((P, cfg.I), dtype=torch.bfloat16, device=dev)
    y = torch.empty((P, cfg.H), dtype=torch.bfloat16, device=dev)
    moe.moe_grouped_fc1_fp8(layer.x_perm, layer.offsets, layer.W1q, layer.s1, None, None, None, h, None, layer.ws)
    moe.moe_grouped_fc2_fp8(h, layer.offsets, layer.W2q, layer.s2, None, None, None, y, None, layer.ws)
    torch.cuda.synchronize()
    q1, s1 = oracle.quantize_fp8_rows(inp["W1"])
    q2, s2 = oracle.quantize_fp8_rows(inp["W2"])
    perm = g["perm_src"].numpy()
    slots = g["slot_ids"].numpy().reshape(-1)
    for r in sample_tokens(g["rows"], 16, seed=3):
        p = int(perm[r])
        t, s = p // cfg.k, int(slots[p])
        y_ref, _ = oracle.expert_mlp_fp8(inp["x"][t], q1[s], s1[s], q2[s], s2[s])
        check_out(y[r:r + 1], y_ref[None, :], f"fp8 y row {r}")


# --------------------------------------------------------------------------- E4M3 weights and activations

def test_quantize_act_rows_bit_exact():
    g = torch.Generator().manual_seed(12)
    rows = [torch.randn(40, 192, generator=g) * sc for sc in (1e-3, 0.02, 1.0, 300.0)]
    v = torch.cat(rows)
    v[3] = 0.0                                        # all zero: scale 2^-126, q = 0
    v[5] = v[5] / v[5].abs().max() * 3584.0           # amax = 448 * 2^3 exactly
    v[6] = v[6] / v[6].abs().max() * 3600.0           # the next bf16 above
    v[7] = torch.full((192,), 2.0 ** -130)            # bf16 subnormals: the scale clamps at 2^-126
    v[8, 0] = 1e30                                    # one huge value: the rest round to zero
    v = v.to(torch.bfloat16)
    # row lengths for each staging layout of the kernel (1, 2, 4 vectors of 8 values
    # per thread and row) and for its two-pass loop (more than 8192 values)
    sets = [(192, v)] + [(K, (torch.randn(n, K, generator=g) * 3).to(torch.bfloat16))
                         for K, n in ((3072, 21), (7168, 33), (8192, 6), (8256, 4), (16448, 3))]
    for K, vv in sets:
        q_ref, s_ref = oracle.quantize_act_rows(vv)
        q = torch.empty(vv.shape, dtype=torch.uint8, device="cuda")
        sc = torch.empty(vv.shape[0], dtype=torch.float32, device="cuda")
        moe.moe_quantize_act_rows(vv.cuda(), q, sc)
        torch.cuda.synchronize()
        assert np.array_equal(q.cpu().numpy(), q_ref), K
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), K


W8A8_MID = MID.with_(name="mid_w8a8", fp8=True, act8=True)


def test_w8a8_mid_layer():
    _full_check(mi.make_inputs(W8A8_MID))


def test_w8a8_ragged_k_partial_tiles_two_shared_and_short_batch():
    # H = 320, I = 320, I_shared = 192: K is not a multiple of the 128-element E4M3 step
    cfg = mi.MoEConfig("odd_w8a8", T=200, H=320, I=320, E=5, k=2, renorm=False, n_shared=2, I_shared=192,
                       fp8=True, act8=True)
    _full_check(mi.make_inputs(cfg))
    # at most 32 tokens: the short-tile variant, and the split shared FC2
    cfg = mi.MoEConfig("short_w8a8", T=24, H=256, I=128, E=9, k=3, renorm=True, n_shared=2, I_shared=256,
                       shared_gate=True, fp8=True, act8=True)
    _full_check(mi.make_inputs(cfg))
    # no shared expert: the token rows' codes go to the pair rows only
    cfg = mi.MoEConfig("noshared_w8a8", T=300, H=256, I=256, E=6, k=2, renorm=True, fp8=True, act8=True)
    _full_check(mi.make_inputs(cfg))


@pytest.mark.parametrize("act8", [False, True])
def test_shared_split_with_more_ranges_than_k_steps(act8):
    # I = 64 and 576 shared columns: the shared FC2 splits into 8 K ranges, more than
    # its K steps fill (9 bf16 steps of 64 or 5 E4M3 steps of 128); empty ranges add zeros
    cfg = mi.MoEConfig("split_empty", T=16, H=128, I=64, E=4, k=2, renorm=True, n_shared=1, I_shared=576,
                       fp8=act8, act8=act8)
    _full_check(mi.make_inputs(cfg))


def test_w8a8_local_ranges_and_routing_on_input():
    inp = mi.make_inputs(W8A8_MID)
    # a local range: fewer routed rows than the buffers hold (the quantiser reads the count on the device)
    _full_check(inp, 4, 5, moe.MOE_NONLOCAL_SKIP)
    _full_check(inp, 4, 5, moe.MOE_NONLOCAL_MOD)
    _on_input_check(mi.make_inputs(W8A8_MID.with_(on_input=True)))


def test_w8a8_replica_slots_grouped_topk_and_k_extremes():
    rep = mi.MoEConfig("rep_w8a8", T=700, H=256, I=256, E=10, S=13, n_hot=3, zipf_s=1.1, k=4, renorm=True,
                       fp8=True, act8=True)
    _full_check(mi.make_inputs(rep))
    grp = mi.MoEConfig("grp_w8a8", T=300, H=256, I=192, E=16, k=4, renorm=False, n_group=4, topk_group=2,
                       n_shared=1, I_shared=256, fp8=True, act8=True)
    _full_check(mi.make_inputs(grp))
    for k in (1, 6):  # top-1, and every expert of the batch
        cfg = mi.MoEConfig(f"k{k}_w8a8", T=130, H=256, I=128, E=6, k=k, renorm=True, fp8=True, act8=True)
        _full_check(mi.make_inputs(cfg))


def test_w8a8_empty_range_zero_tokens_and_determinism():
    cfg = mi.MoEConfig("empty_w8a8", T=100, H=256, I=256, E=8, k=2, renorm=True, fp8=True, act8=True)
    inp = mi.make_inputs(cfg)
    inp["bias"] = torch.zeros(cfg.E)
    inp["bias"][:4] = 60.0  # experts 4..7 are never chosen
    g, _ = _full_check(inp, 4, 4, moe.MOE_NONLOCAL_SKIP)
    assert g["rows"] == 0 and torch.count_nonzero(g["out"].float()) == 0
    layer = layer_from_inputs(mi.make_inputs(W8A8_MID), "cuda")
    assert layer.forward(torch.zeros((0, W8A8_MID.H), dtype=torch.bfloat16, device="cuda")).shape[0] == 0
    x = mi.make_inputs(W8A8_MID)["x"].cuda()
    a = layer.forward(x).clone()
    b = layer.forward(x).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert moe.moe_get_device_status(layer.ws) == 0


def test_w8a8_stage_gemms_against_oracle_rows():
    inp = mi.make_inputs(W8A8_MID)
    g = run_gpu(inp)
    layer = g["layer"]
    cfg = W8A8_MID
    dev = torch.device("cuda")
    P = cfg.T * cfg.k
    xq = torch.empty((P, cfg.H), dtype=torch.uint8, device=dev)
    sx = torch.empty(P, dtype=torch.float32, device=dev)
    h = torch.empty((P, cfg.I), dtype=torch.bfloat16, device=dev)
    hq = torch.empty((P, cfg.I), dtype=torch.uint8, device=dev)
    sh = torch.empty(P, dtype=torch.float32, device=dev)
    y = torch.empty((P, cfg.H), dtype=torch.bfloat16, device=dev)
    permute_with_rows(layer, inp["x"].cuda())  # the layer's own forward copies no rows at this size
    moe.moe_quantize_act_rows(layer.x_perm, xq, sx)
    moe.moe_grouped_fc1_w8a8(xq, sx, layer.offsets, layer.W1q, layer.s1, None, None, None, None, h, None, layer.ws)
    moe.moe_quantize_act_rows(h, hq, sh)
    moe.moe_grouped_fc2_w8a8(hq, sh, layer.offsets, layer.W2q, layer.s2, None, None, None, None, y, None, layer.ws)
    torch.cuda.synchronize()
    q1, s1 = oracle.quantize_fp8_rows(inp["W1"])
    q2, s2 = oracle.quantize_fp8_rows(inp["W2"])
    perm = g["perm_src"].numpy()
    slots = g["slot_ids"].numpy().reshape(-1)
    for r in sample_tokens(g["rows"], 16, seed=4):
        p = int(perm[r])
        t, s = p // cfg.k, int(slots[p])
        y_ref, _ = oracle.expert_mlp_fp8(inp["x"][t], q1[s], s1[s], q2[s], s2[s], act8=True)
        check_out(y[r:r + 1], y_ref[None, :], f"w8a8 y row {r}")
    assert moe.moe_get_device_status(layer.ws) == 0


# --------------------------------------------------------------------------- device-side error paths

def test_out_of_range_expert_ids_are_dropped_and_flagged():
    inp = make("tiny")
    layer = layer_from_inputs(inp, "cuda")
    x = inp["x"].cuda()
    layer.route(x)
    layer.topk_ids[3, 1] = 1000   # caught by the permute kernel's bounds check
    layer.topk_ids[7, 0] = -5
    layer.permute(x)
    layer.expert_forward(x)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(layer.ws) & moe.MOE_ERR_DEVICE_BOUNDS
    assert int(layer.pair_row[3, 1]) == -1 and int(layer.pair_row[7, 0]) == -1
    assert int(layer.counts.sum()) == 64 * 2 - 2
    assert moe.moe_get_device_status(layer.ws) == 0  # reading clears the word


def test_bounded_wait_times_out_with_status():
    ws = torch.zeros(1 << 12, dtype=torch.uint8, device="cuda")
    moe.moe_workspace_init(ws)
    moe.moe_debug_wait_timeout(ws, 2_000_000)  # 2 ms; nothing ever arrives
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_TIMEOUT
    # the context is still usable
    a = torch.ones(4, device="cuda")
    assert float((a + a).sum()) == 8.0


# --------------------------------------------------------------------------- full-size workloads

@pytest.mark.parametrize("T", [1, 8, 32, 128])
def test_decode_workload_full(T):
    _full_check(make(f"dsv2_lite_like_decode_t{T}"))


def _tail_tile_tokens(g, k, n):
    """Tokens with a pair in the last m-tile of its slot, where that tile is partial (fewer
    than 128 rows): the last row of up to n such slots, spread over the slot range."""
    off = g["offsets"].numpy().astype(np.int64)
    perm = g["perm_src"].numpy()
    cnt = off[1:] - off[:-1]
    slots = np.flatnonzero((cnt > 0) & (cnt % 128 != 0))
    if len(slots) > n:
        slots = slots[np.linspace(0, len(slots) - 1, n).astype(np.int64)]
    return np.unique(perm[off[slots + 1] - 1] // k).astype(np.int64)


def _full_size(name, n_samples, local_ranges=None, n_tail=0):
    cfg = mi.CONFIGS[name]
    inp = mi.make_inputs(cfg, device="cpu", weights_device="cuda")
    inp_cpu = to_cpu(inp)
    g = run_gpu(inp)
    ref = oracle_routing(inp_cpu)
    check_routing(g, ref, inp_cpu, masked=False)
    if not cfg.on_input:  # rows scaled by the weights are checked in the routing-on-input tests
        check_x_perm(g, inp["x"].cuda(), cfg.k)
    tok = sample_tokens(cfg.T, n_samples)
    if n_tail:
        tok = np.union1d(tok, _tail_tile_tokens(g, cfg.k, n_tail))
    part = oracle_layer(inp_cpu, tokens=tok)
    check_out(g["out"][tok], part["out"])
    assert moe.moe_get_device_status(g["layer"].ws) == 0
    if local_ranges:
        acc = torch.zeros(cfg.T, cfg.H, dtype=torch.float64)
        for start, count in local_ranges:
            gl = run_gpu(inp, start, count, moe.MOE_NONLOCAL_SKIP)
            refl = oracle_routing(inp_cpu, start, count, moe.MOE_NONLOCAL_SKIP)
            check_routing(gl, refl, inp_cpu, masked=True)
            pl = oracle_layer(inp_cpu, start, count, moe.MOE_NONLOCAL_SKIP, tokens=tok[:8])
            check_out(gl["out"][tok[:8]], pl["out"], f"local range {start}")
            acc += gl["out"].double()
            del gl
        check_out(acc.to(torch.bfloat16), g["out"].double().numpy(), "sum of local ranges")
    return g


def test_qwen2_moe_like_prefill_full_size():
    _full_size("qwen2_moe_like_prefill", 48)


def test_large_expert_prefill_full_size_and_local_ranges():
    _full_size("large_expert_prefill", 64, local_ranges=[(0, 64), (64, 64), (128, 64), (192, 64)], n_tail=16)


def test_redundant_slots_prefill_full_size():
    _full_size("redundant_slots_prefill", 64, n_tail=16)


def test_grouped_topk_prefill_full_size():
    _full_size("grouped_topk_prefill", 32)


def test_routing_on_input_prefill_full_size():
    _full_size("routing_on_input_prefill", 32)


@pytest.mark.parametrize("name", ["dsv2_lite_like_decode_t1_fp8", "dsv2_lite_like_decode_t32_fp8",
                                  "qwen2_moe_like_prefill_fp8"])
def test_fp8_full_size(name):
    _full_size(name, 16 if "prefill" in name else 32)


@pytest.mark.parametrize("name", ["dsv2_lite_like_decode_t1_w8a8", "dsv2_lite_like_decode_t32_w8a8",
                                  "qwen2_moe_like_prefill_w8a8"])
def test_w8a8_full_size(name):
    _full_size(name, 16 if "prefill" in name else 32)
