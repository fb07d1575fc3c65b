"""Pins of the fp64 CPU oracle against what the method and mathematics fix.

Every check here is independent of the oracle's own code path: brute force over
subsets, numpy matrix products, torch casts, hand-worked examples in
tests/golden/, closed forms (top_k = 1, top_k = E, shared expert alone) and
invariants (counts, bijections, token permutation, disjoint local ranges, slot
maps).  A dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""
import itertools
import os

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_np(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def _small_cfg(**kw):
    base = dict(name="pin", T=24, H=64, I=64, E=6, k=2, renorm=True)
    base.update(kw)
    return mi.MoEConfig(**base)


def _numpy_mlp(x64, W1, W2):
    """Dense SwiGLU MLP with numpy products; h rounded through torch's bf16 cast."""
    I = W1.shape[0] // 2
    W1n, W2n = _bf16_np(W1), _bf16_np(W2)
    g = x64 @ W1n[:I].T
    u = x64 @ W1n[I:].T
    a = g / (1.0 + np.exp(-g)) * u
    h = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    return h @ W2n.T


# --------------------------------------------------------------------------- bf16

def test_bf16_round_matches_torch_on_fp32_values():
    g = torch.Generator().manual_seed(1)
    vals = torch.cat([
        torch.randn(20000, generator=g) * 10.0 ** torch.randint(-40, 38, (20000,), generator=g).float(),
        torch.tensor([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-40, -1e-40, 2.0 ** -133, 2.0 ** -134,
                      1.00390625, 1.01171875, 65504.0]),
    ]).float()
    want = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f64_to_bf16(float(v)) for v in vals.tolist()], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_bf16_round_ties_to_even_and_overflow():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to the even significand (1.0)
    assert oracle.f64_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 lies halfway between 1+2^-7 and 1+2^-6: even is 1+2^-6
    assert oracle.f64_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above the halfway point rounds up (a value no fp32 can hold exactly)
    assert oracle.f64_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.f64_to_bf16(1e39) == 0x7F80
    assert oracle.f64_to_bf16(-1e39) == 0xFF80
    for b in (0x0001, 0x3F80, 0x4049, 0xC2F7, 0x7F7F):
        assert oracle.f64_to_bf16(oracle.bf16_to_f64(b)) == b


# --------------------------------------------------------------------------- router

def test_gate_logits_match_numpy_product():
    cfg = _small_cfg(T=40, H=96, E=7, zipf_s=1.1)
    inp = mi.make_inputs(cfg)
    ids, w, logits = oracle.route(inp["x"], inp["Wg"], inp["bias"], cfg.k, cfg.renorm)
    ref = _bf16_np(inp["x"]) @ inp["Wg"].double().numpy().T + inp["bias"].double().numpy()
    np.testing.assert_allclose(logits, ref, rtol=0, atol=1e-12)


def test_topk_matches_brute_force_over_subsets():
    for E, k in ((8, 2), (7, 3), (6, 6), (5, 1)):
        cfg = _small_cfg(T=30, H=48, E=E, k=k)
        inp = mi.make_inputs(cfg)
        ids, w, logits = oracle.route(inp["x"], inp["Wg"], None, k, False)
        for t in range(cfg.T):
            l = logits[t]
            best = max(itertools.combinations(range(E), k), key=lambda s: (sum(l[list(s)]),
                                                                              [-i for i in s]))
            assert sorted(ids[t].tolist()) == sorted(best)
            # descending logit within the selection
            assert all(l[ids[t][j]] >= l[ids[t][j + 1]] for j in range(k - 1))


def test_topk_exact_ties_go_to_lower_index():
    H, E, k = 32, 8, 3
    g = torch.Generator().manual_seed(5)
    Wg = torch.randn(E, H, generator=g) * 0.02
    Wg[6] = Wg[2]          # experts 2 and 6 always tie
    Wg[5] = Wg[1]          # experts 1 and 5 always tie
    x = torch.randn(16, H, generator=g).to(torch.bfloat16)
    x[3] = 0               # an all-zero token: every logit is exactly 0
    ids, w, logits = oracle.route(x, Wg, None, k, False)
    assert ids[3].tolist() == [0, 1, 2]
    for t in range(16):
        sel = ids[t].tolist()
        for lo, hi in ((2, 6), (1, 5)):
            if hi in sel:
                assert lo in sel and sel.index(lo) < sel.index(hi)


def test_softmax_and_renorm_weights():
    cfg = _small_cfg(T=20, H=64, E=6, k=6)
    inp = mi.make_inputs(cfg)
    _, w_all, logits = oracle.route(inp["x"], inp["Wg"], None, 6, False)
    np.testing.assert_allclose(w_all.sum(1), 1.0, atol=1e-14)
    # k < E, renorm off: the weights are the softmax probabilities of the selected experts
    ids, w, logits = oracle.route(inp["x"], inp["Wg"], None, 2, False)
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    np.testing.assert_allclose(w, np.take_along_axis(p, ids, 1), rtol=1e-13)
    # renorm on: the selected probabilities divided by their sum
    ids_r, w_r, _ = oracle.route(inp["x"], inp["Wg"], None, 2, True)
    assert np.array_equal(ids, ids_r)
    sel = np.take_along_axis(p, ids, 1)
    np.testing.assert_allclose(w_r, sel / sel.sum(1, keepdims=True), rtol=1e-13)
    # k = 1 with renorm: weight exactly 1
    _, w1, _ = oracle.route(inp["x"], inp["Wg"], None, 1, True)
    assert np.all(w1 == 1.0)


# --------------------------------------------------------------------------- slots, mask, permute

def _read_golden(name):
    lines = [ln.split("#")[0].strip() for ln in open(os.path.join(GOLDEN, name))]
    return [ln for ln in lines if ln]


def test_slot_map_golden_example():
    lines = _read_golden("slot_map_example.txt")
    ro = np.array(lines[0].split()[1:], np.int32)
    rs = np.array(lines[1].split()[1:], np.int32)
    ids, want = [], []
    for ln in lines[2:]:
        lhs, rhs = ln.split("->")
        ids.append([int(v) for v in lhs.split()[1:]])
        want.append([int(v) for v in rhs.split()])
    got = oracle.slot_map(np.array(ids, np.int32), ro, rs)
    assert got.tolist() == want


def test_identity_slot_table_equals_no_map():
    g = torch.Generator().manual_seed(2)
    ids = torch.randint(0, 9, (50, 3), generator=g).numpy().astype(np.int32)
    ro = np.arange(10, dtype=np.int32)
    rs = np.arange(9, dtype=np.int32)
    assert np.array_equal(oracle.slot_map(ids, ro, rs), oracle.slot_map(ids))
    assert np.array_equal(oracle.slot_map(ids), ids)


def test_ep_mask_and_remap_golden_example():
    lines = _read_golden("ep_mask_and_remap_example.txt")
    start = int(lines[0].split()[1])
    count = int(lines[1].split()[1])
    ids, w, want = [], [], []
    for ln in lines[2:]:
        lhs, rhs = ln.split("->")
        a = lhs.split()
        ids.append(int(a[0]))
        w.append(float(a[1]))
        want.append(rhs.split())
    ids = np.array(ids, np.int32)
    w = np.array(w)
    s_mod, w_mod, m = oracle.local_mask(ids, w, start, count, oracle.NONLOCAL_MOD)
    s_skip, w_skip, m2 = oracle.local_mask(ids, w, start, count, oracle.NONLOCAL_SKIP)
    for i, r in enumerate(want):
        assert int(m[i]) == int(r[0]) and int(m2[i]) == int(r[0])
        assert w_mod[i] == float(r[1]) and w_skip[i] == float(r[1])
        assert s_mod[i] == int(r[2])
        assert s_skip[i] == int(r[3])


def test_permutation_invariants():
    g = torch.Generator().manual_seed(3)
    for S, P in ((1, 1), (5, 0), (7, 300), (40, 1000)):
        slots = torch.randint(-1, S, (P,), generator=g).numpy().astype(np.int32)
        counts, offsets, perm_src, pair_row = oracle.permute(slots, S)
        kept = int((slots >= 0).sum())
        assert counts.sum() == kept and offsets[0] == 0 and offsets[S] == kept
        assert np.array_equal(np.diff(offsets), counts)
        assert np.array_equal(np.bincount(slots[slots >= 0], minlength=S), counts)
        # pair_row and perm_src are mutually inverse on the kept pairs
        assert sorted(perm_src.tolist()) == sorted(np.nonzero(slots >= 0)[0].tolist())
        for r, p in enumerate(perm_src):
            assert pair_row[p] == r
        assert np.all(pair_row[slots < 0] == -1)
        # each slot's rows hold its pairs in ascending pair index
        for s in range(S):
            rows = perm_src[offsets[s]:offsets[s + 1]]
            assert np.all(slots[rows] == s) and np.all(np.diff(rows) > 0)


# --------------------------------------------------------------------------- expert MLP and the layer

def test_expert_mlp_matches_numpy_dense_mlp():
    cfg = _small_cfg(H=96, I=80, E=1)
    inp = mi.make_inputs(cfg)
    x = inp["x"][:5]
    W1, W2 = inp["W1"][0], inp["W2"][0]
    ref = _numpy_mlp(_bf16_np(x), W1, W2)
    for t in range(5):
        y, h = oracle.expert_mlp(x[t], W1, W2)
        np.testing.assert_allclose(y, ref[t], rtol=0, atol=1e-3 * np.abs(ref[t]).max())


def test_top1_with_renorm_equals_single_dense_expert():
    cfg = _small_cfg(T=16, H=64, I=64, E=5, k=1, renorm=True)
    inp = mi.make_inputs(cfg)
    res = oracle.moe_layer(inp["x"], inp["Wg"], None, 1, True, inp["W1"], inp["W2"])
    x64 = _bf16_np(inp["x"])
    for t in range(cfg.T):
        e = int(res["ids"][t, 0])
        ref = _numpy_mlp(x64[t:t + 1], inp["W1"][e], inp["W2"][e])[0]
        np.testing.assert_allclose(res["out"][t], ref, rtol=0, atol=1e-3 * np.abs(ref).max())


def test_topk_all_experts_equals_dense_softmax_mixture():
    cfg = _small_cfg(T=12, H=64, I=64, E=4, k=4, renorm=True)
    inp = mi.make_inputs(cfg)
    res = oracle.moe_layer(inp["x"], inp["Wg"], None, 4, True, inp["W1"], inp["W2"])
    x64 = _bf16_np(inp["x"])
    l = x64 @ inp["Wg"].double().numpy().T
    p = np.exp(l - l.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ref = sum(p[:, e:e + 1] * _numpy_mlp(x64, inp["W1"][e], inp["W2"][e]) for e in range(4))
    np.testing.assert_allclose(res["out"], ref, rtol=0, atol=1e-3 * np.abs(ref).max())


def test_shared_expert_alone_and_sigmoid_gate():
    cfg = _small_cfg(T=10, H=64, I=64, E=4, k=2, n_shared=2, I_shared=48, shared_gate=True)
    inp = mi.make_inputs(cfg)
    W2zero = torch.zeros_like(inp["W2"])
    res = oracle.moe_layer(inp["x"], inp["Wg"], None, 2, True, inp["W1"], W2zero,
                           W1s=inp["W1s"], W2s=inp["W2s"], shared_gate_w=inp["w_s"])
    x64 = _bf16_np(inp["x"])
    gate = 1.0 / (1.0 + np.exp(-(x64 @ _bf16_np(inp["w_s"]))))
    ref = sum(_numpy_mlp(x64, inp["W1s"][i], inp["W2s"][i]) for i in range(2)) * gate[:, None]
    np.testing.assert_allclose(res["out"], ref, rtol=0, atol=1e-3 * np.abs(ref).max())
    # without the gate vector the shared experts are added unscaled
    res2 = oracle.moe_layer(inp["x"], inp["Wg"], None, 2, True, inp["W1"], W2zero,
                            W1s=inp["W1s"], W2s=inp["W2s"])
    ref2 = sum(_numpy_mlp(x64, inp["W1s"][i], inp["W2s"][i]) for i in range(2))
    np.testing.assert_allclose(res2["out"], ref2, rtol=0, atol=1e-3 * np.abs(ref2).max())


def test_token_permutation_invariance_bitwise():
    cfg = _small_cfg(T=20, H=64, I=64, E=6, k=3, n_shared=1, I_shared=64, shared_gate=True)
    inp = mi.make_inputs(cfg)
    perm = torch.randperm(cfg.T, generator=torch.Generator().manual_seed(9))
    args = dict(W1s=inp["W1s"], W2s=inp["W2s"], shared_gate_w=inp["w_s"])
    a = oracle.moe_layer(inp["x"], inp["Wg"], None, 3, True, inp["W1"], inp["W2"], **args)
    b = oracle.moe_layer(inp["x"][perm], inp["Wg"], None, 3, True, inp["W1"], inp["W2"], **args)
    assert np.array_equal(a["out"][perm.numpy()], b["out"])
    assert np.array_equal(a["ids"][perm.numpy()], b["ids"])
    assert np.array_equal(a["counts"], b["counts"])


def test_disjoint_local_ranges_sum_to_full_layer():
    cfg = _small_cfg(T=30, H=64, I=64, E=8, k=3)
    inp = mi.make_inputs(cfg)
    full = oracle.moe_layer(inp["x"], inp["Wg"], None, 3, True, inp["W1"], inp["W2"])
    acc = np.zeros_like(full["out"])
    for start in (0, 2, 4, 6):
        part = oracle.moe_layer(inp["x"], inp["Wg"], None, 3, True, inp["W1"][start:start + 2],
                                inp["W2"][start:start + 2], local_start=start, local_count=2)
        mod = oracle.moe_layer(inp["x"], inp["Wg"], None, 3, True, inp["W1"][start:start + 2],
                               inp["W2"][start:start + 2], local_start=start, local_count=2,
                               mode=oracle.NONLOCAL_MOD)
        # MOD computes the non-local pairs with weight 0: they contribute exactly nothing
        assert np.array_equal(part["out"], mod["out"])
        assert mod["counts"].sum() == cfg.T * 3
        assert part["counts"].sum() == int(((full["ids"] >= start) & (full["ids"] < start + 2)).sum())
        acc += part["out"]
    np.testing.assert_allclose(acc, full["out"], rtol=0, atol=1e-12 * np.abs(full["out"]).max())
    # a range that owns no pair contributes exactly zero
    ids = full["ids"]
    unused = [e for e in range(8) if not (ids == e).any()]
    if unused:
        e = unused[0]
        z = oracle.moe_layer(inp["x"], inp["Wg"], None, 3, True, inp["W1"][e:e + 1],
                             inp["W2"][e:e + 1], local_start=e, local_count=1)
        assert np.all(z["out"] == 0.0)


def test_replica_slots_equal_identity_map():
    cfg = _small_cfg(T=40, H=64, I=64, E=8, k=3, S=11, n_hot=3, zipf_s=1.1)
    inp = mi.make_inputs(cfg)
    tab = mi.slot_table(cfg)
    W1e = inp["W1"].new_empty((8,) + tuple(inp["W1"].shape[1:]))
    W2e = inp["W2"].new_empty((8,) + tuple(inp["W2"].shape[1:]))
    for s, e in enumerate(tab["expert_of_slot"].tolist()):
        W1e[e] = inp["W1"][s]
        W2e[e] = inp["W2"][s]
    rep = oracle.moe_layer(inp["x"], inp["Wg"], inp["bias"], 3, True, inp["W1"], inp["W2"],
                           rep_offset=inp["rep_offset"], rep_slots=inp["rep_slots"])
    ident = oracle.moe_layer(inp["x"], inp["Wg"], inp["bias"], 3, True, W1e, W2e)
    assert np.array_equal(rep["out"], ident["out"])
    assert rep["counts"].sum() == cfg.T * 3
    # replica choice follows the token index
    ro, rs = tab["rep_offset"].numpy(), tab["rep_slots"].numpy()
    for t in range(cfg.T):
        for j in range(3):
            e = rep["ids"][t, j]
            c = ro[e + 1] - ro[e]
            assert rep["slots_global"][t, j] == rs[ro[e] + t % c]


def test_moe_tokens_matches_batch_layer_on_a_sample():
    cfg = _small_cfg(T=25, H=64, I=64, E=6, k=2, n_shared=1, I_shared=32, shared_gate=True)
    inp = mi.make_inputs(cfg)
    args = dict(W1s=inp["W1s"], W2s=inp["W2s"], shared_gate_w=inp["w_s"])
    full = oracle.moe_layer(inp["x"], inp["Wg"], None, 2, True, inp["W1"], inp["W2"], **args)
    tok = np.array([24, 0, 7, 7, 13])
    part = oracle.moe_tokens(inp["x"], inp["Wg"], None, 2, True, inp["W1"], inp["W2"], tokens=tok, **args)
    assert np.array_equal(part["out"], full["out"][tok])
    assert np.array_equal(part["ids"], full["ids"][tok])


@pytest.mark.parametrize("threads", [1, 3])
def test_results_do_not_depend_on_thread_count(threads):
    cfg = _small_cfg(T=33, H=64, I=64, E=6, k=2)
    inp = mi.make_inputs(cfg)
    old = oracle.get_threads()
    try:
        oracle.set_threads(threads)
        a = oracle.moe_layer(inp["x"], inp["Wg"], None, 2, True, inp["W1"], inp["W2"])
    finally:
        oracle.set_threads(old)
    b = oracle.moe_layer(inp["x"], inp["Wg"], None, 2, True, inp["W1"], inp["W2"])
    assert np.array_equal(a["out"], b["out"])


# --------------------------------------------------------------------------- group-limited top-k

def _golden_kv(name):
    kv = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].split()
        if line:
            kv[line[0]] = [float(v) for v in line[1:]]
    return kv


def _route_given_logits(logits, k, n_group, topk_group, renorm=False):
    """x = e_0 (bf16 1.0), Wg[:, 0] = the logits: the oracle's logits are exactly these fp32 values."""
    E = len(logits)
    x = torch.zeros((1, 64), dtype=torch.bfloat16)
    x[0, 0] = 1.0
    Wg = torch.zeros((E, 64), dtype=torch.float32)
    Wg[:, 0] = torch.tensor(logits, dtype=torch.float32)
    return oracle.route(x, Wg, None, k, renorm, n_group, topk_group)


def test_grouped_topk_golden_example():
    g = _golden_kv("grouped_topk_example.txt")
    logits, k = g["logits"], int(g["k"][0])
    ids, w, l = _route_given_logits(logits, k, int(g["n_group"][0]), int(g["topk_group"][0]))
    assert ids[0].tolist() == [int(v) for v in g["grouped_ids"]]
    p = np.exp(np.array(logits) - max(logits))
    p /= p.sum()
    np.testing.assert_allclose(w[0], p[ids[0]], rtol=1e-15)
    ids_plain, _, _ = _route_given_logits(logits, k, 1, 1)
    assert ids_plain[0].tolist() == [int(v) for v in g["plain_ids"]]
    ids_tie, _, _ = _route_given_logits(g["tie_logits"], int(g["tie_k"][0]), int(g["n_group"][0]),
                                        int(g["tie_topk_group"][0]))
    assert ids_tie[0].tolist() == [int(v) for v in g["tie_ids"]]


def test_grouped_topk_reduces_to_plain_topk():
    cfg = _small_cfg(T=40, H=64, E=16, k=4)
    inp = mi.make_inputs(cfg)
    plain = oracle.route(inp["x"], inp["Wg"], None, 4, True)
    for n_group, topk_group in ((1, 1), (4, 4), (8, 8)):
        got = oracle.route(inp["x"], inp["Wg"], None, 4, True, n_group, topk_group)
        assert np.array_equal(got[0], plain[0]) and np.array_equal(got[1], plain[1])


def test_grouped_topk_against_numpy_selection():
    """Independent numpy selection on the oracle's own fp64 logits: the kept groups are
    the topk_group largest group maxima (lower index on ties), the ids the k largest
    logits inside them (lower id on ties), the weights the full-softmax probabilities."""
    cfg = _small_cfg(T=64, H=64, E=24, k=3)
    inp = mi.make_inputs(cfg)
    n_group, topk_group, k = 6, 2, 3
    ids, w, l = oracle.route(inp["x"], inp["Wg"], None, k, False, n_group, topk_group)
    gsize = 24 // n_group
    for t in range(cfg.T):
        gmax = l[t].reshape(n_group, gsize).max(1)
        keep = np.lexsort((np.arange(n_group), -gmax))[:topk_group]
        allowed = np.concatenate([np.arange(g * gsize, (g + 1) * gsize) for g in keep])
        order = allowed[np.lexsort((allowed, -l[t][allowed]))][:k]
        assert ids[t].tolist() == order.tolist()
        assert len({int(e) // gsize for e in ids[t]}) <= topk_group
        p = np.exp(l[t] - l[t].max())
        p /= p.sum()
        np.testing.assert_allclose(w[t], p[ids[t]], rtol=1e-12)


# --------------------------------------------------------------------------- routing applied on the input

def test_routing_on_input_top1_renorm_equals_plain_layer():
    """k = 1 with renorm: w = 1, so scaling the input changes nothing (bitwise)."""
    cfg = _small_cfg(T=16, H=64, I=64, E=5, k=1, renorm=True)
    inp = mi.make_inputs(cfg)
    a = oracle.moe_layer(inp["x"], inp["Wg"], None, 1, True, inp["W1"], inp["W2"])
    b = oracle.moe_layer(inp["x"], inp["Wg"], None, 1, True, inp["W1"], inp["W2"], on_input=True)
    assert np.array_equal(a["out"], b["out"])


def test_routing_on_input_matches_numpy_mlp_of_scaled_rows():
    """out_t = sum_j MLP_j(bf16(w_j x_t)), the scaled row rounded through torch's bf16 cast,
    the MLP a numpy dense product (no oracle arithmetic)."""
    cfg = _small_cfg(T=12, H=64, I=64, E=6, k=3, renorm=False, n_shared=1, I_shared=32)
    inp = mi.make_inputs(cfg)
    res = oracle.moe_layer(inp["x"], inp["Wg"], None, 3, False, inp["W1"], inp["W2"],
                           W1s=inp["W1s"], W2s=inp["W2s"], on_input=True)
    x64 = _bf16_np(inp["x"])
    shared = _numpy_mlp(x64, inp["W1s"][0], inp["W2s"][0])
    for t in range(cfg.T):
        ref = shared[t].copy()
        for j in range(3):
            e = int(res["ids"][t, j])
            xs = torch.from_numpy(res["w"][t, j] * x64[t:t + 1]).to(torch.bfloat16).to(torch.float64).numpy()
            ref += _numpy_mlp(xs, inp["W1"][e], inp["W2"][e])[0]
        np.testing.assert_allclose(res["out"][t], ref, rtol=0, atol=1e-3 * np.abs(ref).max())


def test_routing_on_input_local_ranges_sum_to_full_layer():
    cfg = _small_cfg(T=30, H=64, I=64, E=8, k=3)
    inp = mi.make_inputs(cfg)
    full = oracle.moe_layer(inp["x"], inp["Wg"], None, 3, True, inp["W1"], inp["W2"], on_input=True)
    acc = np.zeros_like(full["out"])
    for start in (0, 4):
        part = oracle.moe_layer(inp["x"], inp["Wg"], None, 3, True, inp["W1"][start:start + 4],
                                inp["W2"][start:start + 4], local_start=start, local_count=4, on_input=True)
        mod = oracle.moe_layer(inp["x"], inp["Wg"], None, 3, True, inp["W1"][start:start + 4],
                               inp["W2"][start:start + 4], local_start=start, local_count=4,
                               mode=oracle.NONLOCAL_MOD, on_input=True)
        assert np.array_equal(part["out"], mod["out"])  # a zero-weight input row gives a zero output
        acc += part["out"]
    np.testing.assert_allclose(acc, full["out"], rtol=0, atol=1e-12 * np.abs(full["out"]).max())


# --------------------------------------------------------------------------- E4M3 weights with row scales

def test_e4m3_decode_matches_torch_for_every_byte():
    q = torch.arange(256, dtype=torch.uint8)
    ref = q.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(int(b)) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_encode_matches_torch_round_to_nearest_even():
    g = torch.Generator().manual_seed(5)
    v = torch.cat([torch.randn(4000, generator=g) * s for s in (1e-3, 0.02, 1.0, 30.0, 120.0)])
    v = v.clamp(-448, 448)
    # exact midpoints between neighbouring E4M3 values, normal and subnormal
    grid = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    grid = grid[torch.isfinite(grid) & (grid >= 0)].unique().sort().values
    mids = ((grid[1:] + grid[:-1]) / 2).to(torch.float32)
    v = torch.cat([v, mids, -mids]).to(torch.float32)
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.f64_to_e4m3(float(a)) for a in v.numpy()], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_row_quantisation_bounds_and_largest_value():
    g = torch.Generator().manual_seed(6)
    w = (torch.randn(40, 96, generator=g) * 0.02).to(torch.bfloat16)
    w[3] = 0.0
    q, sc = oracle.quantize_fp8_rows(w)
    wf = w.float().numpy()
    amax = np.abs(wf).max(1)
    np.testing.assert_array_equal(sc, (amax / np.float32(448.0)).astype(np.float32))
    deq = sc[:, None].astype(np.float64) * torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    err = np.abs(deq - wf)
    # half a unit in the last place: 2^-4 relative for normal values, 2^-10 * scale below 2^-6 * scale
    bound = np.maximum(2.0 ** -4 * np.abs(wf), 2.0 ** -10 * sc[:, None]) * (1 + 1e-6)
    assert np.all(err <= bound)
    assert np.all(q[3] == 0) and sc[3] == 0.0
    for r in range(40):
        if r != 3:  # the row's largest |w| maps to +-448 exactly
            i = int(np.abs(wf[r]).argmax())
            assert abs(oracle.e4m3_to_f64(int(q[r, i]))) == 448.0


def _exact_fp8_weights(shape, gen):
    """bf16 weights that are exactly scale * e4m3 with scale = 2^-10 (each row holds +-448)."""
    grid = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)
    grid = grid[torch.isfinite(grid)]
    idx = torch.randint(0, grid.numel(), shape, generator=gen)
    w = grid[idx]
    w[..., 0] = 448.0
    return (w * 2.0 ** -10).to(torch.bfloat16)


def test_fp8_expert_and_layer_equal_bf16_when_weights_are_exact():
    g = torch.Generator().manual_seed(7)
    cfg = _small_cfg(T=20, H=64, I=64, E=5, k=2, renorm=True, n_shared=1, I_shared=64)
    inp = mi.make_inputs(cfg)
    W1 = _exact_fp8_weights((5, 128, 64), g)
    W2 = _exact_fp8_weights((5, 64, 64), g)
    W1s = _exact_fp8_weights((1, 128, 64), g)
    W2s = _exact_fp8_weights((1, 64, 64), g)
    q1, s1 = oracle.quantize_fp8_rows(W1)
    q2, s2 = oracle.quantize_fp8_rows(W2)
    q1s, s1s = oracle.quantize_fp8_rows(W1s)
    q2s, s2s = oracle.quantize_fp8_rows(W2s)
    assert np.all(s1 == 2.0 ** -10) and np.all(s2 == 2.0 ** -10)
    y8, h8 = oracle.expert_mlp_fp8(inp["x"][0], q1[2], s1[2], q2[2], s2[2])
    yb, hb = oracle.expert_mlp(inp["x"][0], W1[2], W2[2])
    assert np.array_equal(y8, yb) and np.array_equal(h8, hb)
    fp8 = dict(W1q=q1, s1=s1, W2q=q2, s2=s2, W1sq=q1s, s1s=s1s, W2sq=q2s, s2s=s2s)
    a = oracle.moe_layer(inp["x"], inp["Wg"], None, 2, True, W1, W2, W1s=W1s, W2s=W2s)
    b = oracle.moe_layer(inp["x"], inp["Wg"], None, 2, True, W1, W2, W1s=W1s, W2s=W2s, fp8=fp8)
    assert np.array_equal(a["out"], b["out"])


def test_fp8_layer_matches_numpy_mlp_of_dequantised_weights():
    cfg = _small_cfg(T=10, H=64, I=64, E=4, k=1, renorm=True)
    inp = mi.make_inputs(cfg)
    q1, s1 = oracle.quantize_fp8_rows(inp["W1"])
    q2, s2 = oracle.quantize_fp8_rows(inp["W2"])
    res = oracle.moe_layer(inp["x"], inp["Wg"], None, 1, True, inp["W1"], inp["W2"],
                           fp8=dict(W1q=q1, s1=s1, W2q=q2, s2=s2))
    deq = lambda q, s: s[..., None].astype(np.float64) * torch.from_numpy(q).view(  # noqa: E731
        torch.float8_e4m3fn).to(torch.float64).numpy()
    D1, D2 = deq(q1, s1), deq(q2, s2)
    x64 = _bf16_np(inp["x"])
    for t in range(cfg.T):
        e = int(res["ids"][t, 0])
        g = x64[t] @ D1[e][:64].T
        u = x64[t] @ D1[e][64:].T
        h = torch.from_numpy(g / (1 + np.exp(-g)) * u).to(torch.bfloat16).to(torch.float64).numpy()
        ref = h @ D2[e].T
        np.testing.assert_allclose(res["out"][t], ref, rtol=0, atol=1e-9 * np.abs(ref).max())


# --------------------------------------------------------------------------- E4M3 activations (W8A8)

def _act_exponent(amax: float) -> int:
    """Smallest e >= -126 with amax <= 448 * 2^e: a log2 guess corrected by exact compares."""
    if amax == 0.0:
        return -126
    e = max(-126, int(np.ceil(np.log2(amax / 448.0))))
    while e > -126 and amax <= 448.0 * 2.0 ** (e - 1):
        e -= 1
    while amax > 448.0 * 2.0 ** e:
        e += 1
    return e


def _quant_act_ref(v: torch.Tensor):
    """Row quantisation through torch's float8_e4m3fn cast: (q bytes, scales, dequantised fp64)."""
    v64 = v.to(torch.float64).reshape(-1, v.shape[-1]).numpy()
    qs, scs = [], []
    for row in v64:
        e = _act_exponent(float(np.abs(row).max()))
        scaled = torch.from_numpy(np.ldexp(row, -e)).to(torch.float32)
        qs.append(scaled.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
        scs.append(np.float32(2.0 ** e))
    q = np.stack(qs).reshape(v.shape)
    sc = np.array(scs, np.float32).reshape(v.shape[:-1])
    deq = sc[..., None].astype(np.float64) * torch.from_numpy(q).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()
    return q, sc, deq


def _act_rows():
    g = torch.Generator().manual_seed(11)
    rows = [torch.randn(96, generator=g) * s for s in (1e-3, 0.02, 1.0, 300.0, 1e5, 1e-30)]
    r = torch.randn(96, generator=g)
    rows.append(torch.zeros(96))                                   # all zero: e = -126, q = 0
    rows.append(r / r.abs().max() * 3584.0)                        # amax = 448 * 2^3 exactly
    rows.append(r / r.abs().max() * 3600.0)                        # the next bf16 above it
    rows.append(torch.full((96,), 2.0 ** -130) * torch.sign(r))    # bf16 subnormals: clamp at 2^-126
    return torch.stack(rows).to(torch.bfloat16)


def test_act_quantisation_matches_torch_cast_with_power_of_two_scale():
    v = _act_rows()
    q, sc = oracle.quantize_act_rows(v)
    q_ref, sc_ref, _ = _quant_act_ref(v)
    assert np.array_equal(sc, sc_ref)
    assert np.array_equal(q, q_ref)
    assert sc[6] == np.float32(2.0 ** -126) and np.all(q[6] == 0)
    assert sc[7] == 8.0 and sc[8] == 16.0 and sc[9] == np.float32(2.0 ** -126)


def test_act_quantisation_bounds_and_power_of_two_equivariance():
    v = _act_rows()
    q, sc = oracle.quantize_act_rows(v)
    vf = v.to(torch.float64).numpy()
    amax = np.abs(vf).max(1)
    for r in range(v.shape[0]):
        if sc[r] > np.float32(2.0 ** -126):
            assert 224.0 < amax[r] / float(sc[r]) <= 448.0
    deq = sc[:, None].astype(np.float64) * torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    bound = np.maximum(2.0 ** -4 * np.abs(vf), 2.0 ** -10 * sc[:, None]) * (1 + 1e-9)
    assert np.all(np.abs(deq - vf) <= bound)
    # scaling a row by 2^j (no clamp involved) leaves q alone and scales the scale
    for j in (-7, 3, 20):
        keep = [r for r in (0, 1, 2, 3, 7, 8)]
        q2, sc2 = oracle.quantize_act_rows((v[keep].to(torch.float64) * 2.0 ** j).to(torch.bfloat16))
        assert np.array_equal(q2, q[keep])
        assert np.array_equal(sc2.astype(np.float64), sc[keep].astype(np.float64) * 2.0 ** j)


def test_w8a8_layer_matches_numpy_mlp_of_quantised_rows():
    cfg = _small_cfg(T=10, H=64, I=64, E=4, k=1, renorm=True, n_shared=1, I_shared=128)
    inp = mi.make_inputs(cfg)
    q1, s1 = oracle.quantize_fp8_rows(inp["W1"])
    q2, s2 = oracle.quantize_fp8_rows(inp["W2"])
    q1s, s1s = oracle.quantize_fp8_rows(inp["W1s"])
    q2s, s2s = oracle.quantize_fp8_rows(inp["W2s"])
    fp8 = dict(W1q=q1, s1=s1, W2q=q2, s2=s2, W1sq=q1s, s1s=s1s, W2sq=q2s, s2s=s2s, act8=True)
    res = oracle.moe_layer(inp["x"], inp["Wg"], None, 1, True, inp["W1"], inp["W2"], W1s=inp["W1s"],
                           W2s=inp["W2s"], fp8=fp8)
    deq = lambda q, s: s[..., None].astype(np.float64) * torch.from_numpy(q).view(  # noqa: E731
        torch.float8_e4m3fn).to(torch.float64).numpy()
    D1, D2, D1s, D2s = deq(q1, s1), deq(q2, s2), deq(q1s, s1s)[0], deq(q2s, s2s)[0]
    _, _, xq = _quant_act_ref(inp["x"])

    def mlp(xrow, A, B):
        I = A.shape[0] // 2
        g, u = xrow @ A[:I].T, xrow @ A[I:].T
        h = torch.from_numpy(g / (1 + np.exp(-g)) * u).to(torch.bfloat16)
        return _quant_act_ref(h[None])[2][0] @ B.T

    for t in range(cfg.T):
        e = int(res["ids"][t, 0])
        ref = mlp(xq[t], D1[e], D2[e]) + mlp(xq[t], D1s, D2s)
        np.testing.assert_allclose(res["out"][t], ref, rtol=0, atol=1e-9 * np.abs(ref).max())
    # and the activations really are quantised: the weight-only result differs
    w16 = oracle.moe_layer(inp["x"], inp["Wg"], None, 1, True, inp["W1"], inp["W2"], W1s=inp["W1s"],
                           W2s=inp["W2s"], fp8={k: v for k, v in fp8.items() if k != "act8"})
    assert not np.array_equal(w16["out"], res["out"])


def test_w8a8_single_expert_with_routing_on_input_quantises_the_scaled_row():
    cfg = _small_cfg(T=6, H=64, I=64, E=3, k=2, renorm=True)
    inp = mi.make_inputs(cfg)
    q1, s1 = oracle.quantize_fp8_rows(inp["W1"])
    q2, s2 = oracle.quantize_fp8_rows(inp["W2"])
    fp8 = dict(W1q=q1, s1=s1, W2q=q2, s2=s2, act8=True)
    res = oracle.moe_layer(inp["x"], inp["Wg"], None, 2, True, inp["W1"], inp["W2"], on_input=True, fp8=fp8)
    for t in range(cfg.T):
        acc = np.zeros(cfg.H)
        for j in range(2):
            e, w = int(res["ids"][t, j]), float(res["w"][t, j])
            xs = torch.from_numpy(w * _bf16_np(inp["x"][t])).to(torch.bfloat16)
            y, _ = oracle.expert_mlp_fp8(xs, q1[e], s1[e], q2[e], s2[e], act8=True)
            acc += y
        np.testing.assert_allclose(res["out"][t], acc, rtol=0, atol=1e-12 * np.abs(acc).max())


# --------------------------------------------------------------------------- NVFP4 (E2M1 + block scales)

# E2M1 magnitudes by code (bit 0 = mantissa bit): the format's value table, written out
_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_brute(v: float) -> int:
    """Nearest E2M1 code by exhaustive search over the 8 magnitudes; a tie goes to the
    code with mantissa bit 0; beyond 6 the magnitude saturates."""
    a = abs(v)
    best = min(range(8), key=lambda c: (abs(_E2M1[c] - a), c & 1))
    return best | (8 if np.signbit(v) else 0)


def _e4m3_np(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _nvfp4_deq(q, sb, s):
    """Dequantised NVFP4 values from the value table, torch's E4M3 decode and the row scales."""
    mag = np.array(_E2M1)[q & 7] * np.where(q & 8, -1.0, 1.0)
    blk = np.repeat(_e4m3_np(sb), 16, axis=-1)
    return mag * blk * s[..., None].astype(np.float64)


def test_e2m1_decode_and_encode_match_the_value_table():
    for c in range(16):
        v = oracle.e2m1_to_f64(c)
        assert abs(v) == _E2M1[c & 7] and (np.signbit(v) == bool(c & 8))
        assert oracle.f64_to_e2m1(v) == c
    g = np.random.default_rng(11)
    mids = [(a + b) / 2 for a, b in zip(_E2M1[:-1], _E2M1[1:])]
    vals = list(g.uniform(-8, 8, 3000)) + mids + [-m for m in mids] + [6.0001, 7.0, 1e9, 1e-9, -1e-9, 0.2499]
    for v in vals:
        assert oracle.f64_to_e2m1(v) == _e2m1_brute(v), v


def _nvfp4_rows():
    g = torch.Generator().manual_seed(12)
    v = torch.randn(24, 256, generator=g)
    v[1] *= 1e-3                       # small row
    v[2, :16] *= 1e-4                  # a block far below the row's maximum
    v[3] = 0.0                         # all-zero row
    v[4] = 0.0
    v[4, 37] = -3.25                   # a single non-zero element
    v[5, 64:80] = 0.0                  # an all-zero block
    return v.to(torch.bfloat16)


def test_nvfp4_quantisation_closed_forms():
    v = _nvfp4_rows()
    q, sb, s = oracle.quantize_nvfp4_rows(v)
    assert q.shape == (24, 256) and sb.shape == (24, 16) and s.shape == (24,)
    # the zero row: scale 0, zero codes and block scales
    assert s[3] == 0.0 and np.all(q[3] == 0) and np.all(sb[3] == 0)
    # a single non-zero element: its block scale is 448, its code -6, its value the element
    assert _e4m3_np(sb[4, 2:3])[0] == 448.0 and q[4, 37] == (8 | 7)
    assert np.all(q[4, np.arange(256) != 37] == 0)
    assert np.all(sb[4, np.arange(16) != 2] == 0)
    deq = _nvfp4_deq(q, sb, s)
    assert abs(deq[4, 37] - (-3.25)) <= 2.0 ** -21 * 3.25
    # an all-zero block: scale 0, codes 0
    assert sb[5, 4] == 0 and np.all(q[5, 64:80] == 0)
    # every non-zero row: its largest |v| has magnitude code 6 (value 6) in a block of scale 448
    vf = v.float().numpy()
    for r in range(24):
        if r == 3:
            continue
        i = int(np.abs(vf[r]).argmax())
        assert (q[r, i] & 7) == 7 and _e4m3_np(sb[r, i // 16:i // 16 + 1])[0] == 448.0


def test_nvfp4_values_are_exact_for_representable_rows():
    # rows built as e2m1 * sb * s with E4M3 block scales whose block maxima are 6 * sb:
    # the quantiser must give back exactly these codes and scales
    g = np.random.default_rng(13)
    grid_sb = _e4m3_np(np.arange(0x30, 0x7F, dtype=np.uint8))    # block scales 2^-3 .. 448
    for trial in range(20):
        s = 2.0 ** int(g.integers(-20, -8))                         # the row scale, a power of two
        sbv = g.choice(grid_sb, 8)
        sbv[int(g.integers(0, 8))] = 448.0                         # one block carries the row maximum
        codes = g.integers(0, 16, (8, 16))
        codes[:, 0] = 7 | (8 * g.integers(0, 2, 8))                # each block holds +-6
        vals = np.array(_E2M1)[codes & 7] * np.where(codes & 8, -1.0, 1.0) * sbv[:, None] * s
        row = torch.from_numpy(vals.reshape(1, -1)).to(torch.bfloat16)
        assert np.array_equal(row.to(torch.float64).numpy().reshape(8, 16), vals)  # bf16-exact
        q, sb, sc = oracle.quantize_nvfp4_rows(row)
        # s = amax / 2688 with amax = 6 * 448 * s exactly
        assert sc[0] == np.float32(s)
        np.testing.assert_array_equal(_e4m3_np(sb[0]), sbv)
        deq = _nvfp4_deq(q, sb, sc)
        np.testing.assert_array_equal(deq.reshape(8, 16), vals)


def test_nvfp4_bounds_and_power_of_two_equivariance():
    v = _nvfp4_rows()
    q, sb, s = oracle.quantize_nvfp4_rows(v)
    vf = v.to(torch.float64).numpy()
    deq = _nvfp4_deq(q, sb, s)
    blk = np.repeat(_e4m3_np(sb), 16, axis=-1) * s[:, None].astype(np.float64)
    live = blk > 0
    # each element: within half an E2M1 step of its scaled value (the step is 0.5 below 2,
    # 1 below 4, 2 up to 6), or saturated at 6 block units
    t = np.where(live, np.abs(vf) / np.where(live, blk, 1.0), 0.0)
    half = np.where(t < 2.0, 0.25, np.where(t < 4.0, 0.5, 1.0))
    bound = np.where(t <= 6.0, half, t - 6.0) * blk * (1 + 1e-6) + 1e-300
    assert np.all(np.abs(deq - vf)[live] <= bound[live])
    # blocks whose scale rounds to zero hold zeros only
    assert np.all(deq[~live] == 0.0)
    # scaling a row by 2^j scales s by 2^j and keeps every code and block scale
    for j in (-7, -1, 3, 9):
        q2, sb2, s2 = oracle.quantize_nvfp4_rows((v.float() * 2.0 ** j).to(torch.bfloat16))
        keep = np.arange(24) != 3
        assert np.array_equal(q2, q) and np.array_equal(sb2, sb)
        np.testing.assert_array_equal(s2[keep], (s[keep].astype(np.float64) * 2.0 ** j).astype(np.float32))


def test_nvfp4_expert_mlp_matches_numpy_of_dequantised_values():
    cfg = _small_cfg(T=6, H=64, I=64, E=1, k=1, renorm=True)
    inp = mi.make_inputs(cfg)
    q1, sb1, s1 = oracle.quantize_nvfp4_rows(inp["W1"][0])
    q2, sb2, s2 = oracle.quantize_nvfp4_rows(inp["W2"][0])
    D1, D2 = _nvfp4_deq(q1, sb1, s1), _nvfp4_deq(q2, sb2, s2)
    for t in range(cfg.T):
        xrow = inp["x"][t]
        for act4 in (False, True):
            y, h = oracle.expert_mlp_nvfp4(xrow, q1, sb1, s1, q2, sb2, s2, act4=act4)
            if act4:
                xq, xsb, xs = oracle.quantize_nvfp4_rows(xrow[None], pow2=True)
                x64 = _nvfp4_deq(xq, xsb, xs)[0]
            else:
                x64 = _bf16_np(xrow)
            g = x64 @ D1[:64].T
            u = x64 @ D1[64:].T
            hb = torch.from_numpy(g / (1 + np.exp(-g)) * u).to(torch.bfloat16)
            assert np.array_equal(h, hb.view(torch.int16).numpy().view(np.uint16))
            if act4:
                hq, hsb, hs = oracle.quantize_nvfp4_rows(hb[None], pow2=True)
                h64 = _nvfp4_deq(hq, hsb, hs)[0]
            else:
                h64 = hb.to(torch.float64).numpy()
            ref = h64 @ D2.T
            np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12 * np.abs(ref).max())


def test_nvfp4_power_of_two_row_scale_for_activations():
    v = _nvfp4_rows()
    q, sb, s = oracle.quantize_nvfp4_rows(v, pow2=True)
    vf = np.abs(v.to(torch.float64).numpy())
    for r in range(24):
        amax = vf[r].max()
        # the smallest e >= -126 with amax <= 2688 * 2^e, by exact comparisons
        e = -126
        while amax > 2688.0 * 2.0 ** e:
            e += 1
        assert s[r] == np.float32(2.0 ** e)
        if amax > 0:
            assert amax > 2688.0 * 2.0 ** (e - 1) or e == -126
    deq = _nvfp4_deq(q, sb, s)
    blk = np.repeat(_e4m3_np(sb), 16, axis=-1) * s[:, None].astype(np.float64)
    live = blk > 0
    t = np.where(live, vf / np.where(live, blk, 1.0), 0.0)
    half = np.where(t < 2.0, 0.25, np.where(t < 4.0, 0.5, 1.0))
    bound = np.where(t <= 6.0, half, t - 6.0) * blk * (1 + 1e-6)
    vs = v.to(torch.float64).numpy()
    assert np.all(np.abs(deq - vs)[live] <= bound[live] + 1e-300)
    # with a power-of-two row scale, rows equal up to a power of two give the same codes
    q2, sb2, s2 = oracle.quantize_nvfp4_rows((v.float() * 2.0 ** 5).to(torch.bfloat16), pow2=True)
    assert np.array_equal(q2, q) and np.array_equal(sb2, sb)


def _exact_nvfp4_rows(n_rows, K, gen):
    """bf16 rows that are exactly e2m1 * sb * s with s = 2^-12, E4M3 block scales, and a
    +-6 in every block (so each block's scale and the row's largest block, 448, come back)."""
    grid_sb = _e4m3_np(np.arange(0x30, 0x7F, dtype=np.uint8))
    sbv = gen.choice(grid_sb, (n_rows, K // 16))
    sbv[:, 0] = 448.0
    codes = gen.integers(0, 16, (n_rows, K // 16, 16))
    codes[..., 0] = 7 | (8 * gen.integers(0, 2, (n_rows, K // 16)))
    vals = np.array(_E2M1)[codes & 7] * np.where(codes & 8, -1.0, 1.0) * sbv[..., None] * 2.0 ** -12
    return torch.from_numpy(vals.reshape(n_rows, K)).to(torch.bfloat16)


def _nvfp4_dict(W1, W2, W1s=None, W2s=None, act4=False):
    d = {}
    d["W1q"], d["W1sb"], d["s1"] = oracle.quantize_nvfp4_rows(W1)
    d["W2q"], d["W2sb"], d["s2"] = oracle.quantize_nvfp4_rows(W2)
    if W1s is not None:
        d["W1sq"], d["W1ssb"], d["s1s"] = oracle.quantize_nvfp4_rows(W1s)
        d["W2sq"], d["W2ssb"], d["s2s"] = oracle.quantize_nvfp4_rows(W2s)
    d["act4"] = act4
    return d


def test_nvfp4_layer_equals_bf16_when_weights_are_exact():
    g = np.random.default_rng(14)
    cfg = _small_cfg(T=20, H=64, I=64, E=5, k=2, renorm=True, n_shared=1, I_shared=64)
    inp = mi.make_inputs(cfg)
    W1 = _exact_nvfp4_rows(5 * 128, 64, g).reshape(5, 128, 64)
    W2 = _exact_nvfp4_rows(5 * 64, 64, g).reshape(5, 64, 64)
    W1s = _exact_nvfp4_rows(128, 64, g)[None]
    W2s = _exact_nvfp4_rows(64, 64, g)[None]
    d = _nvfp4_dict(W1, W2, W1s, W2s)
    assert np.all(d["s1"] == np.float32(2.0 ** -12)) and np.all(d["s2"] == np.float32(2.0 ** -12))
    y4, h4 = oracle.expert_mlp_nvfp4(inp["x"][0], d["W1q"][2], d["W1sb"][2], d["s1"][2], d["W2q"][2],
                                     d["W2sb"][2], d["s2"][2])
    yb, hb = oracle.expert_mlp(inp["x"][0], W1[2], W2[2])
    assert np.array_equal(y4, yb) and np.array_equal(h4, hb)
    a = oracle.moe_layer(inp["x"], inp["Wg"], None, 2, True, W1, W2, W1s=W1s, W2s=W2s)
    b = oracle.moe_layer(inp["x"], inp["Wg"], None, 2, True, W1, W2, W1s=W1s, W2s=W2s, nvfp4=d)
    assert np.array_equal(a["out"], b["out"])


def test_nvfp4_layer_matches_numpy_mlp_of_dequantised_values():
    cfg = _small_cfg(T=8, H=64, I=64, E=4, k=1, renorm=True, n_shared=1, I_shared=64)
    inp = mi.make_inputs(cfg)
    for act4 in (False, True):
        d = _nvfp4_dict(inp["W1"], inp["W2"], inp["W1s"], inp["W2s"], act4=act4)
        res = oracle.moe_layer(inp["x"], inp["Wg"], None, 1, True, inp["W1"], inp["W2"], W1s=inp["W1s"],
                               W2s=inp["W2s"], nvfp4=d)
        D1, D2 = _nvfp4_deq(d["W1q"], d["W1sb"], d["s1"]), _nvfp4_deq(d["W2q"], d["W2sb"], d["s2"])
        S1, S2 = _nvfp4_deq(d["W1sq"], d["W1ssb"], d["s1s"])[0], _nvfp4_deq(d["W2sq"], d["W2ssb"], d["s2s"])[0]

        def act(row_bf16):
            if not act4:
                return row_bf16.to(torch.float64).numpy()
            q, sb, s = oracle.quantize_nvfp4_rows(row_bf16[None], pow2=True)
            return _nvfp4_deq(q, sb, s)[0]

        def mlp(xr, A, B):
            x64 = act(xr)
            gt, up = x64 @ A[:64].T, x64 @ A[64:].T
            h = torch.from_numpy(gt / (1 + np.exp(-gt)) * up).to(torch.bfloat16)
            return act(h) @ B.T

        for t in range(cfg.T):
            e = int(res["ids"][t, 0])
            ref = mlp(inp["x"][t], D1[e], D2[e]) + mlp(inp["x"][t], S1, S2)
            np.testing.assert_allclose(res["out"][t], ref, rtol=0, atol=1e-9 * np.abs(ref).max())


# --------------------------------------------------------------------------- all-to-all receive order

def _a2a_golden_cases():
    cases, cur = [], None
    for ln in _read_golden("a2a_regroup_example.txt"):
        key, *vals = ln.split()
        if key == "case":
            cur = dict(N=int(vals[0]), S=int(vals[1]))
            cases.append(cur)
        else:
            cur[key] = [int(v) for v in vals]
    return cases


def test_a2a_regroup_golden_examples():
    cases = _a2a_golden_cases()
    assert len(cases) == 3
    for c in cases:
        counts = np.array(c["counts"], np.int32).reshape(c["N"], c["S"])
        offsets, gemm_row, exch_row = oracle.a2a_regroup(counts)
        assert offsets.tolist() == c["offsets"]
        assert gemm_row.tolist() == c["gemm_row"]
        assert exch_row.tolist() == np.argsort(np.array(c["gemm_row"], np.int64)).tolist()


@pytest.mark.parametrize("N,S_l,seed", [(2, 5, 0), (4, 3, 1), (8, 36, 2), (3, 1, 3), (1, 7, 4)])
def test_a2a_regroup_invariants(N, S_l, seed):
    g = torch.Generator().manual_seed(seed)
    counts = torch.randint(0, 6, (N, S_l), generator=g).numpy().astype(np.int32)
    counts[0, 0] = 0  # an empty block
    offsets, gemm_row, exch_row = oracle.a2a_regroup(counts)
    R = int(counts.sum())
    # a bijection of the R received rows
    assert sorted(gemm_row.tolist()) == list(range(R))
    assert np.array_equal(exch_row[gemm_row], np.arange(R))
    # slot c holds the column sum of its counts, contiguously from offsets[c]
    assert np.array_equal(np.diff(offsets), counts.sum(0))
    # walk the arrival order: block (n, c) lands inside slot c, after the blocks of
    # sources n' < n for that slot, its rows in arrival order
    q = 0
    for n in range(N):
        for c in range(S_l):
            base = offsets[c] + counts[:n, c].sum()
            for i in range(counts[n, c]):
                assert gemm_row[q] == base + i
                q += 1
    assert q == R
    # N = 1: arrival order is already grouped by slot (the identity)
    if N == 1:
        assert np.array_equal(gemm_row, np.arange(R))


def test_a2a_regroup_rejects_negative_counts():
    with pytest.raises(ValueError):
        oracle.a2a_regroup(np.array([[1, -1]], np.int32))
