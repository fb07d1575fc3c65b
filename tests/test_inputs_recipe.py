"""The seeded input recipe (moe_inputs) on CPU: inputs are reproducible, the slot table
is a valid replica map, the Zipf bias follows the hotness ranking, and the shared experts'
concatenated layout computes the same MLP as the experts summed."""
import numpy as np
import torch

import moe_inputs as mi
import oracle


def test_inputs_are_reproducible_and_seed_dependent():
    cfg = mi.MoEConfig("rep", T=33, H=64, I=64, E=10, S=13, n_hot=3, zipf_s=1.1, k=3, renorm=True,
                       n_shared=2, I_shared=64, shared_gate=True)
    a, b = mi.make_inputs(cfg), mi.make_inputs(cfg)
    for key in ("x", "Wg", "bias", "W1", "W2", "W1s", "W2s", "w_s", "rep_offset", "rep_slots"):
        assert torch.equal(a[key], b[key]), key
    c = mi.make_inputs(cfg.with_(seed=1))
    assert not torch.equal(a["x"], c["x"]) and not torch.equal(a["W1"], c["W1"])


def test_slot_table_is_a_valid_replica_map():
    cfg = mi.MoEConfig("tab", T=8, H=64, I=64, E=40, S=52, n_hot=12, zipf_s=1.1, k=4, renorm=True)
    tab = mi.slot_table(cfg)
    ro, rs, eos, rank = (tab[k].numpy() for k in ("rep_offset", "rep_slots", "expert_of_slot", "rank"))
    # every slot is used exactly once
    assert sorted(rs.tolist()) == list(range(cfg.slots))
    counts = np.diff(ro)
    # the n_hot hottest experts (rank 1..n_hot) have two slots, the others one
    assert np.array_equal(counts, np.where(rank <= cfg.n_hot, 2, 1))
    # each expert's slots hold that expert
    for e in range(cfg.E):
        assert all(eos[s] == e for s in rs[ro[e]:ro[e + 1]])
    # the bias is -s ln(rank): the hottest expert has bias 0 and biases fall with rank
    bias = tab["bias"].numpy().astype(np.float64)
    np.testing.assert_allclose(bias, -1.1 * np.log(rank), rtol=1e-6)
    assert bias[rank == 1][0] == 0.0
    assert np.all(np.diff(bias[np.argsort(rank)]) < 0)


def test_replica_slots_hold_copies_of_their_expert_weights():
    cfg = mi.MoEConfig("copies", T=8, H=64, I=64, E=6, S=8, n_hot=2, k=2, renorm=True)
    inp = mi.make_inputs(cfg)
    ident = mi.make_inputs(cfg.with_(S=None, n_hot=0))
    eos = inp["expert_of_slot"].numpy()
    for s in range(cfg.slots):
        assert torch.equal(inp["W1"][s], ident["W1"][eos[s]]) and torch.equal(inp["W2"][s], ident["W2"][eos[s]])


def test_shared_concat_equals_the_sum_of_the_shared_experts():
    cfg = mi.MoEConfig("sh", T=4, H=64, I=64, E=2, k=1, renorm=True, n_shared=3, I_shared=32)
    inp = mi.make_inputs(cfg)
    W1c, W2c = mi.shared_concat(inp["W1s"], inp["W2s"])
    for t in range(cfg.T):
        ysum = sum(oracle.expert_mlp(inp["x"][t], inp["W1s"][i], inp["W2s"][i])[0] for i in range(3))
        yc, _ = oracle.expert_mlp(inp["x"][t], W1c, W2c)
        np.testing.assert_allclose(yc, ysum, rtol=0, atol=1e-12 * np.abs(ysum).max())
