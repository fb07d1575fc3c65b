"""The GPU side of expert parallelism on one GPU: each rank's partial output
(its slot range under SKIP and its shard of the shared experts, through the
same library calls a rank runs) is computed in turn, and the partials summed
on the host equal the full layer -- against the fp64 oracle and against the
one-GPU layer, within the output tolerance.  Ranks run one after another on
one GPU: nothing waits on another rank."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import serving_router_gate_gb300 as moe
from serving_router_gate_gb300.expert_parallel import EPMoELayer
from serving_router_gate_gb300.layer import layer_from_inputs

from parity_util import check_out, oracle_layer, oracle_threads, to_cpu

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
