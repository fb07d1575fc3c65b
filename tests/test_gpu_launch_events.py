"""The per-launch timing hook (moe_launch_events_arm / _mark / _used) on the GPU:
labels follow the forward's launches, recorded events give positive intervals
eagerly and from a captured graph, arming with fewer events than launches stops
recording, disarming forgets them, and the hooked forward (launched without
programmatic overlap) gives bitwise the output of the plain one."""
import pytest
import torch

import moe_inputs as mi
import serving_router_gate_gb300 as moe
from serving_router_gate_gb300.layer import layer_from_inputs

pytestmark = pytest.mark.gpu

CFG = mi.MoEConfig("hook", T=300, H=256, I=192, E=8, k=2, renorm=True, n_shared=1, I_shared=128)


def _layer():
    inp = mi.make_inputs(CFG)
    layer = layer_from_inputs(inp, device="cuda")
    x = inp["x"].cuda()
    layer.forward(x)
    torch.cuda.synchronize()
    return layer, x


def _events(n, stream):
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record(stream)
    torch.cuda.synchronize()
    return evs


def _check_labels(labels, n):
    assert len(labels) == n + 1 and labels[-1] == "mark", labels
    assert labels[0] == "router_logits" and labels[1] == "router_select", labels
    assert any(lab.startswith("permute_") for lab in labels), labels
    fc1 = [i for i, lab in enumerate(labels) if lab.startswith("grouped_gemm_fc1")]
    fc2 = [i for i, lab in enumerate(labels) if lab.startswith("grouped_gemm_fc2")]
    assert len(fc1) == 1 and len(fc2) == 1 and fc1[0] < fc2[0], labels
    assert labels[-2] == "finalize", labels


def test_eager_labels_intervals_and_bitwise_output():
    layer, x = _layer()
    ref = layer.forward(x).clone()
    c0 = moe.moe_get_launch_count()
    layer.forward(x)
    n = moe.moe_get_launch_count() - c0
    stream = torch.cuda.current_stream()
    evs = _events(n + 1, stream)
    moe.moe_launch_events_arm(evs)
    try:
        out = layer.forward(x).clone()
        moe.moe_launch_events_mark()
        labels = moe.moe_launch_events_used()
    finally:
        moe.moe_launch_events_arm(None)
    torch.cuda.synchronize()
    _check_labels(labels, n)
    for i in range(n):
        assert evs[i].elapsed_time(evs[i + 1]) > 0.0
    assert torch.equal(out, ref)
    assert moe.moe_launch_events_used() == []
    assert moe.moe_get_device_status(layer.ws) == 0


def test_captured_graph_rerecords_events_on_replay():
    layer, x = _layer()
    ref = layer.forward(x).clone()
    c0 = moe.moe_get_launch_count()
    layer.forward(x)
    n = moe.moe_get_launch_count() - c0
    evs = _events(n + 1, torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    moe.moe_launch_events_arm(evs)
    try:
        with torch.cuda.graph(g):
            layer.forward(x)
            moe.moe_launch_events_mark()
        labels = moe.moe_launch_events_used()
    finally:
        moe.moe_launch_events_arm(None)
    _check_labels(labels, n)
    for _ in range(2):
        layer.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        total = sum(evs[i].elapsed_time(evs[i + 1]) for i in range(n))
        assert total > 0.0
        assert all(evs[i].elapsed_time(evs[i + 1]) > 0.0 for i in range(n))
        assert torch.equal(layer.out[:CFG.T], ref)
    assert moe.moe_get_device_status(layer.ws) == 0


def test_fewer_events_than_launches_and_argument_checks():
    layer, x = _layer()
    evs = _events(2, torch.cuda.current_stream())
    moe.moe_launch_events_arm(evs)
    try:
        layer.forward(x)
        moe.moe_launch_events_mark()
        labels = moe.moe_launch_events_used()
    finally:
        moe.moe_launch_events_arm(None)
    torch.cuda.synchronize()
    assert labels == ["router_logits", "router_select"]
    assert evs[0].elapsed_time(evs[1]) > 0.0
    with pytest.raises(ValueError):
        moe.moe_launch_events_arm([torch.cuda.Event(enable_timing=True)])  # never recorded: no CUDA event yet
    with pytest.raises(moe.MoEError):
        moe._check("moe_launch_events_arm", moe._lib.moe_launch_events_arm(None, 3))
    assert moe.moe_launch_events_used() == []
