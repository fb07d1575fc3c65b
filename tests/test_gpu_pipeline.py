"""HostPipeline: batches whose host<->device copies overlap the neighbouring
batches' forwards must give, bit for bit, the outputs of one forward per batch
(serial copies, one stream), over several distinct batches and across calls."""
import pytest
import torch

import moe_inputs as mi
import serving_router_gate_gb300 as moe
from serving_router_gate_gb300.layer import HostPipeline, layer_from_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", ["bf16", "w8a8", "nvfp4"])
def test_host_pipeline_equals_one_forward_per_batch(fmt):
    extra = dict(fp8=True, act8=True) if fmt == "w8a8" else (dict(fp4=True) if fmt == "nvfp4" else {})
    cfg = mi.MoEConfig(f"pipe_{fmt}", T=300, H=256, I=256, E=8, k=2, renorm=True, n_shared=1, I_shared=256,
                       shared_gate=True, **extra)
    inp = mi.make_inputs(cfg)
    layer = layer_from_inputs(inp, "cuda")
    x = inp["x"]
    # distinct batches: the rows rotated and rescaled, so routing and outputs differ per batch
    xs = [(torch.roll(x.float(), 37 * i, 0) * (1.0 + 0.25 * i)).to(torch.bfloat16) for i in range(5)]
    want = [layer.forward(xi.cuda()).clone().cpu() for xi in xs]
    pipe = HostPipeline(layer, xs[0])
    xs_pin = [xi.pin_memory() for xi in xs]
    outs = [torch.empty_like(xi).pin_memory() for xi in xs]
    pipe.run(xs_pin, outs)
    torch.cuda.synchronize()
    for i, (w, o) in enumerate(zip(want, outs)):
        assert torch.equal(w.view(torch.int16), o.view(torch.int16)), f"batch {i}"
    # a second call continues with the other buffer pair first
    outs2 = [torch.empty_like(xi).pin_memory() for xi in xs[:3]]
    pipe.run(xs_pin[2:5], outs2)
    torch.cuda.synchronize()
    for i, o in enumerate(outs2):
        assert torch.equal(want[2 + i].view(torch.int16), o.view(torch.int16)), f"second call, batch {i}"
    assert moe.moe_get_device_status(layer.ws) == 0
