"""Device-side failure path on the GPU, without faulting it.

A wait that can never be satisfied (an mbarrier nothing arrives at, with the
same bounded wait the tcgen05 pipelines use) must give up after its limit,
report MOE_ERR_TIMEOUT through the status word, and leave the context usable.
"""
import pytest
import torch

import moe_synth
import mixture_experts_layer_routing_gb300 as moe

pytestmark = pytest.mark.gpu


def test_wait_timeout_reported_and_context_survives():
    dev = torch.device("cuda:0")
    spec = moe_synth.LayerSpec("bf16_T128_d256_E8_f128_top2", 128, 256, 8, 0, 128, 2, "softmax", True, 1.0, "bf16",
                               None, 51)
    inp = {k: v.to(dev) for k, v in moe_synth.make_inputs(spec, "cpu").items()}
    layer = moe.MoeLayer.from_spec(spec, device=dev)
    layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
    y0 = layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    moe.moe_selftest_timeout(layer.h, 200)
    assert layer.status() == moe.MOE_ERR_TIMEOUT
    assert layer.status() == moe.MOE_OK                  # reading clears the word
    y1 = layer.forward(inp["x"])                          # the context still works
    torch.cuda.synchronize()
    assert layer.status() == moe.MOE_OK
    assert torch.equal(y0, y1)
    layer.close()
