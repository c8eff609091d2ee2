"""Small-batch decode of an MXFP8 layer (warp-per-output kernels on E4M3 weights, and from the
crossover batch the grouped-GEMM forward).

Decode is the MXFP8 layer forward on B tokens: x quantised along d, the
weights along each product's K, h along f. Checked against the oracle's
MXFP8 forward (relative Frobenius error <= 3e-2, the MXFP8 tolerance) with the
GPU's fp32 router logits on both sides, against the GPU's own MXFP8 forward on
the same B tokens, and for bit-identical reruns.
"""
import numpy as np
import pytest
import torch

import moe_synth
from mixture_experts_layer_routing_gb300 import MoeLayer
from oracle import moe_oracle as oracle

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
TOL_MX = 3e-2
SPEC = moe_synth.LayerSpec("mxfp8_decode_d512_E16+1_f256_top4_sigmoid", 64, 512, 16, 1, 256, 4, "sigmoid", True, 2.5,
                           "mxfp8", None, 71)


def np64(t):
    return t.detach().double().cpu().numpy()


@pytest.fixture(scope="module")
def layer_and_inputs():
    inp = moe_synth.make_inputs(SPEC, "cpu")
    g = {k: v.to(DEV) for k, v in inp.items()}
    layer = MoeLayer.from_spec(SPEC, device=DEV)
    layer.set_weights(g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    yield layer, g, {k: np64(v) for k, v in inp.items()}
    layer.close()


@pytest.mark.parametrize("path", ["warp", "crossover"])
@pytest.mark.parametrize("B", [1, 3, 16, 64])
def test_mx_decode_parity(layer_and_inputs, B, path):
    """path "warp": the warp-per-output kernels at every B; "crossover": the MXFP8 default, where
    moe_decode takes the grouped-GEMM forward from B = 4 (then equal to moe_forward bit for bit)."""
    from mixture_experts_layer_routing_gb300 import moe_set_decode_crossover
    layer, g, n = layer_and_inputs
    moe_set_decode_crossover(layer.h, 65 if path == "warp" else 4)
    x = g["x"][:B].contiguous()
    y = layer.decode(x)
    if path == "crossover" and B >= 4:
        assert torch.equal(y, layer.forward(x))
    y2 = layer.decode(x)
    logits = layer.route(x)["logits"].cpu().numpy()
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(y, y2)
    kw = dict(k=SPEC.k, router=SPEC.router, renorm=SPEC.renorm, scale=SPEC.route_scale, n_shared=SPEC.S)
    ref = oracle.decode(n["x"][:B], n["Wr"], n["b"], n["Wg"], n["Wu"], n["Wd"], logits32=logits, mx=True, **kw)["y"]
    err = oracle.rel_frobenius(np64(y), ref)
    assert err <= TOL_MX, err
    # the GPU's MXFP8 forward on the same tokens computes the same function
    yf = layer.forward(x)
    torch.cuda.synchronize()
    assert oracle.rel_frobenius(np64(y), np64(yf)) <= TOL_MX
