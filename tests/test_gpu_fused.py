"""The forward as one persistent kernel.

moe_set_fused(h, 1): the two expert GEMMs (gate/up and down tiles) in a single
cooperative launch, down tiles released by per-row-block arrival counters.
moe_set_fused(h, 2): the whole forward in one cooperative launch: the router
GEMM (the same K splits), top-k, histogram, scan, permutation, the expert
tiles taken from a device tile queue, and the combine, separated by bounded
grid-wide barriers.

The fused kernels run the same tiles with the same K order as the separate
launches, so:

* y is bit-identical to the unfused forward, and so are the saved activations
  (checked through the backward, whose dx and weight gradients must match
  bit for bit), on cases with a shared expert, a Zipf-like selection bias
  (hot experts with many tiles, cold ones with none), ragged last tiles and
  T = 1;
* against the float64 oracle it is within the bf16 tolerance (5e-3);
* repeated calls (the counters are reset by the kernel's last CTA) and a CUDA
  graph replay on new inputs give the eager results.
"""
import numpy as np
import pytest
import torch

import moe_synth
from mixture_experts_layer_routing_gb300 import MoeLayer, moe_forward, moe_set_fused
from oracle import moe_oracle as oracle

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

CASES = [
    (moe_synth.LayerSpec("bf16_T1000_d512_E16+1_f256_top5_sigmoid", 1000, 512, 16, 1, 256, 5, "sigmoid", True, 2.5,
                         "bf16", None, 91), None),
    (moe_synth.LayerSpec("bf16_T1500_d512_E32_f384_top4_softmax_skewed", 1500, 512, 32, 0, 384, 4, "softmax", True,
                         1.0, "bf16", None, 92), np.linspace(4.0, -4.0, 32)),
    (moe_synth.LayerSpec("bf16_T1_d256_E8+1_f128_top2_softmax", 1, 256, 8, 1, 128, 2, "softmax", True, 1.0, "bf16",
                         None, 93), None),
]


def np64(t):
    return t.detach().double().cpu().numpy()


def make(spec, bias):
    inp = moe_synth.make_inputs(spec, DEV, grad=True)
    if bias is not None:
        inp["b"] = torch.as_tensor(bias, dtype=torch.float32, device=DEV)
    layer = MoeLayer.from_spec(spec, device=DEV)
    layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
    return inp, layer


def step(layer, inp, fused):
    moe_set_fused(layer.h, fused)
    ctx = layer.new_ctx(inp["x"].shape[0])
    y = layer.forward(inp["x"], ctx=ctx)
    grads = layer.backward(inp["x"], inp["dy"], ctx)
    torch.cuda.synchronize()
    assert layer.status() == 0
    return {"y": y.clone(), **{k: v.clone() for k, v in grads.items()}}


@pytest.mark.parametrize("mode", [1, 2], ids=["experts", "whole_forward"])
@pytest.mark.parametrize("spec,bias", CASES, ids=[c[0].name for c in CASES])
def test_fused_matches_separate_launches(spec, bias, mode):
    inp, layer = make(spec, bias)
    sep = step(layer, inp, 0)
    fus = step(layer, inp, mode)
    fus2 = step(layer, inp, mode)
    for k in sep:
        assert torch.equal(fus[k], sep[k]), k
        assert torch.equal(fus2[k], sep[k]), k
    # inference forward (no saved activations) as well
    moe_set_fused(layer.h, mode)
    y_inf = layer.forward(inp["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(y_inf, sep["y"])
    r = layer.route(inp["x"])
    n = {k: np64(inp[k]) for k in ("x", "Wr", "b", "Wg", "Wu", "Wd")}
    y_ref = oracle.forward(n["x"], n["Wr"], n["b"], n["Wg"], n["Wu"], n["Wd"], k=spec.k, router=spec.router,
                           renorm=spec.renorm, scale=spec.route_scale, n_shared=spec.S,
                           logits32=r["logits"].cpu().numpy())["y"]
    assert oracle.rel_frobenius(np64(fus["y"]), y_ref) <= 5e-3
    if bias is not None:
        tiles = (r["cnt"].cpu().numpy() + 127) // 128
        assert (tiles == 0).any() and (tiles >= 3).any()
    layer.close()


@pytest.mark.parametrize("mode", [1, 2], ids=["experts", "whole_forward"])
def test_fused_many_calls_and_graph_replay(mode):
    spec, bias = CASES[0]
    inp, layer = make(spec, bias)
    T = spec.T
    x = inp["x"].clone()
    y = torch.empty_like(x)
    ws = layer.buffer("fwd", layer.sizes(T)["fwd_ws"])
    moe_set_fused(layer.h, 0)
    refs = []
    toks = [moe_synth.make_tokens(spec, 1, DEV, seed_offset=20 + i)[0] for i in range(4)]
    for t in toks:
        refs.append(layer.forward(t).clone())
    moe_set_fused(layer.h, mode)
    for _ in range(2):
        for t, ref in zip(toks, refs):
            assert torch.equal(layer.forward(t), ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe_forward(layer.h, x, T, y, None, ws)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        moe_forward(layer.h, x, T, y, None, ws)
    for t, ref in zip(toks, refs):
        x.copy_(t)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, ref)
    assert layer.status() == 0
    layer.close()


def test_fused_unsupported_layers():
    fp32 = moe_synth.LayerSpec("fp32_T8_d64_E4_f64_top2", 8, 64, 4, 0, 64, 2, "softmax", True, 1.0, "fp32", None, 94)
    layer = MoeLayer.from_spec(fp32, device=DEV)
    with pytest.raises(Exception):
        moe_set_fused(layer.h, 1)
    moe_set_fused(layer.h, 0)
    with pytest.raises(Exception):
        moe_set_fused(layer.h, 2)
    layer.close()
