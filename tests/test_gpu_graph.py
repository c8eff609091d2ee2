"""The layer's calls inside a CUDA graph.

Every compute call only enqueues work on the caller's stream (no host
synchronisation, no allocation), so a training step (forward + backward) and
a decode step can be captured once and replayed: a replay on new input
values must give bit-identical results to the same calls run eagerly.
"""
import pytest
import torch

import moe_synth
from mixture_experts_layer_routing_gb300 import MoeLayer, moe_backward, moe_decode, moe_forward

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
SPEC = moe_synth.LayerSpec("bf16_T256_d512_E16+1_f256_top4_sigmoid", 256, 512, 16, 1, 256, 4, "sigmoid", True, 2.5,
                           "bf16", None, 81)


def test_train_step_graph_replay_matches_eager():
    inp = moe_synth.make_inputs(SPEC, DEV, grad=True)
    layer = MoeLayer.from_spec(SPEC, device=DEV)
    layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
    T = SPEC.T
    x = inp["x"].clone()
    dy = inp["dy"].clone()
    y = torch.empty_like(x)
    ctx = layer.new_ctx(T)
    g = layer.grads_like(x)
    sz = layer.sizes(T)
    ws = layer.buffer("fwd", sz["fwd_ws"])
    bws = layer.buffer("bwd", sz["bwd_ws"])

    def step():
        moe_forward(layer.h, x, T, y, ctx, ws)
        moe_backward(layer.h, x, dy, T, ctx, g["dx"], g["dWr"], g["dWg"], g["dWu"], g["dWd"], bws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    new = moe_synth.make_tokens(SPEC, 2, DEV, seed_offset=5)
    x.copy_(new[0])
    dy.copy_(new[1])
    graph.replay()
    torch.cuda.synchronize()
    got = {"y": y.clone(), **{k: v.clone() for k, v in g.items()}}
    step()                                       # eager, same inputs
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(got["y"], y)
    for k, v in g.items():
        assert torch.equal(got[k], v), k
    layer.close()


def test_decode_graph_replay_matches_eager():
    inp = moe_synth.make_inputs(SPEC, DEV)
    layer = MoeLayer.from_spec(SPEC, device=DEV)
    layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
    B = 4
    x = inp["x"][:B].clone()
    y = torch.empty_like(x)
    ws = layer.buffer("fwd", layer.sizes(B)["fwd_ws"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe_decode(layer.h, x, B, y, ws)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        moe_decode(layer.h, x, B, y, ws)
    x.copy_(inp["x"][B:2 * B])
    graph.replay()
    torch.cuda.synchronize()
    got = y.clone()
    moe_decode(layer.h, x, B, y, ws)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(got, y)
    layer.close()


@pytest.mark.parametrize("prec", ["bf16", "mxfp8"])
def test_chunked_step_graph_replay_matches_eager(prec):
    """The chunked training step forks the next chunk's routing onto the handle's side stream and
    joins it back with events (three chunks over two ring slots, so the fork is taken): captured in
    a graph and replayed on new inputs it must give the eager call's results bit for bit."""
    from mixture_experts_layer_routing_gb300 import moe_train_chunked, moe_train_chunked_sizes
    spec = SPEC.with_(name=f"{prec}_T600_d512_E16+1_f256_top4_chunk256", T=600, dtype=prec, chunk=256, seed=82)
    inp = moe_synth.make_inputs(spec, DEV, grad=True)
    layer = MoeLayer.from_spec(spec, device=DEV)
    layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
    T = spec.T
    z = moe_train_chunked_sizes(layer.h, T)
    assert z["n_chunks"] == 3
    ring = layer.buffer("ring", 2 * z["slot"])
    ws = layer.buffer("chunk_ws", z["workspace"])
    x, dy = inp["x"].clone(), inp["dy"].clone()
    y = torch.empty_like(x)
    g = layer.grads_like(x)

    def step():
        moe_train_chunked(layer.h, x, dy, T, y, g["dx"], g["dWr"], g["dWg"], g["dWu"], g["dWd"], ring, 2 * z["slot"],
                          ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    new = moe_synth.make_tokens(spec, 2, DEV, seed_offset=6)
    x.copy_(new[0])
    dy.copy_(new[1])
    graph.replay()
    torch.cuda.synchronize()
    got = {"y": y.clone(), **{k: v.clone() for k, v in g.items()}}
    step()
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(got["y"], y)
    for k, v in g.items():
        assert torch.equal(got[k], v), k
    layer.close()
