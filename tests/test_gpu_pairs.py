"""The bf16 expert GEMMs on 2-SM CTA pairs (clusters of two CTAs, one
tcgen05.mma.cta_group::2 per K step over a 256-row tile) against the oracle and
against the single-SM schedule.

Cases are chosen so that experts have odd and even numbers of 128-row tiles,
some a single partial tile, and (with a Zipf-biased router) some none; the
pair's second tile is then partly or wholly past the expert's rows.

* forward and backward with pairs forced on: relative Frobenius error <= 5e-3
  against the float64 oracle (the bf16 tolerance);
* pairs on vs off: the same values up to fp32 summation order inside the
  tensor core (relative difference <= 1e-5);
* reruns with pairs on: bit-identical.
"""
import numpy as np
import pytest
import torch

import moe_synth
from mixture_experts_layer_routing_gb300 import MoeLayer, moe_set_pairs
from oracle import moe_oracle as oracle

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

CASES = [
    # ~290 rows per routed expert (2-3 tiles) and a 1000-row shared expert (8 tiles)
    (moe_synth.LayerSpec("bf16_T1000_d512_E16+1_f256_top5_sigmoid", 1000, 512, 16, 1, 256, 5, "sigmoid", True, 2.5,
                         "bf16", None, 61), None),
    # a selection bias falling from +4 to -4 over the experts: hot experts with many tiles, cold ones with none
    (moe_synth.LayerSpec("bf16_T1500_d512_E32_f384_top4_softmax_skewed", 1500, 512, 32, 0, 384, 4, "softmax", True,
                         1.0, "bf16", None, 62), np.linspace(4.0, -4.0, 32)),
]


def np64(t):
    return t.detach().double().cpu().numpy()


def run(layer, g, mode):
    moe_set_pairs(layer.h, mode)
    ctx = layer.new_ctx(g["x"].shape[0])
    y = layer.forward(g["x"], ctx=ctx)
    grads = layer.backward(g["x"], g["dy"], ctx)
    torch.cuda.synchronize()
    assert layer.status() == 0
    out = {"y": y.clone()}
    out.update({k: v.clone() for k, v in grads.items()})
    return out


@pytest.mark.parametrize("spec,bias", CASES, ids=[c[0].name for c in CASES])
def test_pairs_parity(spec, bias):
    inp = moe_synth.make_inputs(spec, DEV, grad=True)
    if bias is not None:
        inp["b"] = torch.as_tensor(bias, dtype=torch.float32, device=DEV)
    layer = MoeLayer.from_spec(spec, device=DEV)
    layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
    on = run(layer, inp, 1)
    on2 = run(layer, inp, 1)
    off = run(layer, inp, 0)
    for k in on:
        assert torch.equal(on[k], on2[k]), k
        diff = oracle.rel_frobenius(np64(on[k]), np64(off[k]))
        assert diff <= 1e-5, (k, diff)
    r = layer.route(inp["x"])
    logits = r["logits"].cpu().numpy()
    n = {k: np64(inp[k]) for k in ("x", "dy", "Wr", "b", "Wg", "Wu", "Wd")}
    args = (n["x"], n["Wr"], n["b"], n["Wg"], n["Wu"], n["Wd"])
    kw = dict(k=spec.k, router=spec.router, renorm=spec.renorm, scale=spec.route_scale, n_shared=spec.S)
    y_ref = oracle.forward(*args, logits32=logits, **kw)["y"]
    ref = oracle.backward(*args, n["dy"], logits32=logits, **kw)
    errs = {"y": oracle.rel_frobenius(np64(on["y"]), y_ref)}
    for k in ("dx", "dWg", "dWu", "dWd", "dWr"):
        errs[k] = oracle.rel_frobenius(np64(on[k]), ref[k])
    assert all(v <= 5e-3 for v in errs.values()), errs
    # the tile structure the cases are meant to cover
    tiles = (r["cnt"].cpu().numpy() + 127) // 128
    assert (tiles % 2 == 1).any() and (tiles >= 2).any()
    if bias is not None:
        assert (tiles == 0).any()
    layer.close()


def interleaved(cnt_with_shared):
    """Whether the routing scan interleaves dense and sparse experts for these counts (its rule:
    experts with >= 3 row tiles hold a quarter of the tiles and the others average under 1.5)."""
    tiles = (np.asarray(cnt_with_shared) + 127) // 128
    cand = tiles >= 3
    return 4 * tiles[cand].sum() >= tiles.sum() and 2 * tiles[~cand].sum() < 3 * np.count_nonzero(~cand & (tiles > 0))


@pytest.mark.parametrize("spec,bias", CASES, ids=[c[0].name for c in CASES])
def test_two_row_tiles_per_cta_bit_identical(spec, bias):
    """Mode 2 (one CTA per two 128-row tiles of an expert, two M = 128 MMAs per K step sharing the
    staged weight tile) computes every output element with the same instructions in the same K order
    as mode 0: results must be bit-identical, forward and backward, and rerun bit-identically. The
    cases give experts odd tile counts (a lone last tile), single partial tiles and no tiles, in the
    segment-major order (uniform case) and the dense/sparse interleave (skewed case)."""
    inp = moe_synth.make_inputs(spec, DEV, grad=True)
    if bias is not None:
        inp["b"] = torch.as_tensor(bias, dtype=torch.float32, device=DEV)
    layer = MoeLayer.from_spec(spec, device=DEV)
    layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
    two = run(layer, inp, 2)
    two2 = run(layer, inp, 2)
    one = run(layer, inp, 0)
    for k in one:
        assert torch.equal(two[k], two2[k]), k
        assert torch.equal(two[k], one[k]), k
    cnt = layer.route(inp["x"])["cnt"].cpu().numpy()
    full = np.concatenate([cnt, [spec.T] * spec.S])
    tiles = (full + 127) // 128
    assert (tiles % 2 == 1).any() and (tiles >= 2).any()
    assert interleaved(full) == (bias is not None)
    moe_set_pairs(layer.h, 0)
    layer.close()
