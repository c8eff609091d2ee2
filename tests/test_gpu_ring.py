"""GPU tests of the chunked training step over a fixed ring of saved activations.

* every ring size R gives bit-identical outputs (recomputation replays the same kernels);
* the backward walks the chunks in reverse and recomputes exactly n - R chunk forwards;
* the results match the oracle's chunked forward + backward (weight gradients summed over
  chunks in backward order) within the path's tolerance: 5e-3 for bf16, 3e-2 for MXFP8.
"""
import numpy as np
import pytest
import torch

import moe_synth
from mixture_experts_layer_routing_gb300 import MoeLayer
from oracle import moe_oracle as oracle

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

BF16_RING = moe_synth.LayerSpec("bf16_T600_d512_E16+1_f256_top4_chunk256", 600, 512, 16, 1, 256, 4, "sigmoid", True,
                                2.5, "bf16", None, 41, chunk=256)
MX_RING = BF16_RING.with_(name="mxfp8_T600_d512_E16+1_f256_top4_chunk256", dtype="mxfp8", seed=42)


def np64(t):
    return t.detach().double().cpu().numpy()


@pytest.mark.parametrize("spec,tol", [(BF16_RING, 5e-3), (MX_RING, 3e-2)], ids=["bf16", "mxfp8"])
def test_ring_reverse_walk(spec, tol):
    inp = moe_synth.make_inputs(spec, "cpu", grad=True)
    g = {k: v.to(DEV) for k, v in inp.items()}
    layer = MoeLayer.from_spec(spec, device=DEV)
    layer.set_weights(g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"])
    runs = {}
    for R in (1, 2, 3, 4):
        out = layer.train_chunked(g["x"], g["dy"], slots=R)
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert out["n_chunks"] == 3
        assert out["recomputed"] == max(0, 3 - R), (R, out["recomputed"])
        runs[R] = {k: v.clone() for k, v in out.items() if torch.is_tensor(v)}
    for R in (2, 3, 4):
        for name, v in runs[R].items():
            assert torch.equal(v, runs[1][name]), (R, name)
    n = {k: np64(v) for k, v in inp.items()}
    kw = dict(k=spec.k, router=spec.router, renorm=spec.renorm, scale=spec.route_scale, n_shared=spec.S,
              mx=spec.dtype == "mxfp8")
    # route both sides with the GPU's fp32 logits (selection is decided in fp32 on both)
    logits = layer.route(g["x"])["logits"].cpu().numpy()
    ref = {}
    ys, dxs = [], []
    for a, b in oracle.chunk_bounds(spec.T, spec.chunk):
        ys.append(oracle.forward(n["x"][a:b], n["Wr"], n["b"], n["Wg"], n["Wu"], n["Wd"], logits32=logits[a:b],
                                 **kw)["y"])
    acc = None
    for a, b in reversed(oracle.chunk_bounds(spec.T, spec.chunk)):
        gr = oracle.backward(n["x"][a:b], n["Wr"], n["b"], n["Wg"], n["Wu"], n["Wd"], n["dy"][a:b],
                             logits32=logits[a:b], **kw)
        dxs.append((a, gr["dx"]))
        if acc is None:
            acc = {k: gr[k].copy() for k in ("dWr", "dWg", "dWu", "dWd")}
        else:
            for k in acc:
                acc[k] += gr[k]
    ref["y"] = np.concatenate(ys)
    ref["dx"] = np.concatenate([d for _, d in sorted(dxs, key=lambda t: t[0])])
    ref.update(acc)
    errs = {k: oracle.rel_frobenius(np64(runs[1][k]), ref[k]) for k in ("y", "dx", "dWr", "dWg", "dWu", "dWd")}
    assert all(v <= tol for v in errs.values()), errs
    layer.close()
