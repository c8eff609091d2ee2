"""GPU parity of the MXFP8 path (E4M3 elements, one E8M0 scale per 32 along each GEMM's K).

* quantiser: the packed weight copies are byte-identical to the oracle's OCP MX quantiser
  (row-wise along d / f, column-wise along the packed 2f rows / d);
* forward and backward: relative Frobenius error <= 3e-2 against the oracle's MXFP8 layer
  (float64 arithmetic on the same bf16 inputs, every operand quantised along its GEMM's K);
  routing uses the GPU's fp32 logits on both sides;
* reruns are bit-identical.
"""
import numpy as np
import pytest
import torch

import moe_synth
from mixture_experts_layer_routing_gb300 import MoeLayer
from oracle import moe_oracle as oracle
from routing_checks import report, routing_exceptions

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
TOL_MX = 3e-2
G_MX = 64      # gate/up interleave of the MXFP8 W13 rows

SMALL_MX = moe_synth.LayerSpec("mxfp8_T300_d512_E16+1_f256_top4_sigmoid", 300, 512, 16, 1, 256, 4, "sigmoid", True,
                               2.5, "mxfp8", None, 31)
# The shared expert's 640 token rows are five 128-row K groups: more than the weight-gradient kernel keeps
# resident, so its A operand streams with B and its tiles are dealt one per unit; the routed experts'
# ~160 rows stay resident.
STREAMED_MX = moe_synth.LayerSpec("mxfp8_T640_d512_E8+1_f256_top2_softmax", 640, 512, 8, 1, 256, 2, "softmax", True,
                                  1.0, "mxfp8", None, 33)


def np64(t):
    return t.detach().double().cpu().numpy()


def kw(spec):
    return dict(k=spec.k, router=spec.router, renorm=spec.renorm, scale=spec.route_scale, n_shared=spec.S)


def setup(spec):
    inp = moe_synth.make_inputs(spec, "cpu", grad=True)
    g = {k: v.to(DEV) for k, v in inp.items()}
    layer = MoeLayer.from_spec(spec, device=DEV)
    layer.set_weights(g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    return layer, g, {k: np64(v) for k, v in inp.items()}


def packed_w13(Wg, Wu, G):
    """[E+S, 2f, d]: gate and up rows interleaved in blocks of G rows."""
    n, f, d = Wg.shape
    out = np.empty((n, 2 * f, d))
    for b in range(f // G):
        out[:, 2 * b * G:(2 * b + 1) * G] = Wg[:, b * G:(b + 1) * G]
        out[:, (2 * b + 1) * G:(2 * b + 2) * G] = Wu[:, b * G:(b + 1) * G]
    return out


def scales_k(raw, rows, K):
    """Scale bytes of a K-major operand as [rows][K/32]. Stored in 512-byte atoms, one per 128 rows and
    128-element K block, in the order the MMA's scale copy takes them: row r of the 128 at byte
    16 (r mod 32) + 4 (r / 32), the four 32-element blocks of the K block in its four bytes."""
    a = raw.reshape(rows // 128, K // 128, 32, 4, 4)          # (row tile, K block, r mod 32, r / 32, block)
    return a.transpose(0, 3, 2, 1, 4).reshape(rows, K // 32)


def scales_mn(raw, Krows, W):
    """Scale bytes of an MN-major operand as [Krows/32][W]: atoms of 128 K rows by 128 columns, column c
    of the 128 at byte 16 (c mod 32) + 4 (c / 32), the four 32-row blocks in its four bytes."""
    a = raw.reshape(Krows // 128, W // 128, 32, 4, 4)        # (K group, column tile, c mod 32, c / 32, block)
    return a.transpose(0, 4, 1, 3, 2).reshape(Krows // 32, W)


def test_mx_weight_quantisation_byte_exact():
    spec = SMALL_MX
    layer, g, n = setup(spec)
    nseg, d, f = spec.E + spec.S, spec.d, spec.f
    al = lambda v: (v + 255) // 256 * 256  # noqa: E731
    raw = layer.packed.cpu().numpy()
    w13, wd = nseg * 2 * f * d, nseg * d * f
    pos = 0
    parts = {}
    for name, size in (("W13q", w13), ("W13s", w13 // 32), ("W13c", w13), ("W13cs", w13 // 32),
                       ("Wdq", wd), ("Wds", wd // 32), ("Wdc", wd), ("Wdcs", wd // 32)):
        parts[name] = raw[pos:pos + size]
        pos += al(size)
    W13 = packed_w13(n["Wg"], n["Wu"], G_MX)
    c, s = oracle.mx_quantize(W13, axis=2)
    assert np.array_equal(parts["W13q"].reshape(c.shape), c)
    assert np.array_equal(scales_k(parts["W13s"], nseg * 2 * f, d).reshape(s.shape), s)
    c, s = oracle.mx_quantize(n["Wd"], axis=2)
    assert np.array_equal(parts["Wdq"].reshape(c.shape), c)
    assert np.array_equal(scales_k(parts["Wds"], nseg * d, f).reshape(s.shape), s)
    c, s = oracle.mx_quantize(W13, axis=1)                 # along the packed 2f rows
    assert np.array_equal(parts["W13c"].reshape(c.shape), c)
    assert np.array_equal(scales_mn(parts["W13cs"], nseg * 2 * f, d).reshape(s.shape), s)
    c, s = oracle.mx_quantize(n["Wd"], axis=1)             # along d
    assert np.array_equal(parts["Wdc"].reshape(c.shape), c)
    assert np.array_equal(scales_mn(parts["Wdcs"], nseg * d, f).reshape(s.shape), s)
    layer.close()


@pytest.mark.parametrize("spec", [SMALL_MX, STREAMED_MX], ids=lambda sp: sp.name)
def test_mx_forward_backward_parity_and_reruns(spec):
    layer, g, n = setup(spec)
    ctx = layer.new_ctx(spec.T)
    y = layer.forward(g["x"], ctx=ctx)
    grads = layer.backward(g["x"], g["dy"], ctx)
    logits = layer.route(g["x"])["logits"].cpu().numpy()
    torch.cuda.synchronize()
    assert layer.status() == 0
    args = (n["x"], n["Wr"], n["b"], n["Wg"], n["Wu"], n["Wd"])
    y_ref = oracle.forward(*args, logits32=logits, mx=True, **kw(spec))["y"]
    ref = oracle.backward(*args, n["dy"], logits32=logits, mx=True, **kw(spec))
    errs = {"y": oracle.rel_frobenius(np64(y), y_ref)}
    for name in ("dx", "dWg", "dWu", "dWd", "dWr"):
        errs[name] = oracle.rel_frobenius(np64(grads[name]), ref[name])
    assert all(v <= TOL_MX for v in errs.values()), errs
    y2 = layer.forward(g["x"], ctx=ctx)
    g2 = layer.backward(g["x"], g["dy"], ctx)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    for name in grads:
        assert torch.equal(grads[name], g2[name]), name
    layer.close()


class DeviceExperts:
    """Indexable view of a device weight stack [E+S, ...] that yields one expert's float64 array at a time."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return self.t[e].double().cpu().numpy()

    def __len__(self):
        return self.t.shape[0]


def test_dsv3_mxfp8_chunked_fullsize_sampled_experts():
    """DeepSeek-V3 shapes, T=8192 in 2368-token chunks, 512 MB ring: properties at full size, the
    weight gradients of sampled experts against the oracle (per chunk, summed in backward order),
    and the y and dx rows of sampled tokens."""
    spec = moe_synth.DSV3_MXFP8
    inp = moe_synth.make_inputs(spec, DEV, grad=True)
    layer = MoeLayer.from_spec(spec, device=DEV)
    layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
    from mixture_experts_layer_routing_gb300 import moe_train_chunked_sizes
    z = moe_train_chunked_sizes(layer.h, spec.T)
    assert z["n_chunks"] == 4
    slots = (512 << 20) // z["slot"]
    assert slots >= 1
    out = layer.train_chunked(inp["x"], inp["dy"], slots=slots)
    keep = {k: v.clone() for k, v in out.items() if torch.is_tensor(v)}
    out4 = layer.train_chunked(inp["x"], inp["dy"], slots=4)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert out["recomputed"] == max(0, 4 - slots) and out4["recomputed"] == 0
    for name, v in keep.items():
        assert torch.equal(v, out4[name]), name           # ring size never changes a result
    r = layer.route(inp["x"])
    cnt = r["cnt"].cpu().numpy()
    assert cnt.sum() == spec.T * spec.k                    # dropless
    logits = r["logits"].cpu().numpy()
    # the MXFP8 layer's router (bf16 tensor-core GEMM) against the oracle's logits, and its selection
    # end to end, over all T tokens
    o4 = routing_exceptions(r["idx"].cpu().numpy(), logits, np64(inp["x"]), np64(inp["Wr"]), np64(inp["b"]),
                            spec.k)
    report(f"routing end to end, {spec.name}", tokens=o4["tokens"], logit_err=o4["logit_err"],
           index_exceptions=o4["exceptions"], near_ties=o4["near_ties"])
    assert o4["logit_err"] < 1e-3 and o4["exceptions"] == 0, (o4["logit_err"], o4["exceptions"])
    rng = np.random.default_rng(1)
    sample = sorted({int(np.argmax(cnt)), spec.E, int(rng.integers(spec.E))})   # hottest, shared, random
    n = {k: np64(inp[k]) for k in ("x", "dy", "Wr", "b")}
    W = {k: DeviceExperts(inp[k]) for k in ("Wg", "Wu", "Wd")}
    acc = {k: {e: 0.0 for e in sample} for k in ("dWg", "dWu", "dWd")}
    for a, b in reversed(oracle.chunk_bounds(spec.T, spec.chunk)):
        g = oracle.backward(n["x"][a:b], n["Wr"], n["b"], W["Wg"], W["Wu"], W["Wd"], n["dy"][a:b],
                            logits32=logits[a:b], mx=True, experts=sample, **kw(spec))
        for k in acc:
            for e in sample:
                acc[k][e] = acc[k][e] + g[k].get(e, 0.0)     # an expert with no token in a chunk adds 0
    for e in sample:
        for k in ("dWg", "dWu", "dWd"):
            err = oracle.rel_frobenius(np64(keep[k][e]), acc[k][e])
            assert err <= TOL_MX, (e, k, err)
    # y and dx rows of two tokens, one in the first chunk (recomputed in the backward: the ring holds
    # fewer slots than there are chunks) and one in the last; every quantised operand of a token's
    # y and dx is quantised along that token's own row, so the oracle can take the tokens alone
    bounds = oracle.chunk_bounds(spec.T, spec.chunk)
    toks = np.array([int(rng.integers(bounds[0][0], bounds[0][1])), int(rng.integers(bounds[-1][0], bounds[-1][1]))])
    ti = torch.as_tensor(toks, device=DEV)
    touched = sorted(set(r["idx"][ti].cpu().numpy().ravel().tolist()) | {spec.E})
    ref = oracle.backward(n["x"][toks], n["Wr"], n["b"], W["Wg"], W["Wu"], W["Wd"], n["dy"][toks],
                          logits32=logits[toks], mx=True, experts=touched, **kw(spec))
    y_ref = oracle.forward(n["x"][toks], n["Wr"], n["b"], W["Wg"], W["Wu"], W["Wd"], logits32=logits[toks],
                           mx=True, **kw(spec))["y"]
    assert oracle.rel_frobenius(np64(keep["y"][ti]), y_ref) <= TOL_MX
    assert oracle.rel_frobenius(np64(keep["dx"][ti]), ref["dx"]) <= TOL_MX
    layer.close()
