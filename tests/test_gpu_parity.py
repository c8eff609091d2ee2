"""GPU parity of the C-ABI path against the CPU oracle (small and ragged sizes).

Tolerances:
  * routing indices, counts, offsets, permutation: bit-exact given the same
    fp32 logits (the selection is an integer decision taken in fp32 on both
    sides); gates within 2e-6 absolute (fp32 expf against float64).
  * bf16 path: relative Frobenius error <= 5e-3 against the float64 oracle on
    the same bf16 inputs.
  * fp32 path: relative Frobenius error <= 1e-5 (fp32 storage of h and o and
    fp32 accumulation over K <= a few thousand terms give ~1e-6).
  * reruns: bit-identical.
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
TOL = {"bf16": 5e-3, "fp32": 1e-5}

SMALL_BF16 = moe_synth.LayerSpec("bf16_T300_d512_E16+1_f256_top4_sigmoid", 300, 512, 16, 1, 256, 4, "sigmoid",
                                 True, 2.5, "bf16", None, 21)
SMALL_SOFTMAX = moe_synth.LayerSpec("bf16_T333_d384_E12_f192_top3_softmax", 333, 384, 12, 0, 192, 3, "softmax",
                                    True, 1.0, "bf16", None, 22)


def np64(t):
    return t.detach().double().cpu().numpy()


def setup(spec, grad=True, bias=None):
    inp = moe_synth.make_inputs(spec, "cpu", grad=grad)
    if bias is not None:
        inp["b"] = torch.as_tensor(bias, dtype=torch.float32)
    g = {k: v.to(DEV) for k, v in inp.items()}
    layer = MoeLayer.from_spec(spec, device=DEV)
    layer.set_weights(g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"])
    n = {k: np64(v) for k, v in inp.items()}
    return layer, g, n


def kw(spec):
    return dict(k=spec.k, router=spec.router, renorm=spec.renorm, scale=spec.route_scale, n_shared=spec.S)


def assert_rel(got, ref, tol, what):
    err = oracle.rel_frobenius(got, ref)
    assert err <= tol, f"{what}: relative Frobenius error {err:.3e} > {tol:.1e}"
    return err


# ---------------------------------------------------------------- routing

def check_route_given_logits(layer, spec, logits, bias):
    r = layer.route(T=logits.shape[0], logits_override=logits)
    torch.cuda.synchronize()
    ref = oracle.route(None, np.zeros((spec.E, 1)), bias, spec.k, spec.router, spec.renorm, spec.route_scale,
                       logits32=logits.cpu().numpy())
    assert np.array_equal(r["idx"].cpu().numpy(), ref["idx"])
    assert np.array_equal(r["cnt"].cpu().numpy(), ref["cnt"])
    assert np.array_equal(r["off"].cpu().numpy(), ref["off"])
    assert np.array_equal(r["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(r["inv"].cpu().numpy(), ref["inv"])
    np.testing.assert_allclose(r["gate"].cpu().numpy(), ref["gate"], rtol=0, atol=2e-6)


@pytest.mark.parametrize("spec", [SMALL_BF16, SMALL_SOFTMAX], ids=lambda s: s.name)
def test_route_bit_exact_given_logits(spec):
    rng = np.random.default_rng(5)
    bias = (rng.standard_normal(spec.E) * 0.5).astype(np.float32)
    layer, g, n = setup(spec, grad=False, bias=bias)
    logits = torch.from_numpy((rng.standard_normal((spec.T, spec.E)) * 2).astype(np.float32)).to(DEV)
    check_route_given_logits(layer, spec, logits, bias)
    # tie-heavy logits: multiples of 0.5 in [-2, 2]
    tied = torch.from_numpy((rng.integers(-4, 5, (spec.T, spec.E)) * 0.5).astype(np.float32)).to(DEV)
    check_route_given_logits(layer, spec, tied, bias)
    layer.close()


def test_route_end_to_end_tiny_fp32():
    spec = moe_synth.TINY_FP32
    layer, g, n = setup(spec, grad=False)
    r = layer.route(g["x"])
    torch.cuda.synchronize()
    o4 = routing_exceptions(r["idx"].cpu().numpy(), r["logits"].cpu().numpy(), n["x"], n["Wr"], n["b"], spec.k)
    report("routing end to end, tiny fp32", tokens=o4["tokens"], logit_err=o4["logit_err"],
           index_exceptions=o4["exceptions"], near_ties=o4["near_ties"])
    assert o4["logit_err"] < 1e-5
    # the reading's requirement for this workload: no exception, and no near-tie either
    assert o4["exceptions"] == 0
    assert o4["near_ties"] == 0
    assert np.array_equal(r["idx"].cpu().numpy(), o4["ref_idx"])
    layer.close()


# ---------------------------------------------------------------- forward

def run_forward_backward(spec, layer, g, grad=True):
    ctx = layer.new_ctx(spec.T) if grad else None
    y = layer.forward(g["x"], ctx=ctx)
    out = {"y": y}
    if grad:
        out.update(layer.backward(g["x"], g["dy"], ctx))
    torch.cuda.synchronize()
    assert layer.status() == 0
    return out


@pytest.mark.parametrize("spec", [moe_synth.TINY_FP32, SMALL_BF16, SMALL_SOFTMAX], ids=lambda s: s.name)
def test_forward_backward_parity(spec):
    layer, g, n = setup(spec, grad=True)
    out = run_forward_backward(spec, layer, g)
    args = (n["x"], n["Wr"], n["b"], n["Wg"], n["Wu"], n["Wd"])
    ref = oracle.backward(*args, n["dy"], **kw(spec))
    y_ref = oracle.forward(*args, **kw(spec))["y"]
    tol = TOL[spec.dtype]
    assert_rel(np64(out["y"]), y_ref, tol, "y")
    for name in ("dx", "dWg", "dWu", "dWd", "dWr"):
        assert_rel(np64(out[name]), ref[name], tol, name)
    layer.close()


def test_reruns_bit_identical():
    spec = SMALL_BF16
    layer, g, n = setup(spec, grad=True)
    a = run_forward_backward(spec, layer, g)
    b = run_forward_backward(spec, layer, g)
    for name in a:
        assert torch.equal(a[name], b[name]), name
    layer.close()


def test_unused_experts_get_zero_gradients():
    spec = SMALL_SOFTMAX
    bias = np.zeros(spec.E, np.float32)
    bias[[2, 7]] = -1e4                                 # never selected
    layer, g, n = setup(spec, grad=True, bias=bias)
    out = run_forward_backward(spec, layer, g)
    for name in ("dWg", "dWu", "dWd"):
        assert torch.count_nonzero(out[name][[2, 7]]) == 0
    assert torch.count_nonzero(out["dWr"][[2, 7]]) == 0
    args = (n["x"], n["Wr"], bias, n["Wg"], n["Wu"], n["Wd"])
    y_ref = oracle.forward(*args, **kw(spec))["y"]
    assert_rel(np64(out["y"]), y_ref, TOL["bf16"], "y")
    layer.close()


def test_all_tokens_to_one_expert_and_single_token():
    spec = SMALL_SOFTMAX.with_(T=257)
    bias = np.zeros(spec.E, np.float32)
    bias[5] = 1e4                                       # every token picks expert 5 first
    layer, g, n = setup(spec, grad=True, bias=bias)
    out = run_forward_backward(spec, layer, g)
    args = (n["x"], n["Wr"], bias, n["Wg"], n["Wu"], n["Wd"])
    ref = oracle.backward(*args, n["dy"], **kw(spec))
    assert_rel(np64(out["y"]), oracle.forward(*args, **kw(spec))["y"], TOL["bf16"], "y")
    for name in ("dx", "dWg", "dWu", "dWd"):
        assert_rel(np64(out[name]), ref[name], TOL["bf16"], name)
    y1 = layer.forward(g["x"][:1].contiguous())
    torch.cuda.synchronize()
    y1_ref = oracle.forward(n["x"][:1], *args[1:], **kw(spec))["y"]
    assert_rel(np64(y1), y1_ref, TOL["bf16"], "y (T=1)")
    layer.close()


# ----------------------------------------------------------------- decode

@pytest.mark.parametrize("path", ["warp", "crossover"])
@pytest.mark.parametrize("B", [1, 4, 16])
def test_decode_parity(B, path):
    """path "warp": the warp-per-output kernels at every B; "crossover": the default, where
    moe_decode takes the grouped-GEMM forward from B = 4 (then equal to moe_forward bit for bit)."""
    from mixture_experts_layer_routing_gb300 import moe_set_decode_crossover
    spec = SMALL_BF16
    layer, g, n = setup(spec, grad=False)
    moe_set_decode_crossover(layer.h, 65 if path == "warp" else 4)
    x = g["x"][:B].contiguous()
    y = layer.decode(x)
    if path == "crossover" and B >= 4:
        assert torch.equal(y, layer.forward(x))
    torch.cuda.synchronize()
    assert layer.status() == 0
    args = (n["x"][:B], n["Wr"], n["b"], n["Wg"], n["Wu"], n["Wd"])
    ref = oracle.decode(*args, **kw(spec))["y"]
    assert_rel(np64(y), ref, TOL["bf16"], f"decode B={B}")
    y2 = layer.decode(x)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    layer.close()
