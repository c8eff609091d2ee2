"""moe_route_noalloc against moe_route (GPU).

moe_route_noalloc serves callers that may not allocate device memory (for
example a plugin whose host program owns all device memory, or a serving loop
that bans cudaMalloc after start-up): its scratch is a fixed array inside the
library instead of a caller workspace. It runs the same routing kernels as
moe_route, so every output must be bit-identical to moe_route's on the same
input, call after call. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import __graft_entry__
import moe_synth

pytestmark = pytest.mark.gpu

SPEC = moe_synth.LayerSpec("bf16_T300_d512_E16+1_f256_top4_sigmoid", 300, 512, 16, 1, 256, 4, "sigmoid", True,
                           2.5, "bf16", None, 21)
# one handle per router path: tensor-core router (bf16, MXFP8 layers) and CUDA-core router (fp32);
# d and f suit every precision's expert path (multiples of 256 and 128)
SPECS = {"bf16": SPEC,
         "mxfp8": SPEC.with_(name="mxfp8_T300_d512_E16+1_f256_top4_sigmoid", dtype="mxfp8", seed=22),
         "fp32": SPEC.with_(name="fp32_T300_d512_E16+1_f256_top4_softmax", dtype="fp32", router="softmax",
                            route_scale=1.0, seed=23)}


def _outputs(T, E, k, dev):
    return dict(logits=torch.full((T, E), float("nan"), device=dev),
                idx=torch.full((T, k), -1, dtype=torch.int32, device=dev),
                gate=torch.full((T, k), float("nan"), device=dev),
                cnt=torch.full((E,), -1, dtype=torch.int32, device=dev),
                off=torch.full((E + 1,), -1, dtype=torch.int32, device=dev),
                perm=torch.full((T * k,), -1, dtype=torch.int32, device=dev),
                inv=torch.full((T * k,), -1, dtype=torch.int32, device=dev))


@pytest.mark.parametrize("prec", list(SPECS))
def test_route_noalloc_matches_route_on_two_calls(prec):
    __graft_entry__.build()
    import mixture_experts_layer_routing_gb300 as moe
    spec = SPECS[prec]
    dev = torch.device("cuda:0")
    inp = moe_synth.make_inputs(spec, "cpu")
    g = {n: v.to(dev) for n, v in inp.items()}
    layer = moe.MoeLayer.from_spec(spec, device=dev)
    layer.set_weights(g["Wr"], g["b"], g["Wg"], g["Wu"], g["Wd"])
    for call in range(2):
        x = moe_synth.make_tokens(spec, 1, "cpu", seed_offset=100 + call)[0].to(dev)
        n0 = moe.moe_launch_count(layer.h)
        want = layer.route(x)
        n1 = moe.moe_launch_count(layer.h)
        got = _outputs(spec.T, spec.E, spec.k, dev)
        moe.moe_route_noalloc(layer.h, x, spec.T, got["logits"], got["idx"], got["gate"], got["cnt"],
                              got["off"], got["perm"], got["inv"])
        n2 = moe.moe_launch_count(layer.h)
        torch.cuda.synchronize()
        assert layer.status() == 0
        # the same kernels as moe_route, counted the same way
        assert n2 - n1 == n1 - n0, (prec, call, n1 - n0, n2 - n1)
        for name in want:
            assert torch.equal(got[name], want[name]), (prec, call, name)
        assert int(got["cnt"].sum()) == spec.T * spec.k
    layer.close()


def test_route_noalloc_rejects_sizes_beyond_its_scratch():
    __graft_entry__.build()
    import mixture_experts_layer_routing_gb300 as moe
    dev = torch.device("cuda:0")
    small = SPEC.with_(T=8, d=256, E=8, S=0, f=128, k=2)
    inp = {n: v.to(dev) for n, v in moe_synth.make_inputs(small, "cpu").items()}
    layer = moe.MoeLayer(1 << 21, small.d, small.E, 0, small.f, small.k, "sigmoid", True, 2.5, "bf16", device=dev)
    layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
    out = _outputs(8, small.E, small.k, dev)
    lib = moe.load_library()
    # 2^21 tokens x 2 experts need far more than the fixed scratch: rejected before any launch
    rc = lib.moe_route_noalloc(layer.h, inp["x"].data_ptr(), 1 << 21, out["logits"].data_ptr(),
                               out["idx"].data_ptr(), out["gate"].data_ptr(), out["cnt"].data_ptr(),
                               out["off"].data_ptr(), out["perm"].data_ptr(), out["inv"].data_ptr(),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == moe.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out["idx"] == -1)
    layer.close()
