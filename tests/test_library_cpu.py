"""CPU checks of the C-ABI library: it builds, loads, exports every declared
symbol, and rejects bad configurations on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

import __graft_entry__
import mixture_experts_layer_routing_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return moe.load_library()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:moe_status|const char\*)\s+(moe_\w+)\s*\(", src, flags=re.M)
    return names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"moe_create", "moe_route", "moe_forward", "moe_backward", "moe_decode"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(moe.EXPORTED) <= set(names)


def _create(**over):
    base = dict(T_max=16, d=256, E=8, n_shared=0, f=128, k=2, router=0, renorm=1, route_scale=1.0, prec=1,
                chunk_tokens=0, ring_bytes=0)
    base.update(over)
    cfg = moe.moe_config(*base.values())
    h = ctypes.c_void_p()
    return moe.load_library().moe_create(ctypes.byref(cfg), ctypes.byref(h))


@pytest.mark.parametrize("over,code", [
    (dict(k=9, E=16), moe.MOE_ERR_INVALID_ARG),       # k above the maximum
    (dict(k=3, E=2), moe.MOE_ERR_INVALID_ARG),        # k > E
    (dict(n_shared=2), moe.MOE_ERR_INVALID_ARG),
    (dict(T_max=0), moe.MOE_ERR_INVALID_ARG),
    (dict(route_scale=-1.0), moe.MOE_ERR_INVALID_ARG),
    (dict(router=5), moe.MOE_ERR_INVALID_ARG),
    (dict(f=96), moe.MOE_ERR_UNSUPPORTED),             # f not a multiple of 64
    (dict(d=100), moe.MOE_ERR_UNSUPPORTED),            # d not a multiple of 8
    (dict(E=300), moe.MOE_ERR_UNSUPPORTED),            # above the routing kernels' expert limit
    (dict(k=0), moe.MOE_ERR_INVALID_ARG),
    (dict(d=0), moe.MOE_ERR_INVALID_ARG),
    (dict(E=0), moe.MOE_ERR_INVALID_ARG),
    (dict(f=0), moe.MOE_ERR_INVALID_ARG),
    (dict(prec=7), moe.MOE_ERR_INVALID_ARG),           # unknown precision
    (dict(route_scale=0.0), moe.MOE_ERR_INVALID_ARG),
    (dict(route_scale=float("nan")), moe.MOE_ERR_INVALID_ARG),
    (dict(route_scale=float("inf")), moe.MOE_ERR_INVALID_ARG),
    (dict(chunk_tokens=-1), moe.MOE_ERR_INVALID_ARG),
    (dict(prec=2, d=192), moe.MOE_ERR_UNSUPPORTED),     # MXFP8: d not a multiple of 128
    (dict(prec=2, f=192), moe.MOE_ERR_UNSUPPORTED),     # MXFP8: f not a multiple of 128
    (dict(T_max=1 << 28, k=4, E=8), moe.MOE_ERR_UNSUPPORTED),   # T*k assignments past 2^30
])
def test_create_rejects_bad_config_on_host(lib, over, code):
    assert _create(**over) == code


def test_create_null_pointers_rejected(lib):
    cfg = moe.moe_config(16, 256, 8, 0, 128, 2, 0, 1, 1.0, 1, 0, 0)
    h = ctypes.c_void_p()
    assert lib.moe_create(None, ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_create(ctypes.byref(cfg), None) == moe.MOE_ERR_INVALID_ARG


def test_null_arguments_rejected(lib):
    assert lib.moe_forward(None, None, 1, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_route(None, None, 1, *([None] * 10)) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_decode(None, None, 1, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_pairs(None, 1) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_fused(None, 1) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_decode_crossover(None, 8) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_status_string(3) == b"workspace or context too small or misaligned"
