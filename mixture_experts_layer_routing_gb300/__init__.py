"""Python binding of the GB300 MoE layer library (libmoe_gb300.so).

Argument marshalling only: every function here forwards to the C ABI of the
same name declared in include/moe.h, passing torch tensors as device pointers
and the current torch stream. All compute runs in the library's CUDA kernels;
there is no fallback. Importing this module fails loudly if the library has not
been built (see build.py).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, \
    MOE_ERR_DEVICE_INDEX, MOE_ERR_NO_WEIGHTS = range(8)
MOE_ROUTER_SOFTMAX, MOE_ROUTER_SIGMOID = 0, 1
MOE_FP32, MOE_BF16, MOE_MXFP8 = 0, 1, 2

EXPORTED = ("moe_create", "moe_destroy", "moe_workspace_size", "moe_set_weights", "moe_route", "moe_forward",
            "moe_backward", "moe_decode", "moe_get_status", "moe_profile_enable", "moe_profile_read",
            "moe_launch_count", "moe_route_noalloc", "moe_train_chunked_sizes", "moe_train_chunked",
            "moe_selftest_timeout", "moe_set_pairs", "moe_set_fused", "moe_set_decode_crossover",
            "moe_status_string")


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


class moe_config(ctypes.Structure):
    _fields_ = [("T_max", ctypes.c_int), ("d", ctypes.c_int), ("E", ctypes.c_int), ("n_shared", ctypes.c_int),
                ("f", ctypes.c_int), ("k", ctypes.c_int), ("router", ctypes.c_int), ("renorm", ctypes.c_int),
                ("route_scale", ctypes.c_float), ("prec", ctypes.c_int), ("chunk_tokens", ctypes.c_int),
                ("ring_bytes", ctypes.c_size_t)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library; raises if it is missing (run build.build() first)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with mixture_experts_layer_routing_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    P = ctypes.POINTER
    lib.moe_create.argtypes = [P(moe_config), P(vp)]
    lib.moe_destroy.argtypes = [vp]
    lib.moe_workspace_size.argtypes = [vp, i32, P(sz), P(sz), P(sz), P(sz)]
    lib.moe_set_weights.argtypes = [vp] + [vp] * 7
    lib.moe_route.argtypes = [vp, vp, i32] + [vp] * 10
    lib.moe_forward.argtypes = [vp, vp, i32, vp, vp, vp, vp]
    lib.moe_backward.argtypes = [vp, vp, vp, i32] + [vp] * 8
    lib.moe_decode.argtypes = [vp, vp, i32, vp, vp, vp]
    lib.moe_get_status.argtypes = [vp, vp, P(i32)]
    lib.moe_profile_enable.argtypes = [vp, i32]
    lib.moe_profile_read.argtypes = [vp, i32, ctypes.c_char_p, P(ctypes.c_longlong), P(ctypes.c_double), P(i32)]
    lib.moe_launch_count.argtypes = [vp, P(ctypes.c_longlong)]
    lib.moe_route_noalloc.argtypes = [vp, vp, i32] + [vp] * 8
    lib.moe_selftest_timeout.argtypes = [vp, i32, vp]
    lib.moe_train_chunked_sizes.argtypes = [vp, i32, P(sz), P(sz), P(i32)]
    lib.moe_train_chunked.argtypes = [vp, vp, vp, i32] + [vp] * 7 + [sz, vp, P(i32), vp]
    lib.moe_set_pairs.argtypes = [vp, i32]
    lib.moe_set_fused.argtypes = [vp, i32]
    lib.moe_set_decode_crossover.argtypes = [vp, i32]
    lib.moe_status_string.argtypes = [i32]
    lib.moe_status_string.restype = ctypes.c_char_p
    for name in EXPORTED[:-1]:
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().moe_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != MOE_OK:
        raise MoeError(code, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ C ABI

def moe_create(T_max: int, d: int, E: int, n_shared: int, f: int, k: int, router: int, renorm: bool,
               route_scale: float, prec: int, chunk_tokens: int = 0, ring_bytes: int = 0) -> int:
    cfg = moe_config(T_max, d, E, n_shared, f, k, router, int(bool(renorm)), route_scale, prec, chunk_tokens,
                     ring_bytes)
    h = ctypes.c_void_p()
    _check(load_library().moe_create(ctypes.byref(cfg), ctypes.byref(h)), "moe_create")
    return h.value


def moe_destroy(h: int):
    _check(load_library().moe_destroy(h), "moe_destroy")


def moe_workspace_size(h: int, T: int) -> dict:
    out = [ctypes.c_size_t() for _ in range(4)]
    _check(load_library().moe_workspace_size(h, T, *[ctypes.byref(o) for o in out]), "moe_workspace_size")
    return dict(fwd_ws=out[0].value, ctx=out[1].value, bwd_ws=out[2].value, packed=out[3].value)


def moe_set_weights(h, Wr, bias, Wg, Wu, Wd, packed, stream=None):
    _check(load_library().moe_set_weights(h, _ptr(Wr), _ptr(bias), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(packed),
                                          _stream(stream)), "moe_set_weights")


def moe_route(h, x, T, logits_override, logits, idx, gate, cnt, off, perm, inv, workspace, stream=None):
    _check(load_library().moe_route(h, _ptr(x), T, _ptr(logits_override), _ptr(logits), _ptr(idx), _ptr(gate),
                                    _ptr(cnt), _ptr(off), _ptr(perm), _ptr(inv), _ptr(workspace), _stream(stream)),
           "moe_route")


def moe_route_noalloc(h, x, T, logits, idx, gate, cnt, off, perm, inv, stream=None):
    """Routing without a workspace (scratch in a fixed array inside the library); see include/moe.h."""
    _check(load_library().moe_route_noalloc(h, _ptr(x), T, _ptr(logits), _ptr(idx), _ptr(gate), _ptr(cnt),
                                            _ptr(off), _ptr(perm), _ptr(inv), _stream(stream)), "moe_route_noalloc")


def moe_forward(h, x, T, y, ctx, workspace, stream=None):
    _check(load_library().moe_forward(h, _ptr(x), T, _ptr(y), _ptr(ctx), _ptr(workspace), _stream(stream)),
           "moe_forward")


def moe_backward(h, x, dy, T, ctx, dx, dWr, dWg, dWu, dWd, workspace, stream=None):
    _check(load_library().moe_backward(h, _ptr(x), _ptr(dy), T, _ptr(ctx), _ptr(dx), _ptr(dWr), _ptr(dWg),
                                       _ptr(dWu), _ptr(dWd), _ptr(workspace), _stream(stream)), "moe_backward")


def moe_selftest_timeout(h, limit_ms: int, stream=None):
    _check(load_library().moe_selftest_timeout(h, limit_ms, _stream(stream)), "moe_selftest_timeout")


def moe_train_chunked_sizes(h, T) -> dict:
    slot, ws, n = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_int()
    _check(load_library().moe_train_chunked_sizes(h, T, ctypes.byref(slot), ctypes.byref(ws), ctypes.byref(n)),
           "moe_train_chunked_sizes")
    return dict(slot=slot.value, workspace=ws.value, n_chunks=n.value)


def moe_train_chunked(h, x, dy, T, y, dx, dWr, dWg, dWu, dWd, ring, ring_bytes, workspace, stream=None) -> int:
    """Returns the number of recomputed chunk forwards."""
    rec = ctypes.c_int(-1)
    _check(load_library().moe_train_chunked(h, _ptr(x), _ptr(dy), T, _ptr(y), _ptr(dx), _ptr(dWr), _ptr(dWg),
                                            _ptr(dWu), _ptr(dWd), _ptr(ring), int(ring_bytes), _ptr(workspace),
                                            ctypes.byref(rec), _stream(stream)), "moe_train_chunked")
    return rec.value


def moe_decode(h, x, B, y, workspace, stream=None):
    _check(load_library().moe_decode(h, _ptr(x), B, _ptr(y), _ptr(workspace), _stream(stream)), "moe_decode")


def moe_set_pairs(h, mode: int):
    """Expert GEMMs on 2-SM CTA pairs (1) or one CTA per tile (0, the default)."""
    _check(load_library().moe_set_pairs(h, mode), "moe_set_pairs")


def moe_set_fused(h, on: int):
    """Forward as one persistent kernel: 1 the two expert GEMMs, 2 the whole forward (routing, both
    expert GEMMs, combine); 0 separate launches (the default). Results are bit-identical."""
    _check(load_library().moe_set_fused(h, on), "moe_set_fused")


def moe_set_decode_crossover(h, b_min: int):
    """Batch size from which moe_decode takes the grouped-GEMM forward (default 8; 65: never)."""
    _check(load_library().moe_set_decode_crossover(h, b_min), "moe_set_decode_crossover")


def moe_get_status(h, stream=None) -> int:
    v = ctypes.c_int()
    _check(load_library().moe_get_status(h, _stream(stream), ctypes.byref(v)), "moe_get_status")
    return v.value


def moe_profile_enable(h, enable: bool = True):
    _check(load_library().moe_profile_enable(h, int(bool(enable))), "moe_profile_enable")


def moe_profile_read(h, max_groups: int = 32) -> dict:
    """{group name: (kernel launches, total ms)} of the launches recorded since the last read."""
    names = ctypes.create_string_buffer(32 * max_groups)
    launches = (ctypes.c_longlong * max_groups)()
    ms = (ctypes.c_double * max_groups)()
    n = ctypes.c_int()
    _check(load_library().moe_profile_read(h, max_groups, names, launches, ms, ctypes.byref(n)), "moe_profile_read")
    out = {}
    for i in range(n.value):
        name = names.raw[32 * i:32 * i + 32].split(b"\0", 1)[0].decode()
        out[name] = (launches[i], ms[i])
    return out


def moe_launch_count(h) -> int:
    v = ctypes.c_longlong()
    _check(load_library().moe_launch_count(h, ctypes.byref(v)), "moe_launch_count")
    return v.value


# --------------------------------------------- buffers owned through torch

_PREC = {"fp32": MOE_FP32, "bf16": MOE_BF16, "mxfp8": MOE_MXFP8}
_ROUTER = {"softmax": MOE_ROUTER_SOFTMAX, "sigmoid": MOE_ROUTER_SIGMOID}


def _bytes(n: int, device) -> torch.Tensor:
    # 256-byte aligned device buffer (torch's caching allocator aligns to 512 bytes)
    return torch.empty(max(int(n), 256), dtype=torch.uint8, device=device)


class MoeLayer:
    """One layer handle plus the torch-allocated buffers its calls need.

    Holds the packed weights and grows its workspaces on demand; every compute
    method forwards to the C ABI.
    """

    def __init__(self, T_max, d, E, n_shared, f, k, router="softmax", renorm=True, route_scale=1.0,
                 prec="bf16", chunk_tokens=0, ring_bytes=0, device="cuda"):
        self.device = torch.device(device)
        self.prec = prec
        self.shape = dict(T_max=T_max, d=d, E=E, S=n_shared, f=f, k=k)
        self.h = moe_create(T_max, d, E, n_shared, f, k, _ROUTER[router], renorm, route_scale, _PREC[prec],
                            chunk_tokens, ring_bytes)
        self.packed = None
        self._ws = {}

    @classmethod
    def from_spec(cls, spec, T_max=None, device="cuda"):
        return cls(T_max or spec.T, spec.d, spec.E, spec.S, spec.f, spec.k, spec.router, spec.renorm,
                   spec.route_scale, spec.dtype, spec.chunk, 0, device)

    def close(self):
        if self.h:
            moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def sizes(self, T):
        return moe_workspace_size(self.h, T)

    def buffer(self, name, nbytes):
        b = self._ws.get(name)
        if b is None or b.numel() < nbytes:
            b = _bytes(nbytes, self.device)
            self._ws[name] = b
        return b

    def set_weights(self, Wr, b, Wg, Wu, Wd, stream=None):
        self.packed = _bytes(self.sizes(1)["packed"], self.device)
        moe_set_weights(self.h, Wr, b, Wg, Wu, Wd, self.packed, stream)

    def new_ctx(self, T):
        return _bytes(self.sizes(T)["ctx"], self.device)

    def forward(self, x, y=None, ctx=None, stream=None):
        T = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        ws = self.buffer("fwd", self.sizes(T)["fwd_ws"])
        moe_forward(self.h, x, T, y, ctx, ws, stream)
        return y

    def backward(self, x, dy, ctx, stream=None):
        T, d = x.shape
        S, E, f = self.shape["S"], self.shape["E"], self.shape["f"]
        wdt = torch.float32 if self.prec == "fp32" else torch.bfloat16
        dx = torch.empty_like(x)
        dWr = torch.empty((E, d), dtype=torch.float32, device=self.device)
        dWg = torch.empty((E + S, f, d), dtype=wdt, device=self.device)
        dWu = torch.empty((E + S, f, d), dtype=wdt, device=self.device)
        dWd = torch.empty((E + S, d, f), dtype=wdt, device=self.device)
        ws = self.buffer("bwd", self.sizes(T)["bwd_ws"])
        moe_backward(self.h, x, dy, T, ctx, dx, dWr, dWg, dWu, dWd, ws, stream)
        return dict(dx=dx, dWr=dWr, dWg=dWg, dWu=dWu, dWd=dWd)

    def grads_like(self, x):
        T, d = x.shape
        S, E, f = self.shape["S"], self.shape["E"], self.shape["f"]
        wdt = torch.float32 if self.prec == "fp32" else torch.bfloat16
        return dict(dx=torch.empty_like(x), dWr=torch.empty((E, d), dtype=torch.float32, device=self.device),
                    dWg=torch.empty((E + S, f, d), dtype=wdt, device=self.device),
                    dWu=torch.empty((E + S, f, d), dtype=wdt, device=self.device),
                    dWd=torch.empty((E + S, d, f), dtype=wdt, device=self.device))

    def train_chunked(self, x, dy, slots, stream=None):
        """Chunked forward + backward with a ring of `slots` activation slots."""
        T = x.shape[0]
        z = moe_train_chunked_sizes(self.h, T)
        ring = self.buffer("ring", z["slot"] * slots)
        ws = self.buffer("chunk_ws", z["workspace"])
        out = self.grads_like(x)
        out["y"] = torch.empty_like(x)
        out["recomputed"] = moe_train_chunked(self.h, x, dy, T, out["y"], out["dx"], out["dWr"], out["dWg"],
                                              out["dWu"], out["dWd"], ring, z["slot"] * slots, ws, stream)
        out["n_chunks"] = z["n_chunks"]
        return out

    def route(self, x=None, T=None, logits_override=None, stream=None):
        T = T if T is not None else x.shape[0]
        E, k = self.shape["E"], self.shape["k"]
        dev = self.device
        out = dict(logits=torch.empty((T, E), dtype=torch.float32, device=dev),
                   idx=torch.empty((T, k), dtype=torch.int32, device=dev),
                   gate=torch.empty((T, k), dtype=torch.float32, device=dev),
                   cnt=torch.empty(E, dtype=torch.int32, device=dev),
                   off=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   perm=torch.empty(T * k, dtype=torch.int32, device=dev),
                   inv=torch.empty(T * k, dtype=torch.int32, device=dev))
        ws = self.buffer("fwd", self.sizes(T)["fwd_ws"])
        moe_route(self.h, x, T, logits_override, out["logits"], out["idx"], out["gate"], out["cnt"], out["off"],
                  out["perm"], out["inv"], ws, stream)
        return out

    def decode(self, x, y=None, stream=None):
        B = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        ws = self.buffer("fwd", self.sizes(max(B, 1))["fwd_ws"])
        moe_decode(self.h, x, B, y, ws, stream)
        return y

    def status(self, stream=None) -> int:
        return moe_get_status(self.h, stream)
