"""Seeded synthetic inputs for the single-GPU Mixture-of-Experts layer.

This module is shared by the CUDA path, the CPU oracle, the tests and the
bench. It draws inputs only: it holds none of the layer's arithmetic (no
routing, no expert math, no quantisation). Random draws use torch generators
so that a full-size layer can be drawn directly on the GPU; the CPU oracle
receives host copies of exactly the tensors the CUDA path receives.

Recipe (the pages print no shapes or distributions; these follow the stated
workload table and are listed with their readings in the design notes):
  x ~ N(0, 1)               [T, d]
  Wr ~ N(0, 0.02^2)          [E, d]        router weight
  Wg, Wu ~ N(0, 1/d)         [E+S, f, d]   gate / up projections (rows = outputs)
  Wd ~ N(0, 1/d)             [E+S, d, f]   down projection
  dy ~ N(0, 1)               [T, d]        upstream gradient
  b                          [E]           router selection bias: 0 for uniform
                                           routing, else a stored vector that makes
                                           the expert load follow a clipped Zipf law
Shared expert, when present, is slot E of the expert weights.
Tensors are rounded to bf16 for the bf16 and mxfp8 workloads (the mxfp8 path
quantises those same bf16 values itself) and kept fp32 for the fp32 workload.
"""
from __future__ import annotations

import dataclasses
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
BIAS_DIR = os.path.join(_HERE, "tests", "golden")


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """Shape and router of one MoE layer workload."""
    name: str
    T: int              # tokens
    d: int              # hidden size
    E: int              # routed experts
    S: int              # shared experts (0 or 1)
    f: int              # SwiGLU intermediate width
    k: int              # experts per token
    router: str         # "softmax" or "sigmoid"
    renorm: bool        # renormalise gates over the k selected experts
    route_scale: float  # multiplies routed gates (sigmoid router)
    dtype: str          # "fp32", "bf16" or "mxfp8"
    zipf_s: float | None  # None: uniform routing (b = 0)
    seed: int
    chunk: int = 0      # tokens per chunk for the chunked fwd+bwd (0: one chunk)

    def with_(self, **kw) -> "LayerSpec":
        return dataclasses.replace(self, **kw)

    @property
    def A(self) -> int:
        return self.T * self.k


TINY_FP32 = LayerSpec("tiny_fp32_T64_d256_E8_f128_top2", 64, 256, 8, 0, 128, 2,
                      "softmax", True, 1.0, "fp32", None, 0)
BF16_T2048 = LayerSpec("bf16_T2048_d2048_E64_f1408_top6_zipf1.0", 2048, 2048, 64, 0, 1408, 6,
                       "softmax", True, 1.0, "bf16", 1.0, 1)
DSV3_UNIFORM = LayerSpec("dsv3_bf16_T8192_d7168_E256+1_f2048_top8_uniform", 8192, 7168, 256, 1,
                         2048, 8, "sigmoid", True, 2.5, "bf16", None, 2)
DSV3_ZIPF = DSV3_UNIFORM.with_(name="dsv3_bf16_T8192_d7168_E256+1_f2048_top8_zipf1.2",
                               zipf_s=1.2, seed=3)
DSV3_MXFP8 = DSV3_UNIFORM.with_(name="dsv3_mxfp8_T8192_d7168_E256+1_f2048_top8_chunk2368",
                                dtype="mxfp8", seed=4, chunk=2368)


def decode_spec(B: int) -> LayerSpec:
    return DSV3_UNIFORM.with_(name=f"dsv3_bf16_decode_B{B}", T=B, seed=5)


WORKLOADS = {s.name: s for s in (TINY_FP32, BF16_T2048, DSV3_UNIFORM, DSV3_ZIPF, DSV3_MXFP8,
                                 decode_spec(1), decode_spec(4), decode_spec(16))}


def bias_file(E: int, k: int, d: int, s: float) -> str:
    return os.path.join(BIAS_DIR, f"router_bias_E{E}_k{k}_d{d}_zipf{s}.txt")


def load_bias(spec: LayerSpec) -> torch.Tensor:
    """Router selection bias [E] fp32: zeros for uniform routing, else the stored vector."""
    if spec.zipf_s is None:
        return torch.zeros(spec.E, dtype=torch.float32)
    path = bias_file(spec.E, spec.k, spec.d, spec.zipf_s)
    with open(path) as fh:
        vals = [float(line.split()[0]) for line in fh if line.strip() and not line.startswith("#")]
    if len(vals) != spec.E:
        raise ValueError(f"{path}: expected {spec.E} values, found {len(vals)}")
    return torch.tensor(vals, dtype=torch.float32)


def _storage_dtype(spec: LayerSpec) -> torch.dtype:
    return torch.float32 if spec.dtype == "fp32" else torch.bfloat16


def _normal(gen: torch.Generator, shape, std: float, dtype: torch.dtype, device) -> torch.Tensor:
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def make_inputs(spec: LayerSpec, device="cpu", *, weights: bool = True, grad: bool = False,
                seed_offset: int = 0) -> dict:
    """Draw one layer's inputs with a seeded generator on `device`.

    Returns a dict of torch tensors: x, Wr, b, and (weights=True) Wg, Wu, Wd
    stacked as [E+S, ...]; (grad=True) dy. Expert weights are drawn one expert
    at a time so that a full-size layer never holds an fp32 copy of all weights.
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1_000_003 * spec.seed + seed_offset)
    dt = _storage_dtype(spec)
    T, d, E, S, f = spec.T, spec.d, spec.E, spec.S, spec.f
    out = {"x": _normal(gen, (T, d), 1.0, dt, dev),
           "Wr": _normal(gen, (E, d), 0.02, dt, dev),
           "b": load_bias(spec).to(dev)}
    if weights:
        wstd = 1.0 / d ** 0.5
        Wg = torch.empty((E + S, f, d), dtype=dt, device=dev)
        Wu = torch.empty((E + S, f, d), dtype=dt, device=dev)
        Wd = torch.empty((E + S, d, f), dtype=dt, device=dev)
        for e in range(E + S):
            Wg[e] = _normal(gen, (f, d), wstd, dt, dev)
            Wu[e] = _normal(gen, (f, d), wstd, dt, dev)
            Wd[e] = _normal(gen, (d, f), wstd, dt, dev)
        out.update(Wg=Wg, Wu=Wu, Wd=Wd)
    if grad:
        out["dy"] = _normal(gen, (T, d), 1.0, dt, dev)
    return out


def make_tokens(spec: LayerSpec, n_batches: int, device="cpu", seed_offset: int = 7) -> torch.Tensor:
    """n_batches independent token batches [n_batches, T, d] drawn with their own seed."""
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(1_000_003 * spec.seed + seed_offset)
    return _normal(gen, (n_batches, spec.T, spec.d), 1.0, _storage_dtype(spec), device)


def zipf_targets(T: int, k: int, E: int, s: float) -> list[float]:
    """Per-expert token loads T*k*p_e with p_e proportional to 1/(e+1)^s, clipped at T.

    No expert can receive more than T tokens (each token picks k distinct
    experts), so the excess of a clipped expert is water-filled over the others
    in proportion to their loads until no load exceeds T. Expert e has Zipf rank e.
    """
    w = [1.0 / (e + 1) ** s for e in range(E)]
    tot = sum(w)
    tgt = [T * k * wi / tot for wi in w]
    clipped = [False] * E
    while True:
        excess = sum(t - T for t in tgt if t > T)
        if excess <= 1e-9:
            return tgt
        for e in range(E):
            if tgt[e] > T:
                tgt[e] = float(T)
                clipped[e] = True
        free = sum(tgt[e] for e in range(E) if not clipped[e])
        for e in range(E):
            if not clipped[e]:
                tgt[e] += excess * tgt[e] / free
