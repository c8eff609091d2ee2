"""End-to-end routing agreement between the GPU and the oracle (test helper).

The selection is an integer decision taken on floating-point logits. Given the
same fp32 logits both sides select bit-identically (tested elsewhere through
moe_route's logits override). End to end, the GPU's logits come from its own
GEMM and differ from the oracle's float64 logits in the last bits, so a token
whose top-k keys are nearly tied may legitimately select differently. The
reading the tests take: compare the GPU's indices with the oracle's own
selection (from the oracle's logits rounded to fp32) wherever every gap among
the token's k+1 largest keys exceeds 4x the measured logit error; a mismatch
there is an "index exception" and must not happen. Tokens inside that margin
are near-ties: counted and reported, not compared.

Counts are reported as ParityReport warnings, which pytest lists in its
warnings summary even when the test passes.
"""
from __future__ import annotations

import warnings

import numpy as np

from oracle import moe_oracle as oracle


class ParityReport(UserWarning):
    """A measured parity figure (error, exception count) worth seeing in a passing run."""


def report(what: str, **figures):
    text = ", ".join(f"{k}={v:.3e}" if isinstance(v, float) else f"{k}={v}" for k, v in figures.items())
    warnings.warn(f"{what}: {text}", ParityReport, stacklevel=2)


def key_margins(logits32, bias, k: int):
    """Per token: the smallest gap between consecutive keys among its k+1 largest keys (fp32 keys,
    formed as the selection forms them). A gap above the logit error fixes the ordered top-k row."""
    key = oracle.selection_keys(logits32, bias).astype(np.float64)
    E = key.shape[1]
    m = min(k, E - 1)
    if m <= 0:
        return np.full(key.shape[0], np.inf)
    s = -np.sort(-key, axis=1)
    return (s[:, :m] - s[:, 1:m + 1]).min(axis=1)


def routing_exceptions(idx_gpu, logits_gpu, x, Wr, bias, k: int, err_floor: float = 0.0) -> dict:
    """Index exceptions of the GPU's selection against the oracle's own (see the module docstring).

    idx_gpu [T, k] and logits_gpu [T, E] come from the GPU; x [T, d], Wr [E, d] and bias [E] are the
    inputs both sides received. The logit error is measured over these T tokens (at least err_floor).
    """
    l_ref = oracle.router_logits(x, Wr)
    err = float(np.max(np.abs(np.asarray(logits_gpu, np.float64) - l_ref))) if logits_gpu is not None else 0.0
    err = max(err, err_floor)
    l32 = l_ref.astype(np.float32)
    ref_idx = oracle.select_experts(l32, bias, k)
    margin = key_margins(l32, bias, k)
    sure = margin > 4 * err
    differ = ~np.all(np.asarray(idx_gpu) == ref_idx, axis=1)
    return dict(tokens=int(len(margin)), logit_err=err, near_ties=int(np.count_nonzero(~sure)),
                exceptions=int(np.count_nonzero(sure & differ)),
                near_tie_disagreements=int(np.count_nonzero(~sure & differ)), sure=sure, ref_idx=ref_idx,
                logits_ref=l_ref)
