"""Writes the stored router selection-bias vectors for the Zipf-routed workloads.

The workloads ask for a router bias that makes the expert load follow a Zipf
law. Each stored vector is calibrated with the oracle's top-k selection on
synthetic logits that follow the router logits' law: with x ~ N(0, 1) and
Wr ~ N(0, 0.02^2), a token's logits x.Wr_e are, given x, independent
N(0, 0.02^2 |x|^2) ~ N(0, 0.0004 d) across experts.

Targets: T*k*p_e with p_e proportional to 1/(e+1)^s, clipped at one token per
expert per token and water-filled (moe_synth.zipf_targets). Calibration: 300
fixed steps of b_e += 0.5 (ln(target_e + 1) - ln(count_e + 1)), then b is
centred (selection is invariant to a common shift).

Run from the repository root:  python tests/golden/make_router_bias.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import moe_oracle as oracle  # noqa: E402
import moe_synth  # noqa: E402

CASES = [  # (E, k, d, s)
    (64, 6, 2048, 1.0),
    (256, 8, 7168, 1.2),
]
T_CAL = 8192
STEPS = 300


def calibrate(E, k, d, s, seed=12345):
    rng = np.random.Generator(np.random.PCG64(seed))
    sigma = 0.02 * np.sqrt(d)
    Z = (rng.standard_normal((T_CAL, E)) * sigma).astype(np.float32)
    tgt = np.array(moe_synth.zipf_targets(T_CAL, k, E, s))
    b = np.zeros(E, np.float64)
    for _ in range(STEPS):
        idx = oracle.select_experts(Z, b.astype(np.float32), k)
        cnt = oracle.expert_counts(idx, E)
        b += 0.5 * (np.log(tgt + 1.0) - np.log(cnt + 1.0))
    b -= b.mean()
    idx = oracle.select_experts(Z, b.astype(np.float32), k)
    cnt = oracle.expert_counts(idx, E)
    return b.astype(np.float32), cnt, tgt


def main():
    for E, k, d, s in CASES:
        b, cnt, tgt = calibrate(E, k, d, s)
        path = moe_synth.bias_file(E, k, d, s)
        with open(path, "w") as fh:
            fh.write(f"# router selection bias, E={E} k={k} d={d} zipf s={s}; "
                     f"written by tests/golden/make_router_bias.py\n")
            fh.write(f"# columns: bias  calibration-load  target-load  (calibration on {T_CAL} tokens)\n")
            for e in range(E):
                fh.write(f"{float(b[e])!r} {int(cnt[e])} {tgt[e]:.1f}\n")
        print(path, "max |load-target|/target:",
              float(np.max(np.abs(cnt - tgt) / np.maximum(tgt, 1))))


if __name__ == "__main__":
    main()
