"""Writes ``zipf_bias_mixtral.txt``: the gate bias of the imbalanced-load
Mixtral-shaped workload (T=8192, H=4096, E=8, top-2, seed 0).

Routing is pushed toward Zipf(s=1.2) expert popularity, the imbalanced
expert load the COMET page tests robustness under ("COMET's Performance",
"Robustness"). Expert e (0 hottest) gets the target share
p_e = (e+1)^-1.2 / sum_e' (e'+1)^-1.2 of the T*k assignments. The bias is
found by the fixed-point iteration b <- b + 0.5 (ln p_target - ln p_observed),
50 rounds from b = 0, where p_observed comes from the oracle's top-k on the
oracle's canonical fp32 logits plus b (one fp32 add, as in the layer).

Only the oracle and the seeded input generator are called.
Run from the repository root: python tests/golden/make_zipf_bias.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle.oracle import Oracle  # noqa: E402
from token_dispatch_grouped_moe_gb300.inputs import bf16_bits, make_inputs  # noqa: E402

T, H, E, K, S, SEED, ROUNDS = 8192, 4096, 8, 2, 1.2, 0, 50
OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "zipf_bias_mixtral.txt")


def main():
    O = Oracle()
    inp = make_inputs(T, H, 64, E, seed=SEED, only=("x", "Wg"))
    logits = O.logits(bf16_bits(inp["x"]), bf16_bits(inp["Wg"]))
    target = (np.arange(1, E + 1, dtype=np.float64)) ** -S
    target /= target.sum()
    b = np.zeros(E, np.float32)
    for _ in range(ROUNDS):
        idx, _ = O.topk(logits + b[None, :], K)
        share = np.bincount(idx.reshape(-1), minlength=E) / (T * K)
        b = (b + 0.5 * (np.log(target) - np.log(np.maximum(share, 1e-9)))).astype(np.float32)
    idx, _ = O.topk(logits + b[None, :], K)
    share = np.bincount(idx.reshape(-1), minlength=E) / (T * K)
    with open(OUT, "w") as f:
        f.write("# gate bias (f32) for the Zipf(1.2) Mixtral-shaped workload; written by\n")
        f.write("# make_zipf_bias.py (oracle only). One value per expert, as float.hex.\n")
        f.write("# target shares: " + " ".join(f"{p:.4f}" for p in target) + "\n")
        f.write("# achieved shares: " + " ".join(f"{p:.4f}" for p in share) + "\n")
        for v in b:
            f.write(float(v).hex() + "\n")
    print("target  ", np.round(target, 4))
    print("achieved", np.round(share, 4))


if __name__ == "__main__":
    main()
