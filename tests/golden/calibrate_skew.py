"""Find the bias strength of the skewed workload.

The skewed workload is the DeepSeek-V3-shaped one (8192 tokens, 256 experts in
8 groups, top-4 groups then top-8 experts) with Zipf(1.2) expert popularity
over a seeded expert permutation folded into the selection bias:
bias[e] = N(0, 0.01) + beta * ln p(perm[e]),  p(i) ~ (i + 1)^-1.2.
This script bisects beta so that the hottest expert receives about 20x the
mean count (T*k/E) under the CPU oracle's gating, and prints the value that
``synth.SKEW_BETA`` holds.  It calls only ``oracle`` and ``synth``.

Run: python tests/golden/calibrate_skew.py
"""
import os
import sys

sys.path.insert(0, os.path.abspath(os.path.join(os.path.dirname(__file__), "..", "..")))

import oracle  # noqa: E402
import synth  # noqa: E402

TARGET = 20.0


def skew_ratio(beta, cfg=None):
    cfg = cfg or synth.config("skewed")
    scores = synth.make_scores(cfg)
    bias = synth.make_bias(cfg, beta=beta)
    idx, _ = oracle.gate(scores, bias, cfg["k"], cfg["n_groups"], cfg["topk_group"],
                         cfg["topk_in_group"], cfg["score_fn"], cfg["normalize"])
    lay = oracle.layout(idx, cfg["E"], cfg["experts_per_rank"])
    mean = cfg["T"] * cfg["k"] / cfg["E"]
    return lay["expert_count"].max() / mean


def main():
    lo, hi = 0.0, 1.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        if skew_ratio(mid) < TARGET:
            lo = mid
        else:
            hi = mid
    beta = round(0.5 * (lo + hi), 4)
    print("SKEW_BETA = %.4f  (max/mean = %.2f)" % (beta, skew_ratio(beta)))


if __name__ == "__main__":
    main()
