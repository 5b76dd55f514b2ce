"""Calibrate the Zipf routing-bias strength beta with the oracle; writes zipf_beta.json.

The skewed-routing workloads add a selection-only bias b_e = -1.1 * beta * ln(r_e)
(r_e = a seeded popularity rank) to the sigmoid router scores.  beta is chosen by
bisection so that, over a seeded sample of 16,384 full-size tokens (H 4096,
E 288, top-8), the least-squares slope of log(pick count) against log(count rank)
is -1.10 (Zipf s = 1.1).  Only ``oracle/`` and the input generator are called.

Run from the repository root:  python tests/golden/make_zipf_beta.py
"""

from __future__ import annotations

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402
from oracle import moe  # noqa: E402

H, E, K, T = 4096, 288, 8, 16384
TARGET = -synthetic.ZIPF_S


def slope_for(scores: np.ndarray, ranks: np.ndarray, beta: float) -> tuple[float, np.ndarray]:
    bias = -synthetic.ZIPF_S * beta * np.log(ranks.astype(np.float64))
    sel = scores + bias[None, :]
    order = np.argsort(-sel, axis=1, kind="stable")[:, :K]
    counts = np.bincount(order.reshape(-1), minlength=E)
    c = np.sort(counts)[::-1]
    c = c[c > 0]
    r = np.arange(1, c.size + 1)
    slope = np.polyfit(np.log(r), np.log(c), 1)[0]
    return float(slope), counts


def main() -> None:
    x = moe.bf16_bits_to_f64(synthetic.activations_bits(T, H, seed=0, layer=0, step=10_000))
    wr = synthetic.router_weights(E, H, seed=0, layer=0)
    scores = moe.sigmoid(moe.router_logits(x, wr))
    ranks = synthetic.popularity_ranks(E, seed=0, layer=0)
    lo, hi = 0.0, 2.0
    s_hi, _ = slope_for(scores, ranks, hi)
    assert s_hi < TARGET, f"upper bracket too small: slope {s_hi}"
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        s, _ = slope_for(scores, ranks, mid)
        if s > TARGET:
            lo = mid
        else:
            hi = mid
    beta = 0.5 * (lo + hi)
    slope, counts = slope_for(scores, ranks, beta)
    # Unique experts per step at the batch sizes of the decode workloads.
    bias = -synthetic.ZIPF_S * beta * np.log(ranks.astype(np.float64))
    top = np.argsort(-(scores + bias[None, :]), axis=1, kind="stable")[:, :K]
    uniq = {}
    for b in (1, 4, 8):
        n = (T // b) * b
        u = [np.unique(top[i:i + b]).size for i in range(0, n, b)]
        uniq[str(b)] = float(np.mean(u))
    host_mass = float(counts[np.argsort(ranks)][188:].sum() / counts.sum())
    out = {
        "beta": beta,
        "fitted_slope": slope,
        "target_slope": TARGET,
        "sample": {"tokens": T, "hidden": H, "experts": E, "top_k": K, "seed": 0, "layer": 0, "step": 10000},
        "mean_unique_experts_per_step": uniq,
        "pick_share_of_ranks_189_288": host_mass,
        "pick_counts_by_expert": counts.tolist(),
        "written_by": "tests/golden/make_zipf_beta.py (oracle only)",
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "zipf_beta.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps({k: v for k, v in out.items() if k != "pick_counts_by_expert"}, indent=1))


if __name__ == "__main__":
    main()
