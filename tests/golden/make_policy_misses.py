"""Expert-cache policies replayed over seeded full-size routing traces; writes policy_misses.json.

The RTX PRO 6000 recipe (``config.expert_cache.policy_data``) compares the
misses per token of four placements of the routed experts over replayed
routing traces: a static hot set, LRU, LFU with a 0.995 decay, and Belady's
offline optimum.  Its traces are not published, so this script builds its own
from the seeded synthetic inputs of the two skewed-routing workloads and the
oracle router, and replays the oracle's four policies over them.

Traces.  For each of the 42 layers of a workload (T tokens per decode step,
H 4096, E 288, top-8, the layer's Zipf(1.1) selection bias) and each step j,
the step's tokens are ``synthetic.activations_bits(T, 4096, seed 0, layer,
step j)``, routed by ``oracle.moe.route``; the call is the union of their picks.

Cache layout (the expert-cache workload's, per layer): popularity ranks 1-40
are static (always resident), 148 slots are managed by the policy and start out
holding ranks 41-188, the other experts live in host memory.  ``static`` keeps
ranks 1-188 resident for good.  A miss is an expert a call uses that is neither
static nor in a slot at the time of the call.

Reported per workload and policy: misses, misses per layer-call, misses per
token summed over the 42 layers (misses / (steps * T)), and the host-link bytes
per token those misses move (misses x 12,976,128 B per expert).  Only
``oracle/`` and the input generator are called.

Run from the repository root:  python tests/golden/make_policy_misses.py
"""

from __future__ import annotations

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402
from oracle import cache as ocache  # noqa: E402
from oracle import moe as omoe  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "policy_misses.json")
N_STATIC, N_SLOTS, DECAY = 40, 148, 0.995
EXPERT_BYTES = 12_976_128
STEPS = 256
WORKLOADS = ("decode8_zipf_x42", "cache4_x42")


def layer_trace(name: str, layer: int, steps: int) -> list:
    """Expert unions of `steps` decode steps of one layer of a workload."""
    cfg = synthetic.CONFIGS[name]
    wr = synthetic.router_weights(cfg.n_experts, cfg.hidden, cfg.seed, layer)
    bias = synthetic.zipf_bias(cfg.n_experts, cfg.seed, layer)
    x = np.concatenate([omoe.bf16_bits_to_f64(synthetic.activations_bits(cfg.tokens, cfg.hidden, cfg.seed, layer, j))
                        for j in range(steps)])
    idx = omoe.route(x, wr, bias, cfg.top_k)["idx"].reshape(steps, cfg.tokens * cfg.top_k)
    return [sorted(set(int(e) for e in row)) for row in idx]


def layer_misses(name: str, layer: int, steps: int) -> dict:
    """Misses of each policy over one layer's trace."""
    cfg = synthetic.CONFIGS[name]
    E = cfg.n_experts
    trace = layer_trace(name, layer, steps)
    ranks = synthetic.popularity_ranks(E, cfg.seed, layer)
    by_rank = np.argsort(ranks)                      # expert of rank r + 1
    static = [int(e) for e in by_rank[:N_STATIC]]
    init = [int(e) for e in by_rank[N_STATIC:N_STATIC + N_SLOTS]]
    return {
        "static": ocache.static_replay(trace, static + init)["misses"],
        "lru": ocache.lru_replay(trace, static, N_SLOTS, init_slots=init)["misses"],
        "lfu_0.995": ocache.lfu_replay(trace, E, static, N_SLOTS, decay=DECAY, init_slots=init)["misses"],
        "belady": ocache.belady_replay(trace, static, N_SLOTS, init_slots=init)["misses"],
        "unique_experts": sum(len(c) for c in trace),
    }


def policy_misses(name: str, layers, steps: int) -> dict:
    cfg = synthetic.CONFIGS[name]
    per_layer = [layer_misses(name, layer, steps) for layer in layers]
    out = {"tokens_per_step": cfg.tokens, "layers": len(per_layer), "steps": steps,
           "unique_experts_per_call": round(sum(p["unique_experts"] for p in per_layer) / (len(per_layer) * steps), 3),
           "per_layer": per_layer, "policies": {}}
    for pol in ("static", "lru", "lfu_0.995", "belady"):
        m = sum(p[pol] for p in per_layer)
        out["policies"][pol] = {
            "misses": m,
            "misses_per_layer_call": round(m / (len(per_layer) * steps), 4),
            "misses_per_token": round(m / (steps * cfg.tokens), 3),
            "host_bytes_per_token": int(round(m * EXPERT_BYTES / (steps * cfg.tokens))),
        }
    return out


def main() -> None:
    result = {
        "what": "Misses of four expert placements over seeded full-size routing traces (oracle router, Zipf(1.1) "
                "bias, 42 layers); layout per layer: 40 static + 148 policy slots (initially ranks 41-188), "
                "the rest in host memory",
        "script": "tests/golden/make_policy_misses.py",
        "expert_bytes": EXPERT_BYTES,
        "workloads": {name: policy_misses(name, range(synthetic.CONFIGS[name].layers), STEPS) for name in WORKLOADS},
        # a small slice the tests recompute to tie this file to the code that wrote it
        "check": {name: policy_misses(name, range(2), 16)["per_layer"] for name in WORKLOADS},
    }
    with open(OUT, "w") as f:
        json.dump(result, f, indent=1)
        f.write("\n")
    for name, w in result["workloads"].items():
        print(name, {p: v["misses_per_token"] for p, v in w["policies"].items()})


if __name__ == "__main__":
    main()
