"""Pins for the expert-cache policy replay oracle (CPU only)."""

import json
import os

import numpy as np
import pytest

import synthetic
from oracle import cache as ocache
from oracle import moe as omoe

from conftest import GOLDEN


def _fx():
    with open(os.path.join(GOLDEN, "cache_trace_tiny.json")) as f:
        return json.load(f)


def test_lfu_hand_derived_trace():
    fx = _fx()
    r = ocache.lfu_replay(fx["trace"], 6, fx["static"], fx["n_slots"], decay=fx["decay"])
    assert [[list(a) for a in call] for call in r["admitted"]] == fx["lfu_admitted"]
    assert r["slot_expert"] == fx["lfu_final_slots"]
    np.testing.assert_array_equal(r["scores"], np.array(fx["lfu_final_scores"], np.float32))
    assert r["misses"] == fx["lfu_misses"]


def test_static_hand_derived_trace():
    fx = _fx()
    assert ocache.static_replay(fx["trace"], fx["static_resident"])["misses"] == fx["static_misses"]


def _zipf_trace(n_calls, T, E=64, k=4, seed=0):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    perm = rng.permutation(E)
    trace = []
    for _ in range(n_calls):
        picks = set()
        for _ in range(T):
            picks |= set(perm[rng.choice(E, size=k, replace=False, p=p)].tolist())
        trace.append(sorted(picks))
    return trace


@pytest.mark.parametrize("slots", [4, 12, 30])
def test_belady_is_a_lower_bound(slots):
    trace = _zipf_trace(300, T=2)
    b = ocache.belady_replay(trace, [], slots)["misses"]
    assert b <= ocache.lru_replay(trace, [], slots)["misses"]
    assert b <= ocache.lfu_replay(trace, 64, [], slots)["misses"]
    assert b <= ocache.static_replay(trace, range(slots))["misses"]


def test_cache_never_holds_duplicates_or_statics():
    trace = _zipf_trace(200, T=4)
    static = [0, 5, 9]
    r = ocache.lfu_replay(trace, 64, static, 16)
    live = [e for e in r["slot_expert"] if e >= 0]
    assert len(live) == len(set(live)) and not set(live) & set(static)
    for call, adm in zip(trace, r["admitted"]):
        assert all(e in call and e not in static for e, _, _ in adm)
        assert all(old not in call for _, _, old in adm)


def test_lfu_without_decay_keeps_the_most_frequent():
    """decay = 1: after a long trace the slots hold experts with the largest
    counts among those that ever missed last (a frequency cache)."""
    trace = [[0], [1], [0], [2], [0], [1], [3]] * 5
    r = ocache.lfu_replay(trace, 4, [], 2, decay=1.0)
    counts = {e: sum(e in c for c in trace) for e in range(4)}
    np.testing.assert_array_equal(r["scores"], np.array([counts[e] for e in range(4)], np.float32))
    assert 0 in r["slot_expert"]


def test_infinite_cache_misses_once_per_expert():
    trace = _zipf_trace(100, T=4)
    first = len(set(e for c in trace for e in c))
    assert ocache.lfu_replay(trace, 64, [], 64)["misses"] == first
    assert ocache.lru_replay(trace, [], 64)["misses"] == first
    assert ocache.belady_replay(trace, [], 64)["misses"] == first


def test_lfu_admission_cap_hand_derived():
    """At most max_admit admissions per call; later misses of the call stay on the host tier."""
    fx = _fx()
    c = fx["capped"]
    r = ocache.lfu_replay(fx["trace"], 6, fx["static"], fx["n_slots"], decay=fx["decay"], max_admit=c["max_admit"])
    assert [[list(a) for a in call] for call in r["admitted"]] == c["admitted"]
    assert r["bypassed"] == c["bypassed"]
    assert r["slot_expert"] == c["final_slots"]
    np.testing.assert_array_equal(r["scores"], np.array(c["final_scores"], np.float32))
    assert r["misses"] == c["misses"]


def _pol():
    with open(os.path.join(GOLDEN, "cache_policies_tiny.json")) as f:
        return json.load(f)


def test_lru_hand_derived_trace():
    fx = _pol()["lru"]
    r = ocache.lru_replay(fx["trace"], [], fx["n_slots"])
    assert [[list(a) for a in call] for call in r["admitted"]] == fx["admitted"]
    assert r["slot_expert"] == fx["final_slots"]
    assert r["misses"] == fx["misses"]


def test_belady_hand_derived_trace():
    fx = _pol()["belady"]
    r = ocache.belady_replay(fx["trace"], [], fx["n_slots"])
    assert [[list(a) for a in call] for call in r["admitted"]] == fx["admitted"]
    assert r["slot_expert"] == fx["final_slots"]
    assert r["misses"] == fx["misses"]
    assert ocache.lru_replay(fx["trace"], [], fx["n_slots"])["misses"] == fx["lru_misses"]


def test_belady_brute_force_optimum_on_tiny_traces():
    """Belady's miss count is the minimum over every eviction choice (exhaustive
    search on short random traces with one expert per call)."""
    rng = np.random.default_rng(11)

    def best(trace, slots, i=0):
        if i == len(trace):
            return 0
        e = trace[i]
        if e in slots:
            return best(trace, slots, i + 1)
        if len(slots) < 2:
            return 1 + best(trace, slots | {e}, i + 1)
        return 1 + min(best(trace, (slots - {v}) | {e}, i + 1) for v in slots)

    for _ in range(30):
        trace = [int(v) for v in rng.integers(0, 5, size=9)]
        got = ocache.belady_replay([[e] for e in trace], [], 2)["misses"]
        assert got == best(trace, frozenset())


def test_policy_report_is_reproducible_and_consistent():
    """tests/golden/policy_misses.json: a recomputed slice equals the stored one,
    Belady is the lowest of the four everywhere, and the per-token figures follow
    from the counts."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_policy_misses", os.path.join(GOLDEN, "make_policy_misses.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(GOLDEN, "policy_misses.json")) as f:
        rep = json.load(f)
    for name in mod.WORKLOADS:
        assert mod.policy_misses(name, range(2), 16)["per_layer"] == rep["check"][name]
        w = rep["workloads"][name]
        assert w["layers"] == 42 and len(w["per_layer"]) == 42
        for layer in w["per_layer"]:
            for pol in ("static", "lru", "lfu_0.995"):
                assert layer["belady"] <= layer[pol]
        for pol, v in w["policies"].items():
            assert v["misses"] == sum(layer[pol] for layer in w["per_layer"])
            assert v["misses_per_token"] == pytest.approx(v["misses"] / (w["steps"] * w["tokens_per_step"]), abs=1e-3)
