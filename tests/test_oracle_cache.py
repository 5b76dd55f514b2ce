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
