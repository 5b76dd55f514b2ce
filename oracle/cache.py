"""Oracle: expert-cache policies replayed over a trace of expert sets.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The RTX PRO 6000 recipe (``config.expert_cache.layout`` and ``.mechanism``)
keeps, per MoE layer, the most-routed experts static in VRAM, a set of VRAM
slots run as an LFU cache whose scores decay by 0.995 per call, and the rest in
pinned host memory; each miss takes the lowest-scoring slot that the current
call does not use.  Its ``policy_data`` compares static, LRU, LFU(0.995) and the
Belady bound on replayed traces.  This module replays a trace with each policy.

A trace is a list of calls; a call is the set of distinct experts one layer
uses in one decode step (the union of its tokens' picks).

Readings (the recipe states the rule in one sentence):
  * scores are fp32; per call every score is multiplied by ``decay`` (rounded to
    fp32), then 1 is added (rounded to fp32) for each expert the call uses;
  * misses are handled after the score update, in ascending expert id;
  * a miss takes the slot, among those whose expert the call does not use, with
    the lowest score of its current expert (an empty slot counts as -inf); ties
    go to the lowest slot index; if every slot holds an expert the call uses,
    the miss is served from host memory and nothing is admitted ("bypass");
  * LRU and Belady use the same candidate rule with their own victim key
    (oldest last use; farthest next use, never-again = +inf), ties to the
    lowest slot index;
  * the recipe's copy kernel moves the admitted experts of a call into their
    slots; a call admits at most ``max_admit`` experts (the capacity of its copy
    list), and a miss beyond that is served from host memory like a bypass, with
    the cache left as it was for that expert.
"""

from __future__ import annotations

import numpy as np


def _calls(trace):
    return [sorted(set(int(e) for e in c)) for c in trace]


def lfu_replay(trace, n_experts: int, static, n_slots: int, decay: float = 0.995, init_slots=None,
               init_scores=None, max_admit=None) -> dict:
    """LFU with multiplicative decay (fp32), the recipe's dynamic cache.

    Returns per-call lists of (expert, slot, evicted_expert) admissions, the
    bypassed misses, the final slot contents and scores.  ``max_admit`` (None =
    unlimited) caps the admissions of one call.
    """
    static = set(int(e) for e in static)
    slot_expert = [-1] * n_slots if init_slots is None else [int(e) for e in init_slots]
    assert len(slot_expert) == n_slots
    where = {e: s for s, e in enumerate(slot_expert) if e >= 0}
    scores = (np.zeros(n_experts, np.float32) if init_scores is None
              else np.asarray(init_scores, np.float32).copy())
    d = np.float32(decay)
    one = np.float32(1.0)
    admitted, bypassed, misses = [], [], 0
    for call in _calls(trace):
        scores = (scores * d).astype(np.float32)
        for e in call:
            scores[e] = np.float32(scores[e] + one)
        used = set(call)
        adm, byp = [], []
        for e in call:
            if e in static or e in where:
                continue
            misses += 1
            if max_admit is not None and len(adm) >= max_admit:
                byp.append(e)
                continue
            best = None
            for s, cur in enumerate(slot_expert):
                if cur in used:
                    continue
                key = -np.inf if cur < 0 else float(scores[cur])
                if best is None or key < best[0]:
                    best = (key, s)
            if best is None:
                byp.append(e)
                continue
            s = best[1]
            old = slot_expert[s]
            if old >= 0:
                del where[old]
            slot_expert[s] = e
            where[e] = s
            adm.append((e, s, old))
        admitted.append(adm)
        bypassed.append(byp)
    return {"admitted": admitted, "bypassed": bypassed, "misses": misses, "slot_expert": slot_expert,
            "scores": scores}


def lru_replay(trace, static, n_slots: int, init_slots=None) -> dict:
    """Least recently used: a miss evicts the candidate expert whose last use is
    oldest (an expert preloaded by ``init_slots`` and never used counts as used
    before the first call).  Returns per-call (expert, slot, evicted_expert)
    admissions, the misses and the final slot contents."""
    static = set(int(e) for e in static)
    slot_expert = [-1] * n_slots if init_slots is None else [int(e) for e in init_slots]
    last = {}
    misses = 0
    admitted = []
    for i, call in enumerate(_calls(trace)):
        used = set(call)
        adm = []
        for e in call:
            if e in static or e in slot_expert:
                continue
            misses += 1
            best = None
            for s, cur in enumerate(slot_expert):
                if cur in used:
                    continue
                key = -np.inf if cur < 0 else last.get(cur, -1)
                if best is None or key < best[0]:
                    best = (key, s)
            if best is not None:
                adm.append((e, best[1], slot_expert[best[1]]))
                slot_expert[best[1]] = e
        for e in call:
            last[e] = i
        admitted.append(adm)
    return {"misses": misses, "slot_expert": slot_expert, "admitted": admitted}


def belady_replay(trace, static, n_slots: int, init_slots=None) -> dict:
    """Offline optimum: a miss evicts the candidate expert whose next use lies
    farthest ahead (never again = +inf; an empty slot also counts as +inf).
    Returns per-call admissions, the misses and the final slot contents."""
    static = set(int(e) for e in static)
    calls = _calls(trace)
    slot_expert = [-1] * n_slots if init_slots is None else [int(e) for e in init_slots]
    uses = {}
    for i, c in enumerate(calls):
        for e in c:
            uses.setdefault(e, []).append(i)
    ptr = {e: 0 for e in uses}
    misses = 0
    admitted = []
    for i, call in enumerate(calls):
        used = set(call)
        adm = []
        for e in call:
            ptr[e] += 1          # the use at call i is consumed
        for e in call:
            if e in static or e in slot_expert:
                continue
            misses += 1
            best = None
            for s, cur in enumerate(slot_expert):
                if cur in used:
                    continue
                if cur < 0:
                    key = np.inf
                else:
                    u = uses.get(cur, [])
                    p = ptr.get(cur, 0)
                    key = u[p] if p < len(u) else np.inf
                if best is None or key > best[0]:
                    best = (key, s)
            if best is not None:
                adm.append((e, best[1], slot_expert[best[1]]))
                slot_expert[best[1]] = e
        admitted.append(adm)
    return {"misses": misses, "slot_expert": slot_expert, "admitted": admitted}


def static_replay(trace, resident) -> dict:
    resident = set(int(e) for e in resident)
    misses = sum(1 for c in _calls(trace) for e in c if e not in resident)
    return {"misses": misses}
