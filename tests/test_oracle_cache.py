"""Pins of the expert-cache policy oracle (oracle/cache.py).

The policy is least-recently-used eviction (the K3-Stuff model page,
"llama-cpp-patches", change 2: the page cache as the hot-expert cache), with
every expert of a call used at the same moment.  Checked against a library
LRU cache, a recency-only statement of the resident set, a hand-worked
sequence and invariants.
"""
import functools

import numpy as np
import pytest

from oracle.cache import CacheState, cache_call, lru_resident


def resident(st):
    return {e for e in st.expert_of if e >= 0}


def test_one_expert_per_call_is_textbook_lru():
    """One expert per call: hits and misses are those of functools.lru_cache."""
    rng = np.random.default_rng(1)
    for S, E in ((1, 5), (3, 8), (7, 20), (16, 64)):
        seq = rng.integers(0, E, 400)
        lib = functools.lru_cache(maxsize=S)(lambda e: e)
        st = CacheState.empty(E, S)
        for e in seq:
            lib(int(e))
            cache_call(st, [e])
        info = lib.cache_info()
        assert (st.hits, st.misses) == (info.hits, info.misses)


def test_resident_set_is_the_most_recently_used():
    """Batched calls: the resident set is the S most recently used experts
    (where recency alone decides it)."""
    rng = np.random.default_rng(2)
    checked = 0
    for S, E, kmax in ((4, 16, 4), (10, 40, 6), (32, 128, 16)):
        calls = [rng.choice(E, rng.integers(1, kmax + 1), replace=False) for _ in range(300)]
        st = CacheState.empty(E, S)
        for used, want in zip(calls, lru_resident(calls, S)):
            cache_call(st, used)
            if want is not None:
                assert resident(st) == want
                checked += 1
    assert checked > 300


def test_hand_worked_sequence():
    """S = 3 slots, the rule applied by hand:
    {0,1}: slots 0,1 (empty slots in order)          -> [0, 1, -1]
    {2}:   empty slot 2                              -> [0, 1, 2]
    {3}:   oldest stamps 1,1 (slots 0,1): slot 0     -> [3, 1, 2]  (evicts 0)
    {1,4}: 1 hits; oldest of slots 0 (3), 2 (2): 2   -> [3, 1, 4]  (evicts 2)
    {0,2,3}: 3 hits; victims slots 1,2 (stamp 4 each), 0 -> 1, 2 -> 2
                                                     -> [3, 0, 2]
    {3}, {0}: hits; stamps become [6, 7, 5]
    {5,6}: victims slot 2 (5) and slot 0 (6); in slot order 5 -> 0, 6 -> 2
                                                     -> [5, 0, 6]"""
    st = CacheState.empty(8, 3)
    want = [([0, 1, -1], 0, 2), ([0, 1, 2], 0, 1), ([3, 1, 2], 0, 1), ([3, 1, 4], 1, 1),
            ([3, 0, 2], 1, 2), ([3, 0, 2], 1, 0), ([3, 0, 2], 1, 0), ([5, 0, 6], 0, 2)]
    calls = [{0, 1}, {2}, {3}, {1, 4}, {0, 2, 3}, {3}, {0}, {5, 6}]
    for used, (slots, h, m) in zip(calls, want):
        r = cache_call(st, used)
        assert st.expert_of == slots
        assert (r["hits"], r["misses"]) == (h, m)
    assert (st.hits, st.misses, st.clock) == (4, 9, 8)
    assert st.stamp == [8, 7, 8]
    assert st.slot_of == [1, -1, -1, -1, -1, 0, 2, -1]


def test_invariants():
    rng = np.random.default_rng(3)
    E, S = 50, 12
    st = CacheState.empty(E, S)
    seen = set()
    for _ in range(500):
        used = set(rng.choice(E, rng.integers(1, S + 1), replace=False).tolist())
        before = resident(st)
        r = cache_call(st, used)
        seen |= used
        assert used <= resident(st)
        assert r["misses"] == len(used - before) and r["hits"] == len(used & before)
        assert len(resident(st)) == min(S, len(seen))
        slots = [v for _, v in r["fetched"]]
        assert len(set(slots)) == len(slots) == r["misses"]
        assert [e for e, _ in r["fetched"]] == sorted(used - before)
        assert slots == sorted(slots)
        for s, e in enumerate(st.expert_of):
            if e >= 0:
                assert st.slot_of[e] == s
        for e, s in enumerate(st.slot_of):
            if s >= 0:
                assert st.expert_of[s] == e
        # only experts not used by the call were evicted
        assert before - resident(st) <= before - used


def test_rejects_oversized_calls():
    st = CacheState.empty(10, 3)
    with pytest.raises(ValueError):
        cache_call(st, [0, 1, 2, 3])
    with pytest.raises(ValueError):
        CacheState.empty(3, 4)
