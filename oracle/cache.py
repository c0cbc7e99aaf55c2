"""Expert cache policy (test infrastructure only; see the package docstring).

Sources:

* The K3-Stuff model page, "llama-cpp-patches", change 2: the model runs with
  less memory than its size when the operating system's page cache serves as
  the hot-expert cache - experts are faulted in when first used and the
  least recently used pages are evicted.
* Lucebox PR #573 "feat(kimi-k3): add DSpark Q8 artifact and shared
  speculative runtime", "Runtime validation": routed experts read from SSD
  behind an 8 GiB device expert cache, with verification batched per route
  (the experts of a whole batch of draft tokens fetched together).

Reading (the pages name the policy, least recently used, but fix no slot
granularity): a cache of ``S`` expert slots serves a sequence of calls; each
call uses a SET of experts (the union of its tokens' selections) and every
expert of the set counts as used at the same moment, the call's number
``clock`` (1, 2, ...).  Used experts already resident are hits and their
slot's stamp becomes ``clock``.  Each missing expert needs a slot: the
victims are the slots not used by this call with the oldest stamps (a slot
never used has stamp 0), equal stamps taken in ascending slot order; the
i-th missing expert in ascending expert order takes the i-th victim in
ascending SLOT order.  The evicted expert (if any) leaves the cache.  A
call never uses more experts than there are slots.

The simulation is a plain loop over slots; ``lru_resident`` states the same
policy without slots (what is resident after each call), which is what the
tests pin against a textbook LRU (functools.lru_cache) in the one-expert-per-
call case.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass
class CacheState:
    E: int
    S: int
    clock: int = 0
    slot_of: list = field(default_factory=list)    # [E] slot or -1
    expert_of: list = field(default_factory=list)  # [S] expert or -1
    stamp: list = field(default_factory=list)      # [S] clock of last use, 0 = never
    hits: int = 0
    misses: int = 0

    @classmethod
    def empty(cls, E: int, S: int) -> "CacheState":
        if not 1 <= S <= E:
            raise ValueError("need 1 <= S <= E")
        return cls(E=E, S=S, slot_of=[-1] * E, expert_of=[-1] * S, stamp=[0] * S)


def cache_call(state: CacheState, used) -> dict:
    """One call using the experts ``used`` (any iterable; duplicates count
    once).  Updates ``state`` in place and returns the call's hits, misses and
    the (expert, slot) pairs fetched, in fetch order."""
    used = sorted(set(int(e) for e in used))
    if len(used) > state.S:
        raise ValueError("a call uses more experts than the cache holds")
    for e in used:
        if not 0 <= e < state.E:
            raise ValueError("expert out of range")
    state.clock += 1
    clock = state.clock
    hits = [e for e in used if state.slot_of[e] >= 0]
    missing = [e for e in used if state.slot_of[e] < 0]
    for e in hits:
        state.stamp[state.slot_of[e]] = clock
    # candidate slots: not used by this call; oldest stamp first, then slot index
    candidates = [s for s in range(state.S) if state.stamp[s] != clock]
    by_age = sorted(candidates, key=lambda s: (state.stamp[s], s))
    victims = sorted(by_age[:len(missing)])
    fetched = []
    for e, v in zip(missing, victims):
        old = state.expert_of[v]
        if old >= 0:
            state.slot_of[old] = -1
        state.expert_of[v] = e
        state.slot_of[e] = v
        state.stamp[v] = clock
        fetched.append((e, v))
    state.hits += len(hits)
    state.misses += len(missing)
    return {"hits": len(hits), "misses": len(missing), "fetched": fetched}


def lru_resident(calls, S: int):
    """The resident set after each call, from recency alone: the experts of
    the last call, then the most recently used others until S are held (among
    experts last used in the same call, which of them stays is left to slot
    order, so this returns None for a call where that choice matters)."""
    last_use = {}
    out = []
    for n, used in enumerate(calls, start=1):
        for e in set(int(x) for x in used):
            last_use[e] = n
        ranked = sorted(last_use.items(), key=lambda kv: -kv[1])
        if len(ranked) <= S:
            out.append(set(last_use))
            continue
        cut = ranked[S - 1][1]
        if ranked[S][1] == cut:  # a tie at the boundary: slot order decides
            out.append(None)
        else:
            out.append({e for e, _ in ranked[:S]})
    return out
