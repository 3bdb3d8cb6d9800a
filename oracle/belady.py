"""Offline reference for the eviction policies (test infrastructure only).

The slot table has to pick a victim without knowing the future. This module
replays an adapter trace with the future known: on a miss with no free slot it
evicts the resident adapter whose next use is farthest away (never used again
counts as infinitely far), the rule of Belady's MIN algorithm for demand
caching. The churn steps are cut into the same groups as the serving loop
(distinct adapters in first-appearance order, at most max_loras per group;
all of a group's adapters are resident at once, so none of them may be
evicted while the group is admitted). The hit count is the yardstick for the
LRU, pinned warm set and keep_score policies of the "Multi-LoRA
适配器缓存生产实战" page, section 为什么纯 LRU 在多租户场景下容易失效.
"""
from __future__ import annotations

import bisect


def groups_of(trace_steps, max_loras):
    """The trace as a list of groups (lists of adapter ids), in serving order."""
    out = []
    for ids in trace_steps:
        order = list(dict.fromkeys(int(a) for a in ids))
        for g in range(0, len(order), max_loras):
            out.append(order[g:g + max_loras])
    return out


def farthest_next_use(groups, max_loras):
    """Replay `groups` with the farthest-next-use rule.
    Returns (hits, misses, evictions)."""
    uses = {}
    for gi, grp in enumerate(groups):
        for a in grp:
            uses.setdefault(a, []).append(gi)

    def next_use(a, gi):
        u = uses[a]
        k = bisect.bisect_right(u, gi)
        return u[k] if k < len(u) else float("inf")

    resident = set()
    hits = misses = evictions = 0
    for gi, grp in enumerate(groups):
        members = set(grp)
        for a in grp:
            if a in resident:
                hits += 1
                continue
            misses += 1
            if len(resident) >= max_loras:
                victim = max((r for r in resident if r not in members),
                             key=lambda r: (next_use(r, gi), r))
                resident.remove(victim)
                evictions += 1
            resident.add(a)
    return hits, misses, evictions
