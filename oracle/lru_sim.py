"""Independent simulator of the GPU adapter slot table (test infrastructure only).

Semantics, as read from the "Multi-LoRA 适配器缓存生产实战" page:

* section 核心原理 (parameter table): ``max_loras`` bounds how many adapters one
  batch can use at once, i.e. the number of GPU slots.
* section 核心原理 (last paragraph): on a hit the adapter is touched (moved to
  most recent); when capacity is short the new adapter is validated first and
  then the oldest adapter by LRU is removed; an adapter in use by an executing
  task is never evicted.
* section 数据面: per-adapter residency fields (load_count, hit_count,
  eviction_count, inflight_requests).
* section 需要重点监控哪些指标, item 3: thrash ratio = reloads within a short
  window after eviction / total evictions.

* section 为什么纯 LRU 在多租户场景下容易失效: platform policies on top of
  LRU — a pinned warm set that low-priority traffic cannot push out, a cooling
  window (minimum residency) against short bursts, and a recency + frequency
  keep_score  w1 recent + w2 frequency + w3 priority + w4 reload_cost - w5 size.

A failed upload (the "load failed" outcome of a dynamic load on the "vLLM LoRA
Resolver 插件详解" page, section 6.1) is undone with ``abort_load`` while that
upload is pending (bound by a miss, no upload recorded since with ``loaded``):
the adapter is unbound; the adapter the assign evicted stays evicted;
references already taken stay until released, and the slot is free for a new
adapter only once none is left (so a late release can never lower the count
of an adapter bound there later).

Readings where the page is silent: the LRU clock is a counter that advances by
one on every touch or bind, so no two slots tie; a free slot (lowest index
first) is used before anything is evicted; the rank is validated before any
eviction, so a rejected adapter never costs a resident one its slot; the
thrash window is counted in caller-declared epochs (steps). For the policies:
a pinned slot is never a victim; the cooling window protects adapters whose
last access (hit or bind) is fewer than `min_residency` epochs old; keep_score
takes recent = 1 / (1 + epochs since the last access), frequency = accesses
(hits and binds) in the last `thrash_window` epochs, priority as set by the caller,
reload_cost = size = rank / max_lora_rank, and the lowest score is evicted,
ties going to the least recently used.
"""
from __future__ import annotations

from dataclasses import dataclass, field

OK = 0
ARG_ERR = -1
RANK_ERR = -2
NO_SLOT = -3
STATE_ERR = -5


LRU, KEEP_SCORE = 0, 1


@dataclass
class AdapterRecord:
    load_count: int = 0
    hit_count: int = 0
    eviction_count: int = 0
    last_evict_epoch: int | None = None
    last_access: int | None = None
    access_epochs: list = field(default_factory=list)   # one entry per access
    rank: int = 0
    priority: float = 0.0


class LruSlotSim:
    def __init__(self, max_loras: int, max_lora_rank: int, thrash_window: int = 10):
        self.S = max_loras
        self.R = max_lora_rank
        self.window = thrash_window
        self.slot_id: list[int | None] = [None] * max_loras
        self.last_use = [0] * max_loras
        self.refs = [0] * max_loras
        self.clock = 0
        self.epoch = 0
        self.where: dict[int, int] = {}
        self.records: dict[int, AdapterRecord] = {}
        self.hits = self.misses = self.evictions = self.reloads = self.rejected = 0
        self.aborted = 0
        self.log: list[tuple] = []
        self.pinned = [False] * max_loras
        self.pending = [False] * max_loras      # bound by a miss, upload not recorded yet
        self.min_residency = 0
        self.policy = LRU
        self.weights = (1.0, 1.0, 1.0, 0.0, 0.0)

    def _touch(self, s: int) -> None:
        self.clock += 1
        self.last_use[s] = self.clock
        rec = self.records[self.slot_id[s]]
        rec.last_access = self.epoch
        # history older than the window is dropped at each access (a window
        # changed later applies to what is left)
        rec.access_epochs = [e for e in rec.access_epochs if e > self.epoch - self.window]
        rec.access_epochs.append(self.epoch)

    def _may_evict(self, s: int) -> bool:
        aid = self.slot_id[s]
        if aid is None or self.refs[s] > 0 or self.pinned[s]:
            return False
        if self.min_residency > 0 and self.epoch - self.records[aid].last_access < self.min_residency:
            return False
        return True

    def keep_score(self, s: int) -> float:
        rec = self.records[self.slot_id[s]]
        w1, w2, w3, w4, w5 = self.weights
        recent = 1.0 / (1.0 + float(self.epoch - rec.last_access))
        freq = float(sum(1 for e in rec.access_epochs if e > self.epoch - self.window))
        rel = float(rec.rank) / float(self.R)
        k = w1 * recent
        k += w2 * freq
        k += w3 * rec.priority
        k += w4 * rel
        k -= w5 * rel
        return k

    def _victim(self) -> int | None:
        cands = [s for s in range(self.S) if self._may_evict(s)]
        if not cands:
            return None
        if self.policy == LRU:
            return min(cands, key=lambda s: self.last_use[s])
        return min(cands, key=lambda s: (self.keep_score(s), self.last_use[s]))

    def pin(self, s: int, on: bool = True) -> int:
        if not 0 <= s < self.S:
            return ARG_ERR
        if self.slot_id[s] is None:
            return STATE_ERR
        self.pinned[s] = bool(on)
        return OK

    def set_priority(self, aid: int, p: float) -> None:
        self.records.setdefault(aid, AdapterRecord()).priority = float(p)

    def _evict(self, s: int) -> int:
        aid = self.slot_id[s]
        self.slot_id[s] = None
        self.pinned[s] = False
        self.pending[s] = False
        del self.where[aid]
        self.evictions += 1
        rec = self.records[aid]
        rec.eviction_count += 1
        rec.last_evict_epoch = self.epoch
        return aid

    def lookup(self, aid: int) -> int:
        s = self.where.get(aid, -1)
        if s >= 0:
            self._touch(s)
            self.hits += 1
            self.records[aid].hit_count += 1
        self.log.append(("lookup", aid, s))
        return s

    def assign(self, aid: int, rank: int):
        """Returns (status, slot, needs_load, evicted_id or -1)."""
        if aid in self.where:
            s = self.lookup(aid)
            self.log[-1] = ("assign", aid, OK, s, 0, -1)
            return OK, s, 0, -1
        if rank < 1 or rank > self.R:
            self.rejected += 1
            self.log.append(("assign", aid, RANK_ERR, -1, 0, -1))
            return RANK_ERR, -1, 0, -1
        free = [s for s in range(self.S) if self.slot_id[s] is None and self.refs[s] == 0]
        evicted = -1
        if free:
            s = free[0]
        else:
            s = self._victim()
            if s is None:
                self.log.append(("assign", aid, NO_SLOT, -1, 0, -1))
                return NO_SLOT, -1, 0, -1
            evicted = self._evict(s)
        rec = self.records.setdefault(aid, AdapterRecord())
        if rec.last_evict_epoch is not None and self.epoch - rec.last_evict_epoch <= self.window:
            self.reloads += 1
        rec.load_count += 1
        rec.rank = rank
        self.slot_id[s] = aid
        self.where[aid] = s
        self.refs[s] = 0
        self.pinned[s] = False
        self.pending[s] = True
        self._touch(s)
        self.misses += 1
        self.log.append(("assign", aid, OK, s, 1, evicted))
        return OK, s, 1, evicted

    def acquire(self, s: int) -> int:
        if not (0 <= s < self.S) or self.slot_id[s] is None:
            return STATE_ERR
        self.refs[s] += 1
        return OK

    def release(self, s: int) -> int:
        if not (0 <= s < self.S) or self.refs[s] <= 0:
            return STATE_ERR
        self.refs[s] -= 1
        return OK

    def evict_lru(self):
        """Returns (status, slot or -1, evicted id or -1)."""
        if all(a is None for a in self.slot_id):
            self.log.append(("evict", OK, -1, -1))
            return OK, -1, -1
        s = self._victim()
        if s is None:
            self.log.append(("evict", NO_SLOT, -1, -1))
            return NO_SLOT, -1, -1
        aid = self._evict(s)
        self.log.append(("evict", OK, s, aid))
        return OK, s, aid

    def loaded(self, s: int) -> int:
        """An upload into slot s was queued: its adapter is no longer pending."""
        if not 0 <= s < self.S:
            return ARG_ERR
        self.pending[s] = False
        return OK

    def abort_load(self, s: int):
        """The pending upload into slot s failed: the adapter is unbound (not
        an eviction; the pin ends, references stay until released). Returns
        (status, id that was bound or -1)."""
        if not 0 <= s < self.S:
            return ARG_ERR, -1
        aid = self.slot_id[s]
        if aid is None or not self.pending[s]:
            return STATE_ERR, -1
        self.slot_id[s] = None
        self.pinned[s] = False
        self.pending[s] = False
        del self.where[aid]
        self.aborted += 1
        self.log.append(("abort", s, aid))
        return OK, aid

    def tick(self) -> None:
        self.epoch += 1

    def thrash_ratio(self) -> float:
        return self.reloads / self.evictions if self.evictions else 0.0
