"""Pins for the independent LRU slot-table simulator: scripted sequences whose
victims are derived by hand from the "Multi-LoRA 适配器缓存生产实战" page
(section 核心原理: touch on hit, oldest evicted, in-flight adapters never
evicted; section 为什么纯 LRU 在多租户场景下容易失效: the 4-slot / 20-adapter
burst)."""
from oracle.lru_sim import LruSlotSim, OK, NO_SLOT, RANK_ERR, STATE_ERR


def test_touch_changes_victim():
    s = LruSlotSim(2, 16)
    assert s.assign(10, 4) == (OK, 0, 1, -1)        # free slot 0
    assert s.assign(11, 4) == (OK, 1, 1, -1)        # free slot 1
    assert s.lookup(10) == 0                        # hit: 10 becomes most recent
    assert s.assign(12, 4) == (OK, 1, 1, 11)        # 11 is oldest
    assert s.assign(13, 4) == (OK, 0, 1, 10)        # 10 (touched before 12 loaded)
    assert s.hits == 1 and s.misses == 4 and s.evictions == 2


def test_hit_does_not_reload():
    s = LruSlotSim(3, 16)
    s.assign(1, 8)
    assert s.assign(1, 8) == (OK, 0, 0, -1)
    assert s.misses == 1 and s.hits == 1


def test_lowest_free_slot_first_after_explicit_evict():
    s = LruSlotSim(3, 16)
    for a in (5, 6, 7):
        s.assign(a, 8)
    assert s.evict_lru() == (OK, 0, 5)
    s.lookup(6)
    assert s.assign(8, 8) == (OK, 0, 1, -1)         # reuses the free slot, evicts nothing


def test_in_flight_is_never_evicted():
    s = LruSlotSim(2, 16)
    s.assign(1, 4)
    s.assign(2, 4)
    assert s.acquire(0) == OK                       # adapter 1 is in flight
    assert s.assign(3, 4) == (OK, 1, 1, 2)          # 2 evicted although 1 is older
    assert s.acquire(1) == OK
    assert s.assign(4, 4) == (NO_SLOT, -1, 0, -1)   # both in flight
    assert s.evict_lru() == (NO_SLOT, -1, -1)
    assert s.release(0) == OK
    assert s.assign(4, 4) == (OK, 0, 1, 1)
    assert s.release(0) == STATE_ERR                # refcount already zero


def test_rank_validated_before_eviction():
    s = LruSlotSim(2, 16)
    s.assign(1, 16)
    s.assign(2, 16)
    assert s.assign(3, 17) == (RANK_ERR, -1, 0, -1)
    assert s.assign(3, 0) == (RANK_ERR, -1, 0, -1)
    assert s.slot_id == [1, 2] and s.evictions == 0 and s.rejected == 2


def test_evict_on_empty_table():
    s = LruSlotSim(4, 16)
    assert s.evict_lru() == (OK, -1, -1)


def test_burst_of_cold_adapters_flushes_hot_set():
    """4 GPU slots, hot adapters 0..3 in use; a batch tenant then touches 20
    low-frequency adapters in a row; pure LRU evicts every hot adapter, and the
    hot set reloads afterwards (4 reloads inside the window)."""
    s = LruSlotSim(4, 16, thrash_window=10)
    for rnd in range(3):
        for a in range(4):
            s.assign(a, 16)
        s.tick()
    assert s.misses == 4 and s.hits == 8
    evicted = []
    for a in range(100, 120):
        st, slot, load, ev = s.assign(a, 16)
        assert st == OK and load == 1
        evicted.append(ev)
    assert evicted[:4] == [0, 1, 2, 3]
    assert evicted[4:] == list(range(100, 116))
    s.tick()
    again = [s.assign(a, 16) for a in range(4)]
    assert [g[3] for g in again] == [116, 117, 118, 119]
    assert all(g[2] == 1 for g in again)
    assert s.evictions == 24 and s.reloads == 4
    assert abs(s.thrash_ratio() - 4 / 24) < 1e-15


def test_reload_outside_window_is_not_thrash():
    s = LruSlotSim(1, 16, thrash_window=2)
    s.assign(1, 8)
    s.assign(2, 8)          # evicts 1 at epoch 0
    for _ in range(3):
        s.tick()
    s.assign(1, 8)          # epoch 3: 3 > window
    assert s.reloads == 0
    s.assign(2, 8)          # 2 evicted at epoch 3, reloaded at epoch 3
    assert s.reloads == 1


# ---- platform policies (section 为什么纯 LRU 在多租户场景下容易失效) ----------

from oracle.lru_sim import ARG_ERR, KEEP_SCORE  # noqa: E402


def _hot_rounds(s, rounds=3):
    for _ in range(rounds):
        for a in range(4):
            s.assign(a, 16)
        s.tick()


def test_pinned_warm_set_survives_burst():
    """Slots of adapters 0 and 1 pinned: the 20-adapter burst cycles through the
    two unpinned slots only (2 and 3 go first, then the burst evicts itself)."""
    s = LruSlotSim(4, 16, thrash_window=10)
    _hot_rounds(s)
    assert s.pin(0) == OK and s.pin(1) == OK
    evicted = [s.assign(a, 16)[3] for a in range(100, 120)]
    assert evicted[:2] == [2, 3]
    assert evicted[2:] == list(range(100, 118))
    s.tick()
    assert s.assign(0, 16) == (OK, 0, 0, -1) and s.assign(1, 16) == (OK, 1, 0, -1)


def test_pin_errors_and_unpin():
    s = LruSlotSim(2, 16)
    assert s.pin(0) == STATE_ERR                     # empty slot
    assert s.pin(5) == ARG_ERR
    s.assign(1, 8)
    s.assign(2, 8)
    s.pin(0)
    s.pin(1)
    assert s.assign(3, 8) == (NO_SLOT, -1, 0, -1)    # everything pinned
    assert s.evict_lru() == (NO_SLOT, -1, -1)
    s.pin(1, False)
    assert s.assign(3, 8) == (OK, 1, 1, 2)


def test_cooling_window_defers_until_old_enough():
    s = LruSlotSim(2, 16)
    s.min_residency = 2
    s.assign(1, 8)
    s.assign(2, 8)
    assert s.assign(3, 8) == (NO_SLOT, -1, 0, -1)    # both accessed this epoch
    s.tick()
    assert s.assign(3, 8) == (NO_SLOT, -1, 0, -1)    # 1 epoch old < 2
    s.lookup(2)                                      # 2 accessed again at epoch 1
    s.tick()
    assert s.assign(3, 8) == (OK, 0, 1, 1)           # 1 is 2 epochs old, 2 only 1


def test_keep_score_hand_example_differs_from_lru():
    """w = (1, 1, 0, 0, 0). A: bound at epoch 0 and hit twice; B bound at
    epoch 1; C bound at epoch 2; at epoch 3:
      A: recent 1/(1+3) = 0.25, frequency 3  -> 3.25
      B: recent 1/(1+2),        frequency 1  -> 1.333...
      C: recent 1/(1+1) = 0.5,  frequency 1  -> 1.5
    keep_score evicts B; LRU would evict A (oldest last use)."""
    def build(policy):
        s = LruSlotSim(3, 16)
        s.policy = policy
        s.weights = (1.0, 1.0, 0.0, 0.0, 0.0)
        s.assign(10, 16); s.lookup(10); s.lookup(10); s.tick()
        s.assign(11, 16); s.tick()
        s.assign(12, 16); s.tick()
        return s
    k = build(KEEP_SCORE)
    assert [k.keep_score(i) for i in range(3)] == [3.25, 1.0 + 1.0 / 3.0, 1.5]
    assert k.assign(13, 16) == (OK, 1, 1, 11)
    assert build(0).assign(13, 16) == (OK, 0, 1, 10)


def test_keep_score_priority_and_size_terms():
    s = LruSlotSim(2, 64)
    s.policy = KEEP_SCORE
    s.weights = (1.0, 1.0, 1.0, 0.0, 1.0)
    s.assign(1, 64)                                  # size term 1.0
    s.assign(2, 16)                                  # size term 0.25
    # both: recent 1, frequency 1 -> 2 - size: 1 -> 1.0, 2 -> 1.75
    assert s.assign(3, 16) == (OK, 0, 1, 1)
    s.set_priority(3, 5.0)
    # 3: 2 + 5 - 0.25 = 6.75 ; 2: 1.75 -> 2 goes
    assert s.assign(4, 16) == (OK, 1, 1, 2)


def test_keep_score_burst_keeps_hot_set():
    """The page's scenario under keep_score (1, 1, 0, 0, 0): at the burst epoch
    the hot adapters score 1/2 + 3 = 3.5 and each newcomer 1 + 1 = 2, so the
    first burst adapter costs one hot adapter (the LRU tie-break) and every
    later one evicts the previous newcomer."""
    s = LruSlotSim(4, 16, thrash_window=10)
    s.policy = KEEP_SCORE
    s.weights = (1.0, 1.0, 0.0, 0.0, 0.0)
    _hot_rounds(s)
    evicted = [s.assign(a, 16)[3] for a in range(100, 120)]
    assert evicted[0] == 0
    assert evicted[1:] == list(range(100, 119))
    s.tick()
    hot = [s.assign(a, 16) for a in range(4)]
    assert [h[2] for h in hot] == [1, 0, 0, 0]       # only adapter 0 reloads
    assert s.reloads == 1


def test_reload_at_the_window_edge_is_thrash():
    """A reload exactly `thrash_window` epochs after the eviction still counts
    (the window is inclusive); one epoch later it does not."""
    s = LruSlotSim(1, 16, thrash_window=2)
    s.assign(1, 8)
    s.assign(2, 8)          # evicts 1 at epoch 0
    s.tick()
    s.tick()
    s.assign(1, 8)          # epoch 2: 2 - 0 <= 2, and evicts 2 at epoch 2
    assert s.reloads == 1
    for _ in range(3):
        s.tick()
    s.assign(2, 8)          # epoch 5: 5 - 2 > 2
    assert s.reloads == 1 and s.evictions == 3


def test_frequency_counts_an_access_for_window_epochs():
    """keep_score with only the frequency term, window 3: an access made at
    epoch 0 counts at epochs 0, 1 and 2 and no longer at epoch 3."""
    s = LruSlotSim(2, 16, thrash_window=3)
    s.policy = KEEP_SCORE
    s.weights = (0.0, 1.0, 0.0, 0.0, 0.0)
    s.assign(7, 16)
    seen = []
    for _ in range(4):
        seen.append(s.keep_score(0))
        s.tick()
    assert seen == [1.0, 1.0, 1.0, 0.0]


def test_keep_score_priority_outweighs_recency():
    """Weights (1, 1, 1, 0, 0), two adapters bound in the same epoch (recency
    1 and frequency 1 each): with priority 5 on the older one, the newer one
    scores 2 against 7 and is evicted; without it the scores tie and the
    least recently used (the older one) goes."""
    def run(prio):
        s = LruSlotSim(2, 16)
        s.policy = KEEP_SCORE
        s.weights = (1.0, 1.0, 1.0, 0.0, 0.0)
        s.assign(1, 16)
        s.assign(2, 16)
        if prio:
            s.set_priority(1, 5.0)
        return s.assign(3, 16)
    assert run(True) == (OK, 1, 1, 2)
    assert run(False) == (OK, 0, 1, 1)


def test_abort_load_frees_the_slot():
    """2 slots: 3 evicts 1 from slot 0, then its upload fails. Slot 0 is empty:
    3 is not resident, 1 stays evicted, the next miss takes slot 0 without an
    eviction, and a retry of 3 is a miss again."""
    s = LruSlotSim(2, 16)
    s.assign(1, 8)
    s.assign(2, 8)
    assert s.assign(3, 8) == (OK, 0, 1, 1)
    assert s.abort_load(0) == (OK, 3)
    assert s.lookup(3) == -1 and s.lookup(1) == -1
    assert s.assign(4, 8) == (OK, 0, 1, -1)          # the free slot, nothing evicted
    assert s.assign(3, 8) == (OK, 1, 1, 2)           # 3 loads again, evicting 2 (LRU)
    assert (s.evictions, s.aborted, s.misses) == (2, 1, 5)
    assert s.abort_load(0) == (OK, 4)
    assert s.abort_load(0) == (STATE_ERR, -1)        # already empty
    assert s.abort_load(9) == (ARG_ERR, -1)


def test_abort_load_ends_pin_and_keeps_references():
    """The pin ends with the abort; a reference taken before it stays until it
    is released, and the slot is not reused meanwhile."""
    s = LruSlotSim(2, 16)
    s.assign(1, 8)
    s.acquire(0)
    s.pin(0)
    assert s.abort_load(0) == (OK, 1)
    assert s.pin(0) == STATE_ERR                     # bound to nothing
    assert s.acquire(0) == STATE_ERR                 # no new reference on an unbound slot
    assert s.assign(2, 8) == (OK, 1, 1, -1)          # slot 0 still referenced: slot 1 is the free one
    assert s.release(0) == OK                        # the reference taken before the abort
    assert s.release(0) == STATE_ERR                 # none left
    assert s.assign(3, 8) == (OK, 0, 1, -1)          # slot 0 is free again
    assert s.assign(4, 8) == (OK, 1, 1, 2)           # an ordinary LRU table again: 2 is the oldest


def test_abort_only_while_the_upload_is_pending():
    """An adapter whose upload was recorded cannot be aborted (it is removed by
    eviction instead); a new bind of the slot makes it pending again."""
    s = LruSlotSim(2, 16)
    s.assign(1, 8)
    assert s.loaded(0) == OK
    assert s.abort_load(0) == (STATE_ERR, -1)
    assert s.lookup(1) == 0                          # still resident
    s.assign(2, 8)
    assert s.assign(3, 8) == (OK, 0, 1, 1)           # evicts 1; 3 is pending in slot 0
    assert s.abort_load(0) == (OK, 3)
    assert s.loaded(7) == ARG_ERR


def test_late_release_after_abort_cannot_touch_a_later_adapter():
    """Holder A takes a reference on its adapter's slot, the upload fails and is
    aborted; holder B's adapter cannot be bound to that slot while A's
    reference stays, so A's release (however late) lowers no count of B's."""
    s = LruSlotSim(2, 16)
    assert s.assign(10, 8) == (OK, 0, 1, -1)
    s.acquire(0)                                     # holder A
    assert s.abort_load(0) == (OK, 10)
    assert s.assign(20, 8) == (OK, 1, 1, -1)         # holder B: slot 1, not the referenced slot 0
    s.loaded(1)
    s.acquire(1)
    assert s.release(0) == OK                        # A's release hits its own slot
    assert s.assign(30, 8) == (OK, 0, 1, -1)         # slot 0 free now; B's adapter untouched
    assert s.evict_lru() == (OK, 0, 30)              # B's slot is in flight: never the victim
    assert s.refs == [0, 1]
