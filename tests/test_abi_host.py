"""CPU tests of the C ABI: the library loads, exports every declared symbol, and
its host slot table takes the same decisions as the independent simulator."""
import os
import re

import numpy as np
import pytest

import oracle
from oracle.lru_sim import LruSlotSim
from rank_adapter_apply_gb300 import binding as B
from rank_adapter_apply_gb300 import build as build_mod

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "rank_adapter_apply.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 19
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.EXPORTED) == names


def test_workspace_and_byte_count(lib):
    assert B.lora_workspace_bytes(8, 16, 256, 2) > 0
    assert B.lora_workspace_bytes(0, 16, 256, 2) == 0
    assert B.lora_workspace_bytes(8, 16, 256, 9) == 0
    cases = [([(4096, 4096), (4096, 4096)], 16, 2),
             ([(5120, 8192), (5120, 1024), (5120, 1024), (8192, 5120)], 32, 2),
             ([(4096, 4096), (4096, 1024), (4096, 1024), (4096, 4096), (4096, 14336),
               (4096, 14336), (14336, 4096)], 64, 2)]
    for layers, r, bpp in cases:
        assert B.lora_adapter_bytes(layers, r, bpp) == oracle.adapter_bytes(layers, r, bpp)


def test_init_rejects_bad_arguments(lib):
    with pytest.raises(B.LoraError):
        B.lora_slots_init(0, 16, 1, 1, 1, [], None, None, None, 0, None, None)
    with pytest.raises(B.LoraError):
        B.lora_slots_init(4, 12, 1, 1, 1, [], None, None, None, 0, None, None)   # rank % 8
    with pytest.raises(B.LoraError):
        B.lora_slots_init(4, 128, 1, 1, 1, [], None, None, None, 0, None, None)  # bf16 > 64


def _host_ctx(S, R):
    return B.lora_slots_init(S, R, 0, 1, B.LORA_DTYPE_BF16, [], None, None, None, 0, None, None)


def _host_load(ctx, slot, rank=8):
    """lora_load_slot on a host-only context: records the upload, copies nothing."""
    try:
        B.lora_load_slot(ctx, slot, [], [], rank, 16.0)
        return 0
    except B.LoraError as e:
        return e.code


def _run_script(ctx, sim, ops):
    last_bound = [None]
    for op in ops:
        kind = op[0]
        if kind == "assign":
            got = B.lora_assign(ctx, op[1], op[2])
            exp = sim.assign(op[1], op[2])
            assert got == exp, (op, got, exp)
            last_bound[0] = got[1] if got[0] == 0 and got[2] == 1 else None
        elif kind == "lookup":
            assert B.lora_lookup(ctx, op[1]) == sim.lookup(op[1]), op
        elif kind == "acquire":
            assert B.lora_acquire(ctx, op[1]) == sim.acquire(op[1]), op
        elif kind == "release":
            assert B.lora_release(ctx, op[1]) == sim.release(op[1]), op
        elif kind == "evict":
            assert B.lora_evict_lru(ctx) == sim.evict_lru(), op
        elif kind == "abort":
            assert B.lora_abort_load(ctx, op[1]) == sim.abort_load(op[1]), op
        elif kind == "abort_last":         # the upload of the last assign that bound a slot failed
            if last_bound[0] is not None:
                assert B.lora_abort_load(ctx, last_bound[0]) == sim.abort_load(last_bound[0]), op
        elif kind == "loaded_last":        # the upload of the last assign that bound a slot
            if last_bound[0] is not None:
                assert _host_load(ctx, last_bound[0]) == sim.loaded(last_bound[0]) == 0
        elif kind == "loaded":             # an upload queued into the slot (host-only: recorded)
            rc = _host_load(ctx, op[1])
            assert rc == sim.loaded(op[1]), op
        elif kind == "tick":
            B.lora_tick(ctx)
            sim.tick()
    st = B.lora_stats(ctx)
    assert (st["hits"], st["misses"], st["evictions"], st["reloads_after_eviction"],
            st["rejected"], st["aborted_loads"]) == (sim.hits, sim.misses, sim.evictions, sim.reloads,
                                                     sim.rejected, sim.aborted)


def test_scripted_decisions_match_simulator(lib):
    ctx = _host_ctx(2, 16)
    try:
        sim = LruSlotSim(2, 16)
        _run_script(ctx, sim, [
            ("assign", 10, 4), ("assign", 11, 4), ("lookup", 10), ("assign", 12, 4),
            ("assign", 13, 4), ("acquire", 0), ("assign", 14, 4), ("acquire", 1),
            ("assign", 15, 4), ("evict",), ("release", 0), ("release", 0), ("assign", 15, 17),
            ("assign", 15, 16), ("evict",), ("evict",), ("release", 1), ("evict",), ("evict",),
        ])
    finally:
        B.lora_destroy(ctx)


def test_random_decision_log_matches_simulator(lib):
    """Zipf adapter streams with in-flight sub-batches: every decision equal."""
    rng = np.random.default_rng(0)
    S, R = 8, 16
    ctx = _host_ctx(S, R)
    sim = LruSlotSim(S, R)
    try:
        p = np.arange(1, 65, dtype=float) ** -1.2
        p /= p.sum()
        for step in range(300):
            ids = np.unique(rng.choice(64, size=12, p=p))[:S]
            held = []
            for a in ids:
                rank = int(rng.choice([8, 16, 16, 16, 24]))
                got = B.lora_assign(ctx, int(a), rank)
                assert got == sim.assign(int(a), rank)
                if got[0] == 0 and rng.random() < 0.7:
                    assert B.lora_acquire(ctx, got[1]) == sim.acquire(got[1])
                    held.append(got[1])
            if rng.random() < 0.1:
                assert B.lora_evict_lru(ctx) == sim.evict_lru()
            for s in held:
                assert B.lora_release(ctx, s) == sim.release(s)
            B.lora_tick(ctx)
            sim.tick()
        st = B.lora_stats(ctx)
        assert st["misses"] == sim.misses and st["evictions"] == sim.evictions
        assert st["reloads_after_eviction"] == sim.reloads and st["epoch"] == 300
    finally:
        B.lora_destroy(ctx)


def test_thrash_burst_through_abi(lib):
    ctx = _host_ctx(4, 16)
    sim = LruSlotSim(4, 16)
    try:
        ops = []
        for _ in range(3):
            ops += [("assign", a, 16) for a in range(4)] + [("tick",)]
        ops += [("assign", a, 16) for a in range(100, 120)] + [("tick",)]
        ops += [("assign", a, 16) for a in range(4)]
        _run_script(ctx, sim, ops)
        assert B.lora_stats(ctx)["reloads_after_eviction"] == 4
    finally:
        B.lora_destroy(ctx)


def _policy_stream(ctx, sim, rng, steps, S, pin_p, set_prio):
    p = np.arange(1, 97, dtype=float) ** -1.1
    p /= p.sum()
    for step in range(steps):
        ids = list(dict.fromkeys(int(a) for a in rng.choice(96, size=14, p=p)))[:S]
        held = []
        for a in ids:
            if set_prio and rng.random() < 0.05:
                pr = float(rng.integers(0, 4))
                B.lora_set_adapter_priority(ctx, a, pr)
                sim.set_priority(a, pr)
            rank = int(rng.choice([8, 16, 32]))
            got = B.lora_assign(ctx, a, rank)
            assert got == sim.assign(a, rank), (step, a, got)
            if got[0] == 0 and rng.random() < 0.6:
                assert B.lora_acquire(ctx, got[1]) == sim.acquire(got[1])
                held.append(got[1])
        if rng.random() < pin_p:
            s = int(rng.integers(0, S))
            on = bool(rng.random() < 0.6)
            assert B.lora_pin(ctx, s, on) == sim.pin(s, on)
        if rng.random() < 0.1:
            assert B.lora_evict_lru(ctx) == sim.evict_lru()
        for s in held:
            assert B.lora_release(ctx, s) == sim.release(s)
        B.lora_tick(ctx)
        sim.tick()
    st = B.lora_stats(ctx)
    assert (st["hits"], st["misses"], st["evictions"], st["reloads_after_eviction"]) == \
        (sim.hits, sim.misses, sim.evictions, sim.reloads)


@pytest.mark.parametrize("policy", [0, 1])
@pytest.mark.parametrize("min_res", [0, 2])
def test_policy_decision_log_matches_simulator(lib, policy, min_res):
    """Pins, the cooling window and both eviction policies: every decision of
    the library equals the independent simulator's."""
    from oracle.lru_sim import LruSlotSim
    rng = np.random.default_rng(10 * policy + min_res)
    S, R = 8, 32
    ctx = _host_ctx(S, R)
    sim = LruSlotSim(S, R, thrash_window=6)
    try:
        B.lora_set_thrash_window(ctx, 6)
        B.lora_set_policy(ctx, policy)
        sim.policy = policy
        w = (1.0, 0.5, 2.0, 0.25, 0.75)
        B.lora_set_keep_score_weights(ctx, w)
        sim.weights = w
        B.lora_set_min_residency(ctx, min_res)
        sim.min_residency = min_res
        _policy_stream(ctx, sim, rng, 250, S, pin_p=0.2, set_prio=True)
    finally:
        B.lora_destroy(ctx)


def test_window_edges_and_priority_match_simulator(lib):
    """The boundary cases pinned on the simulator, through the library: a
    reload exactly thrash_window epochs after its eviction, and a priority that
    decides a keep_score eviction."""
    from oracle.lru_sim import LruSlotSim, KEEP_SCORE
    ctx = _host_ctx(1, 16)
    sim = LruSlotSim(1, 16, thrash_window=2)
    try:
        B.lora_set_thrash_window(ctx, 2)
        _run_script(ctx, sim, [("assign", 1, 8), ("assign", 2, 8), ("tick",), ("tick",), ("assign", 1, 8),
                               ("tick",), ("tick",), ("tick",), ("assign", 2, 8)])
        assert sim.reloads == 1
    finally:
        B.lora_destroy(ctx)
    for prio in (True, False):
        ctx = _host_ctx(2, 16)
        sim = LruSlotSim(2, 16)
        try:
            B.lora_set_policy(ctx, KEEP_SCORE)
            sim.policy = KEEP_SCORE
            B.lora_set_keep_score_weights(ctx, (1.0, 1.0, 1.0, 0.0, 0.0))
            sim.weights = (1.0, 1.0, 1.0, 0.0, 0.0)
            _run_script(ctx, sim, [("assign", 1, 16), ("assign", 2, 16)])
            if prio:
                B.lora_set_adapter_priority(ctx, 1, 5.0)
                sim.set_priority(1, 5.0)
            _run_script(ctx, sim, [("assign", 3, 16)])
        finally:
            B.lora_destroy(ctx)


def test_policy_argument_errors(lib):
    ctx = _host_ctx(2, 16)
    try:
        assert B.lora_pin(ctx, 0) == B.LORA_ERR_STATE          # empty slot
        assert B.lora_pin(ctx, 7) == B.LORA_ERR_ARG
        with pytest.raises(B.LoraError):
            B.lora_set_policy(ctx, 9)
        with pytest.raises(B.LoraError):
            B.lora_set_min_residency(ctx, -1)
        with pytest.raises(B.LoraError):
            B.lora_set_keep_score_weights(ctx, [1, float("nan"), 0, 0, 0])
        with pytest.raises(B.LoraError):
            B.lora_set_adapter_priority(ctx, 3, float("inf"))
    finally:
        B.lora_destroy(ctx)


def test_pinned_burst_through_abi(lib):
    from oracle.lru_sim import LruSlotSim
    ctx = _host_ctx(4, 16)
    sim = LruSlotSim(4, 16)
    try:
        ops = []
        for _ in range(3):
            ops += [("assign", a, 16) for a in range(4)] + [("tick",)]
        _run_script(ctx, sim, ops)
        for s in (0, 1):
            assert B.lora_pin(ctx, s) == sim.pin(s) == 0
        ops = [("assign", a, 16) for a in range(100, 120)] + [("tick",)]
        ops += [("assign", a, 16) for a in range(4)]
        _run_script(ctx, sim, ops)
        assert sim.reloads == 2                      # only the unpinned 2 and 3
    finally:
        B.lora_destroy(ctx)


def test_assign_batch_equals_sequential_calls(lib):
    """lora_assign_batch / lora_release_batch take the decisions of the
    equivalent lora_assign + lora_acquire / lora_release sequence."""
    from oracle.lru_sim import LruSlotSim
    rng = np.random.default_rng(5)
    S, R = 6, 16
    ctx = _host_ctx(S, R)
    sim = LruSlotSim(S, R)
    try:
        for step in range(120):
            ids = list(dict.fromkeys(int(a) for a in rng.integers(0, 20, size=8)))[:S]
            ranks = [int(rng.choice([8, 16])) for _ in ids]
            rc, done, slots, need, ev = B.lora_assign_batch(ctx, ids, ranks)
            assert rc == 0 and done == len(ids)
            for a, r, s_, n_, e_ in zip(ids, ranks, slots, need, ev):
                assert sim.assign(a, r) == (0, int(s_), int(n_), int(e_))
                assert sim.acquire(int(s_)) == 0
            assert B.lora_release_batch(ctx, slots) == 0
            for s_ in slots:
                sim.release(int(s_))
            B.lora_tick(ctx)
            sim.tick()
        # a failing entry stops the batch: rank too large after two good ones
        rc, done, slots, need, ev = B.lora_assign_batch(ctx, [1001, 1002, 1003], [8, 8, 99])
        assert rc == B.LORA_ERR_RANK and done == 2
        assert B.lora_release_batch(ctx, slots[:2]) == 0
        assert B.lora_release_batch(ctx, slots[:1]) == B.LORA_ERR_STATE
    finally:
        B.lora_destroy(ctx)


def test_assign_tokens_matches_simulator_and_maps_tokens(lib):
    """lora_assign_tokens admits the batch's distinct adapters in order of first
    appearance with the simulator's decisions, and maps every token to its
    adapter's slot (-1 for base-only tokens)."""
    rng = np.random.default_rng(11)
    S, R = 6, 16
    ctx = _host_ctx(S, R)
    sim = LruSlotSim(S, R)
    try:
        for step in range(150):
            T = int(rng.integers(1, 40))
            ids = rng.integers(0, 25, size=T).astype(np.int64)
            ids[rng.random(T) < 0.15] = -1
            # at most S distinct adapters, so every admission succeeds (all in flight)
            keep = list(dict.fromkeys(int(a) for a in ids if a >= 0))[:S]
            ids = np.where(np.isin(ids, keep), ids, -1)
            rank_of = {a: int(rng.choice([8, 16])) for a in keep}
            ranks = np.array([rank_of.get(int(a), 0) for a in ids], np.int32)
            rc, tsi, dids, slots, need, ev, done = B.lora_assign_tokens(ctx, ids, ranks, max_distinct=S)
            assert rc == 0 and done == len(keep)
            assert list(dids) == keep
            for a, s_, n_, e_ in zip(keep, slots, need, ev):
                assert sim.assign(a, rank_of[a]) == (0, int(s_), int(n_), int(e_))
                assert sim.acquire(int(s_)) == 0
            slot_of = dict(zip(keep, (int(x) for x in slots)))
            expect = np.array([slot_of[int(a)] if a >= 0 else -1 for a in ids], np.int32)
            assert np.array_equal(tsi, expect)
            assert B.lora_release_batch(ctx, slots) == 0
            for s_ in slots:
                sim.release(int(s_))
            B.lora_tick(ctx)
            sim.tick()
        # a failing admission stops the batch: its tokens and later ones map to -1
        ids = np.array([2001, -1, 2002, 2001, 2003, 2002], np.int64)
        ranks = np.array([8, 0, 8, 8, 99, 8], np.int32)
        rc, tsi, dids, slots, need, ev, done = B.lora_assign_tokens(ctx, ids, ranks)
        assert rc == B.LORA_ERR_RANK and done == 2 and list(dids) == [2001, 2002, 2003]
        assert list(tsi) == [slots[0], -1, slots[1], slots[0], -1, slots[1]]
        assert B.lora_release_batch(ctx, slots[:2]) == 0
        # more distinct adapters than max_distinct: rejected before any admission
        before = [B.lora_lookup(ctx, a) for a in (2001, 2002)]
        rc, tsi, dids, slots, need, ev, done = B.lora_assign_tokens(ctx, [3001, 3002, 3003], [8, 8, 8],
                                                                     max_distinct=2)
        assert rc == B.LORA_ERR_ARG and done == 0 and list(tsi) == [-1, -1, -1]
        assert B.lora_lookup(ctx, 3001) == -1
        assert [B.lora_lookup(ctx, a) for a in (2001, 2002)] == before
        # all base-only, and an empty batch
        rc, tsi, dids, slots, need, ev, done = B.lora_assign_tokens(ctx, [-1, -1], [0, 0])
        assert rc == 0 and done == 0 and len(dids) == 0 and list(tsi) == [-1, -1]
        rc, tsi, dids, slots, need, ev, done = B.lora_assign_tokens(ctx, np.zeros(0, np.int64), [])
        assert rc == 0 and len(tsi) == 0
    finally:
        B.lora_destroy(ctx)


def test_assign_tokens_large_batches_and_colliding_ids(lib):
    """Thousands of tokens over 200 distinct adapters, with ids drawn from the
    whole 63-bit range and with ids that differ only in their top bits (they
    all land on one bucket of the call's hash table): the distinct list is in
    order of first appearance and every token gets its adapter's slot."""
    rng = np.random.default_rng(5)
    for kind in ("random", "top_bits"):
        ctx = _host_ctx(256, 16)
        try:
            if kind == "random":
                pool = rng.integers(0, 2 ** 63 - 1, size=200, dtype=np.int64)
            else:
                pool = (np.arange(1, 201, dtype=np.int64) << 47)
            T = 3000
            ids = pool[rng.integers(0, len(pool), size=T)]
            ids[rng.random(T) < 0.1] = -1
            rc, tsi, dids, slots, need, ev, done = B.lora_assign_tokens(ctx, ids, np.full(T, 8, np.int32))
            first = list(dict.fromkeys(int(a) for a in ids if a >= 0))
            assert rc == 0 and done == len(first) and [int(a) for a in dids] == first
            assert sorted(int(s_) for s_ in slots) == list(range(len(first)))   # lowest free slots
            slot_of = dict(zip(first, (int(x) for x in slots)))
            assert np.array_equal(tsi, np.array([slot_of[int(a)] if a >= 0 else -1 for a in ids], np.int32))
            assert all(B.lora_lookup(ctx, a) == slot_of[a] for a in first[:20])
        finally:
            B.lora_destroy(ctx)


def test_small_batch_limit_arguments(lib):
    """-1 restores the rank-based limit; 0..1024 set it; anything else is refused."""
    ctx = _host_ctx(4, 16)
    try:
        for n in (-1, 0, 512, 1024, -1):
            assert lib.lora_set_small_batch_tokens(ctx, n) == 0
        for n in (-2, 1025):
            assert lib.lora_set_small_batch_tokens(ctx, n) == B.LORA_ERR_ARG
    finally:
        B.lora_destroy(ctx)


def test_selftest_needs_a_device_context(lib):
    ctx = _host_ctx(2, 16)
    try:
        import ctypes
        g = ctypes.c_int(0)
        assert lib.lora_selftest_wait_timeout(ctx, ctypes.byref(g)) == B.LORA_ERR_STATE
    finally:
        B.lora_destroy(ctx)


def test_static_scratch_validates_before_touching_the_device(lib):
    """lora_apply_static_scratch checks its arguments before any CUDA call, so
    every rejection below (and the empty batch) is decided on the host. The
    pointer values are never dereferenced: each case returns before a launch."""
    P = 0x10000                                     # 16-byte aligned stand-in address
    ok = dict(x=P, y=P, idx=P, T=64, d_in=512, d_out=512, S=4, R=16, dtype=B.LORA_DTYPE_BF16,
              A=P, B=P, scale=P, rank=P)

    def call(**kw):
        a = {**ok, **kw}
        return lib.lora_apply_static_scratch(a["x"], a["y"], a["idx"], a["T"], a["d_in"],
                                             a["d_out"], a["S"], a["R"], a["dtype"], a["A"],
                                             a["B"], a["scale"], a["rank"], None)

    assert call(T=0) == B.LORA_OK                      # empty batch: nothing to do
    assert call(T=0, x=None, A=None) == B.LORA_OK      # not even the pointers are read
    bad = [dict(dtype=9), dict(S=0), dict(S=257), dict(R=4), dict(R=12), dict(R=72),
           dict(R=264, dtype=B.LORA_DTYPE_F32), dict(d_in=0), dict(d_out=0), dict(T=-1),
           dict(x=None), dict(y=None), dict(idx=None), dict(A=None), dict(B=None),
           dict(scale=None), dict(rank=None), dict(A=P + 8), dict(B=P + 2),
           dict(T=9000, R=64)]                      # partials of 9000 x 64 fp32 exceed 4 MiB
    for kw in bad:
        assert call(**kw) == B.LORA_ERR_ARG, kw
    assert "static scratch" in B.last_error()


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """With the compiled library absent the binding raises; there is no other
    implementation to fall back on."""
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        B.load(str(tmp_path / "librank_adapter_apply.so"))


def test_stats_struct_matches_the_header(lib):
    """lora_stats writes exactly the binding's LoraStats: a buffer with guard
    bytes after it comes back with every struct byte written and the guard
    untouched, and a host-only context reports no kernel launches."""
    import ctypes
    n = ctypes.sizeof(B.LoraStats)
    buf = (ctypes.c_ubyte * (n + 64))(*([0xAB] * (n + 64)))
    ctx = _host_ctx(4, 16)
    try:
        assert lib.lora_stats(ctx, ctypes.cast(buf, ctypes.POINTER(B.LoraStats))) == 0
        assert all(b == 0xAB for b in bytes(buf)[n:])
        st = B.LoraStats.from_buffer_copy(bytes(buf)[:n])
        assert all(getattr(st, k) == 0 for k, _ in B.LoraStats._fields_)
        # the header declares the same fields in the same order
        src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
        body = re.search(r"typedef struct \{([^}]*)\} lora_stats_t;", src).group(1)
        names = re.findall(r"\b(\w+)\s*;", body)
        assert names == [k for k, _ in B.LoraStats._fields_]
    finally:
        B.lora_destroy(ctx)


def test_failed_load_leaves_the_table_consistent(lib):
    """A serving step whose upload fails part-way: the adapters whose uploads
    failed are unbound with lora_abort_load, the others stay resident, nothing
    else is evicted, and the next step loads the failed ones again; every
    decision equals the simulator's."""
    from oracle.lru_sim import LruSlotSim
    ctx = _host_ctx(4, 16)
    sim = LruSlotSim(4, 16)
    try:
        _run_script(ctx, sim, [("assign", a, 16) for a in (1, 2, 3, 4)] + [("tick",)])
        # next step: 5 and 6 miss (evicting 1 and 2) and are taken in flight;
        # the upload of 6 fails
        got = [B.lora_assign(ctx, a, 16) for a in (5, 6)]
        assert got == [sim.assign(a, 16) for a in (5, 6)]
        slot5, slot6 = got[0][1], got[1][1]
        _run_script(ctx, sim, [("loaded", slot5), ("acquire", slot5), ("acquire", slot6), ("abort", slot6),
                               ("abort", slot5),          # its upload was queued: refused
                               ("release", slot6),        # the reference outlives the abort
                               ("release", slot6),        # ... once
                               ("release", slot5), ("tick",)])
        assert B.lora_lookup(ctx, 6) == -1 and B.lora_lookup(ctx, 5) == got[0][1]
        sim.lookup(5)
        assert [B.lora_lookup(ctx, a) for a in (3, 4)] == [sim.lookup(a) for a in (3, 4)]
        # the retry is a miss into the emptied slot, evicting nothing
        assert B.lora_assign(ctx, 6, 16) == sim.assign(6, 16) == (0, slot6, 1, -1)
        # out of range; the retried load of 6 fails again; then the slot is empty
        _run_script(ctx, sim, [("abort", 9), ("abort", slot6), ("abort", slot6), ("abort", slot5),
                               ("assign", 7, 16)])
        assert B.lora_stats(ctx)["aborted_loads"] == sim.aborted == 2
    finally:
        B.lora_destroy(ctx)


def test_late_release_after_abort_matches_simulator(lib):
    """Holder A's adapter is bound and referenced, its upload fails and is
    aborted; holder B's adapter is bound while A's reference stays (it cannot
    take A's slot), A releases late, and B's adapter stays protected from
    eviction while in flight. Every status and decision equals the simulator's."""
    from oracle.lru_sim import LruSlotSim
    ctx = _host_ctx(2, 16)
    sim = LruSlotSim(2, 16)
    try:
        _run_script(ctx, sim, [("assign", 10, 8), ("acquire", 0), ("abort", 0), ("acquire", 0),
                               ("assign", 20, 8), ("loaded", 1), ("acquire", 1), ("release", 0),
                               ("release", 0), ("assign", 30, 8), ("loaded", 0), ("evict",), ("evict",),
                               ("abort", 1), ("release", 1), ("evict",)])
        assert B.lora_lookup(ctx, 20) == sim.lookup(20) == -1
        assert sim.log[-1] == ("lookup", 20, -1)
    finally:
        B.lora_destroy(ctx)


def test_random_decisions_with_aborted_loads_match_simulator(lib):
    """Zipf admission with about one upload in ten failing (and aborted), plus
    in-flight references taken and dropped and explicit evictions: every
    decision, status and counter equal to the simulator's."""
    from oracle.lru_sim import LruSlotSim
    rng = np.random.default_rng(21)
    S, R = 6, 32
    ctx = _host_ctx(S, R)
    sim = LruSlotSim(S, R)
    try:
        ops = []
        for step in range(300):
            a = int(rng.zipf(1.3)) % 40
            ops.append(("assign", a, int(rng.choice([8, 16, 32]))))
            u = rng.random()
            if u < 0.12:                                 # the upload fails
                ops.append(("abort_last",))
            elif u < 0.8:                                # the upload is queued
                ops.append(("loaded_last",))
            r = rng.random()
            if r < 0.1:
                ops.append(("abort", int(rng.integers(0, S))))
            elif r < 0.12:
                ops.append(("loaded", int(rng.integers(-1, S + 1))))
            elif r < 0.15:
                ops.append(("evict",))
            elif r < 0.35:
                ops.append(("acquire", int(rng.integers(0, S))))
            elif r < 0.55:
                ops.append(("release", int(rng.integers(0, S))))
            if step % 7 == 0:
                ops.append(("tick",))
        _run_script(ctx, sim, ops)
        assert sim.aborted > 10
    finally:
        B.lora_destroy(ctx)


def _serve(ctx, ids, max_distinct=None):
    """lora_serve_step on a host-only context: (status, decisions, n_groups)."""
    import ctypes
    lib = B.load()
    T = len(ids)
    md = T if max_distinct is None else max_distinct
    arr = (ctypes.c_uint64 * max(1, T))(*[int(a) for a in ids])
    o_ids = (ctypes.c_uint64 * max(1, md))()
    o_sl = (ctypes.c_int * max(1, md))()
    o_nd = (ctypes.c_int * max(1, md))()
    o_ev = (ctypes.c_uint64 * max(1, md))()
    nd, ng = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib.lora_serve_step(ctx, T, arr, 0, None, None, None, None, 0, md, o_ids, o_sl, o_nd, o_ev,
                             ctypes.byref(nd), ctypes.byref(ng))
    dec = [(int(o_ids[i]), int(o_sl[i]), int(o_nd[i]), -1 if o_ev[i] == B.NO_ID else int(o_ev[i]))
           for i in range(nd.value)]
    return rc, dec, ng.value


def _serve_against_simulator(S, warm, steps):
    """Serve `steps` on a host-only context with warm set `warm` and replay
    them on the simulator, group by group as churn.plan_groups cuts them;
    every step must succeed with the simulator's decisions. Returns the
    number of groups of each step."""
    from oracle.lru_sim import LruSlotSim
    from rank_adapter_apply_gb300 import churn
    R = 16
    ctx = _host_ctx(S, R)
    sim = LruSlotSim(S, R)
    n_groups = []
    try:
        B.lora_register_host_adapters(ctx, list(range(20)), [8] * 20, [16.0] * 20)
        B.lora_set_warm_set(ctx, list(warm))
        pinned = {}
        for k, ids in enumerate(steps):
            rc, dec, ng = _serve(ctx, ids)
            assert rc == 0, (k, B.last_error())
            order = list(dict.fromkeys(a for a in ids if a != B.NO_ID))
            groups = churn.plan_groups(order, pinned, S - len(pinned), set(warm))
            exp = []
            for group in groups:
                held = []
                for a in group:
                    st, slot, need, ev = sim.assign(a, 8)
                    assert st == 0
                    exp.append((a, slot, need, ev))
                    if a in warm and a not in pinned:
                        sim.pin(slot)
                        pinned[a] = slot
                    sim.acquire(slot)
                    held.append(slot)
                for s_ in held:
                    sim.release(s_)
            sim.tick()
            assert dec == exp and ng == len(groups), (k, dec, exp)
            n_groups.append(ng)
        st = B.lora_stats(ctx)
        assert (st["hits"], st["misses"], st["evictions"], st["epoch"]) == \
            (sim.hits, sim.misses, sim.evictions, len(steps))
        assert st["uploads"] == sim.misses                  # host-only: uploads are recorded
    finally:
        B.lora_destroy(ctx)
    return n_groups


def test_serve_step_groups_and_decisions_match_simulator(lib):
    """A step with more distinct adapters than slots is cut into groups in
    first-appearance order (a warm-set adapter resident in a pinned slot needs
    no slot); each adapter's admission, in order, equals the simulator's; the
    epoch advances once per step; base-model tokens are skipped."""
    steps = [[0, 1, 2, B.NO_ID, 1, 3], [4, 5, 0, 6, 7, 8, 5, 9, 10], [0, 11, 12, 13, 14, 15, 16, 17, 0]]
    _serve_against_simulator(4, [0], steps)


def test_serve_step_warm_pins_leave_later_groups_fewer_slots(lib):
    """Warm-set adapters bound by a step's first group pin their slots, so the
    next group has that many evictable slots fewer: 4 slots, warm set {0, 1},
    seven new adapters in one step are served in groups of 4, 2 and 1 (cut
    at the start-of-step count, 4 and 3, the second group would find only two
    evictable slots and fail); later steps keep the two pinned slots."""
    steps = [[0, 1, 2, 3, 4, 5, 6], [7, 0, 8, 9, 1, 10], [11, 12, 13, 14, 15]]
    assert _serve_against_simulator(4, [0, 1], steps) == [3, 2, 3]


def test_serve_step_rejects_before_any_admission(lib):
    """An unregistered adapter id, more adapters than max_distinct, a bad
    registration: the call fails and the table is unchanged."""
    ctx = _host_ctx(4, 16)
    try:
        with pytest.raises(B.LoraError) as ei:                       # rank above max_lora_rank
            B.lora_register_host_adapters(ctx, [1, 2], [8, 32], [16.0, 16.0])
        assert ei.value.code == B.LORA_ERR_RANK
        with pytest.raises(B.LoraError):                             # an id twice
            B.lora_register_host_adapters(ctx, [1, 1], [8, 8], [16.0, 16.0])
        B.lora_register_host_adapters(ctx, [1, 2, 3], [8, 8, 8], [16.0, 16.0, 16.0])
        rc, dec, ng = _serve(ctx, [1, 7, 2])                          # 7 was never registered
        assert rc == B.LORA_ERR_ARG and "not registered" in B.last_error()
        rc, dec, ng = _serve(ctx, [1, 2, 3], max_distinct=2)
        assert rc == B.LORA_ERR_ARG
        st = B.lora_stats(ctx)
        assert (st["hits"], st["misses"], st["epoch"]) == (0, 0, 0)
        rc, dec, ng = _serve(ctx, [])                                 # an empty step only ticks
        assert rc == 0 and dec == [] and ng == 0 and B.lora_stats(ctx)["epoch"] == 1
    finally:
        B.lora_destroy(ctx)


@pytest.mark.parametrize("seed", range(8))
def test_serve_step_random_steps_match_simulator(lib, seed):
    """Random serving steps on 2-8 slots: ids from a small pool with base-model
    tokens mixed in, often more distinct adapters than slots (several groups
    per step), a warm set of up to max_loras - 1 adapters, LRU or keep_score.
    Every step succeeds, and every admission equals the simulator's replay of
    the groups that churn.plan_groups cuts (the warm adapters pinned as they
    are bound)."""
    from oracle.lru_sim import KEEP_SCORE, LRU
    from rank_adapter_apply_gb300 import churn
    rng = np.random.default_rng(1000 + seed)
    S, R = int(rng.integers(2, 9)), 16
    n_ad = int(rng.integers(S + 2, 4 * S + 3))
    ranks = [int(r) for r in rng.integers(1, R + 1, size=n_ad)]
    warm = set(int(a) for a in rng.choice(n_ad, size=int(rng.integers(0, S)), replace=False))
    policy = LRU if seed % 2 == 0 else KEEP_SCORE
    weights = (1.0, 1.0, 0.5, 0.25, 0.75)
    ctx = _host_ctx(S, R)
    sim = LruSlotSim(S, R)
    sim.policy = policy
    sim.weights = weights
    try:
        B.lora_set_policy(ctx, policy)
        B.lora_set_keep_score_weights(ctx, weights)
        B.lora_register_host_adapters(ctx, list(range(n_ad)), ranks, [2.0 * r for r in ranks])
        B.lora_set_warm_set(ctx, sorted(warm))
        pinned = {}
        for k in range(25):
            T = int(rng.integers(1, 3 * S + 4))
            ids = [B.NO_ID if rng.random() < 0.15 else int(rng.integers(0, n_ad)) for _ in range(T)]
            rc, dec, ng = _serve(ctx, ids)
            assert rc == 0, (seed, k, B.last_error())
            order = list(dict.fromkeys(a for a in ids if a != B.NO_ID))
            groups = churn.plan_groups(order, pinned, S - len(pinned), warm)
            exp = []
            for group in groups:
                held = []
                for a in group:
                    st, slot, need, ev = sim.assign(a, ranks[a])
                    assert st == 0, (seed, k, a)
                    exp.append((a, slot, need, ev))
                    if a in warm and a not in pinned:
                        sim.pin(slot)
                        pinned[a] = slot
                    sim.acquire(slot)
                    held.append(slot)
                for s_ in held:
                    sim.release(s_)
            sim.tick()
            assert dec == exp and ng == len(groups), (seed, k, dec, exp)
        st = B.lora_stats(ctx)
        assert (st["hits"], st["misses"], st["evictions"]) == (sim.hits, sim.misses, sim.evictions)
    finally:
        B.lora_destroy(ctx)


def test_serve_step_failed_admission_uploads_the_bound_misses(lib):
    """A group whose second admission fails: the miss bound before it is still
    uploaded (its slot is loaded, so lora_abort_load refuses it and a later
    step finds it resident with its weights), every reference of the step is
    released, the epoch stays."""
    ctx = _host_ctx(2, 16)
    try:
        B.lora_register_host_adapters(ctx, [1, 2, 3], [8, 8, 8], [16.0] * 3)
        st, held, need, ev = B.lora_assign(ctx, 1, 8)
        B.lora_acquire(ctx, held)                                     # slot of 1 in flight elsewhere
        up0 = B.lora_stats(ctx)["uploads"]
        rc, dec, ng = _serve(ctx, [2, 3])                             # 2 binds the free slot, 3 finds none
        assert rc == B.LORA_ERR_NO_SLOT
        slot2 = B.lora_lookup(ctx, 2)
        assert slot2 >= 0 and slot2 != held and B.lora_lookup(ctx, 3) == -1
        assert B.lora_stats(ctx)["uploads"] == up0 + 1
        assert B.lora_abort_load(ctx, slot2)[0] == B.LORA_ERR_STATE    # loaded, not pending
        assert B.lora_release(ctx, slot2) == B.LORA_ERR_STATE          # the step's reference is gone
        assert B.lora_stats(ctx)["epoch"] == 0
        assert B.lora_release(ctx, held) == 0
        rc, dec, ng = _serve(ctx, [2, 3])                             # now both fit
        assert rc == 0 and [d[2] for d in dec] == [0, 1]              # 2 resident (hit), 3 uploaded
    finally:
        B.lora_destroy(ctx)


def test_serve_step_no_slot_releases_its_group(lib):
    """Every slot in flight elsewhere: the first admission of the step fails
    with NO_SLOT, the step's own references are released, the epoch stays."""
    ctx = _host_ctx(2, 16)
    try:
        B.lora_register_host_adapters(ctx, [1, 2, 3], [8, 8, 8], [16.0] * 3)
        for a in (1, 2):
            st, slot, need, ev = B.lora_assign(ctx, a, 8)
            B.lora_acquire(ctx, slot)                                 # held by another request
        rc, dec, ng = _serve(ctx, [1, 3])
        assert rc == B.LORA_ERR_NO_SLOT
        assert B.lora_release(ctx, 0) == 0 and B.lora_release(ctx, 1) == 0
        assert B.lora_release(ctx, 0) == B.LORA_ERR_STATE            # no reference left behind
        assert B.lora_stats(ctx)["epoch"] == 0
    finally:
        B.lora_destroy(ctx)
