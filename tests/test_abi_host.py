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


def _run_script(ctx, sim, ops):
    for op in ops:
        kind = op[0]
        if kind == "assign":
            got = B.lora_assign(ctx, op[1], op[2])
            exp = sim.assign(op[1], op[2])
            assert got == exp, (op, got, exp)
        elif kind == "lookup":
            assert B.lora_lookup(ctx, op[1]) == sim.lookup(op[1]), op
        elif kind == "acquire":
            assert B.lora_acquire(ctx, op[1]) == sim.acquire(op[1]), op
        elif kind == "release":
            assert B.lora_release(ctx, op[1]) == sim.release(op[1]), op
        elif kind == "evict":
            assert B.lora_evict_lru(ctx) == sim.evict_lru(), op
        elif kind == "tick":
            B.lora_tick(ctx)
            sim.tick()
    st = B.lora_stats(ctx)
    assert (st["hits"], st["misses"], st["evictions"], st["reloads_after_eviction"],
            st["rejected"]) == (sim.hits, sim.misses, sim.evictions, sim.reloads, sim.rejected)


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
