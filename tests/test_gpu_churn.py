"""Slot churn on the GPU: 64 slots, 512 host adapters, Zipf(1.2) ids with cold
bursts. Every eviction decision matches the independent LRU simulator bit for
bit, and the deltas of checked steps match the oracle computed directly from
the adapter ids (independent of the slot mapping)."""
import numpy as np
import pytest

import oracle
from oracle.lru_sim import LruSlotSim
from rank_adapter_apply_gb300 import workloads as wl
from tests.parity_util import TOL, decode

pytestmark = pytest.mark.gpu


def _sim_decisions(trace, S, R):
    sim = LruSlotSim(S, R)
    out = []
    for k, ids in enumerate(trace.steps):
        order = list(dict.fromkeys(int(a) for a in ids))
        for g0 in range(0, len(order), S):
            group = order[g0:g0 + S]
            held = []
            for a in group:
                st, slot, need, ev = sim.assign(a, R)
                out.append((k, a, st, slot, need, ev))
                sim.acquire(slot)
                held.append(slot)
            for s in held:
                sim.release(s)
        sim.tick()
    return out, sim


def _check_step(runner, n_adapters, R, alpha):
    ids, slot_tok, ys = runner.checked
    host = runner.host_np
    idx = np.asarray(ids, np.int32)
    for li, name in enumerate(runner.layers):
        A = host[name][0]                       # [n, r, d]: pool indexed by adapter id
        B = np.ascontiguousarray(host[name][1])
        ref = oracle.lora_apply_ref(runner.x_np, runner.y_np[li], A, B,
                                    np.full(n_adapters, R, np.int32), np.full(n_adapters, alpha), idx)
        got = decode(ys[li].view(np.int16).numpy().view(np.uint16) if hasattr(ys[li], "numpy") else ys[li],
                     wl.DTYPE_BF16)
        atol, rtol = TOL[wl.DTYPE_BF16]
        assert np.all(np.abs(got - ref) <= atol + rtol * np.abs(ref)), name


def test_churn_decisions_and_outputs():
    import torch
    from rank_adapter_apply_gb300 import build
    from rank_adapter_apply_gb300.churn import ChurnRunner
    build.build()
    n_adapters, S, R, steps = 512, 64, 16, 60
    trace = wl.churn_trace(0, n_adapters=n_adapters, n_steps=steps, burst_every=20)
    r = ChurnRunner(n_adapters=n_adapters, max_loras=S, rank=R)
    try:
        res = r.run(trace, record=True, check_step=40)
        exp, sim = _sim_decisions(trace, S, R)
        assert res.decisions == exp
        st = res.stats
        assert (st["hits"], st["misses"], st["evictions"], st["reloads_after_eviction"]) == \
               (sim.hits, sim.misses, sim.evictions, sim.reloads)
        assert st["uploads"] == sim.misses
        assert st["upload_bytes"] == sim.misses * 524_288
        assert st["device_wait_timeouts"] == 0 and st["invalid_token_index"] == 0
        ids, slot_tok, ys = r.checked
        ys_np = [y.view(torch.int16).numpy().view(np.uint16) for y in ys]
        r.checked = (ids, slot_tok, ys_np)
        _check_step(r, n_adapters, R, 32.0)
    finally:
        r.close()


def test_churn_overlap_tracking_outputs_and_decisions():
    """Uploads ordered per slot (slot tracking) with the host running ahead of
    the GPU: the same decisions, and a checked step still matches the oracle."""
    import torch
    from rank_adapter_apply_gb300 import build
    from rank_adapter_apply_gb300.churn import ChurnRunner
    build.build()
    n_adapters, S, R, steps = 512, 64, 16, 45
    trace = wl.churn_trace(1, n_adapters=n_adapters, n_steps=steps, burst_every=15)
    r = ChurnRunner(n_adapters=n_adapters, max_loras=S, rank=R, overlap=True)
    try:
        res = r.run(trace, record=True, check_step=31)
        exp, sim = _sim_decisions(trace, S, R)
        assert res.decisions == exp
        st = res.stats
        assert st["device_wait_timeouts"] == 0 and st["uploads"] == sim.misses
        ids, slot_tok, ys = r.checked
        r.checked = (ids, slot_tok, [y.view(torch.int16).numpy().view(np.uint16) for y in ys])
        _check_step(r, n_adapters, R, 32.0)
    finally:
        r.close()


def test_churn_pinned_warm_set_and_keep_score_outputs():
    """Policies on the GPU path: decisions equal the simulator's replay and the
    checked step matches the oracle."""
    import torch
    from rank_adapter_apply_gb300 import build
    from rank_adapter_apply_gb300 import churn
    build.build()
    n_adapters, S, R, steps = 512, 64, 16, 40
    trace = wl.churn_trace(2, n_adapters=n_adapters, n_steps=steps, burst_every=20)
    for kw in ({"pin_top": 16}, {"policy": 1, "weights": (1.0, 1.0, 0.0, 0.0, 0.0)}):
        r = churn.ChurnRunner(n_adapters=n_adapters, max_loras=S, rank=R, **kw)
        try:
            res = r.run(trace, record=True, check_step=25)
            host = churn.admission_stats(trace, max_loras=S, rank=R, record=True, **kw)
            assert res.decisions == host["log"]
            ids, slot_tok, ys = r.checked
            r.checked = (ids, slot_tok, [y.view(torch.int16).numpy().view(np.uint16) for y in ys])
            _check_step(r, n_adapters, R, 32.0)
        finally:
            r.close()
