"""Slot-churn driver: decode steps whose adapters come and go.

Each step is one lora_serve_step call: the batch's tokens name their
adapters, and the library cuts the step's distinct adapters (first-appearance
order) into groups that fit the max_loras slots ("Multi-LoRA 适配器缓存生产实战"
page, section 核心原理, parameter table); for every group it
  1. assigns each adapter a slot (hit: touch; miss: free slot or the policy's
     victim among slots not in flight) and takes an in-flight reference,
  2. uploads the missing adapters from the pinned host store registered once
     (tier L1, CPU hit -> H2D upload, section 冷加载延迟),
  3. applies the delta to q_proj and v_proj for the group's tokens,
  4. releases the references;
then advances the epoch (the thrash window counts epochs). This module only
moves data and calls the C ABI.

`admission_stats` replays the same steps on a host-only context (no GPU) to
compare the eviction policies of the section 为什么纯 LRU 在多租户场景下容易
失效: pure LRU, a pinned warm set of the most popular adapters, and keep_score.
`plan_groups` / `plan_step` restate the grouping rule in Python for the tests
(an independent statement of what the library does inside lora_serve_step).
"""
from __future__ import annotations

import ctypes

import time
from dataclasses import dataclass, field

import numpy as np
import torch

from . import binding as B
from . import workloads as wl
from .harness import to_torch
from .slots import LoraSlots


# A warm set of the 32 most popular adapters (ids 0..31 of the Zipf trace)
# with keep_score weights (1, 1, 0, 0, 0) over a 40-epoch frequency window:
# on the churn trace this takes 99.7 % of the hits of an offline replay that
# evicts the adapter used farthest in the future (pure LRU: 31 %).
KEEP_PIN32 = {"policy": 1, "weights": (1.0, 1.0, 0.0, 0.0, 0.0), "pin_top": 32, "window": 40}


def plan_groups(order, pinned_resident, capacity, warm=()):
    """Split a step's distinct adapters (first-appearance order) into groups:
    every adapter not already resident in a pinned slot needs one of
    `capacity` evictable slots (max_loras minus the pinned ones). A warm-set
    adapter outside the pinned slots pins its slot when its group is
    admitted, which leaves one evictable slot fewer to every later group."""
    groups, cur, cost, new_pins = [], [], 0, 0
    for a in order:
        c = 0 if a in pinned_resident else 1
        if cur and cost + c > capacity:
            groups.append(cur)
            cur, cost = [], 0
            capacity -= new_pins
            new_pins = 0
        cur.append(a)
        cost += c
        if c and a in warm:
            new_pins += 1
    if cur:
        groups.append(cur)
    return groups


def plan_step(ids, pinned_resident, capacity, warm=()):
    """A step's distinct adapters in first-appearance order, cut into groups by
    plan_groups, and the group of every token (numpy int32 per token). Plain
    dict passes over the few hundred tokens of a step: cheaper than sorting
    them with numpy."""
    ids_l = np.asarray(ids).tolist()
    groups = plan_groups(list(dict.fromkeys(ids_l)), pinned_resident, capacity, warm)
    group_of = {a: gi for gi, g in enumerate(groups) for a in g}
    return groups, np.fromiter(map(group_of.__getitem__, ids_l), dtype=np.int32, count=len(ids_l))


def _serve_outputs(T):
    """ctypes output arrays for lora_serve_step (up to T distinct adapters)."""
    ids = (ctypes.c_uint64 * T)()
    slots = (ctypes.c_int * T)()
    need = (ctypes.c_int * T)()
    ev = (ctypes.c_uint64 * T)()
    return ids, slots, need, ev, ctypes.c_int(0), ctypes.c_int(0)


def _decisions(k, out, n):
    ids, slots, need, ev = out[:4]
    return [(k, int(ids[i]), 0, int(slots[i]), int(need[i]), -1 if ev[i] == B.NO_ID else int(ev[i]))
            for i in range(n)]


def admission_stats(trace, max_loras=64, rank=16, policy=0, weights=None, pin_top=0,
                    min_residency=0, window=10, record=False):
    """Host-only replay of the churn admission through lora_serve_step: per
    step, groups of adapters are assigned (hit: touch; miss: free slot or
    policy victim), acquired, then released; adapters with id < pin_top form
    the warm set (pinned when bound). Returns the slot-table statistics (and
    the decision log if record)."""
    ctx = B.lora_slots_init(max_loras, rank, 0, 1, B.LORA_DTYPE_BF16, [], None, None, None, 0,
                            None, None)
    lib = B.load()
    log = []
    try:
        B.lora_set_thrash_window(ctx, window)
        B.lora_set_policy(ctx, policy)
        if weights is not None:
            B.lora_set_keep_score_weights(ctx, weights)
        B.lora_set_min_residency(ctx, min_residency)
        n = trace.n_adapters
        B.lora_register_host_adapters(ctx, list(range(n)), [rank] * n, [2.0 * rank] * n)
        B.lora_set_warm_set(ctx, list(range(min(pin_top, n))))
        T = max(len(ids) for ids in trace.steps)
        out = _serve_outputs(T)
        for k, ids in enumerate(trace.steps):
            ids_u = np.ascontiguousarray(ids, dtype=np.uint64)
            rc = lib.lora_serve_step(ctx, len(ids_u), ids_u.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                                     0, None, None, None, None, 0, T, out[0], out[1], out[2], out[3],
                                     ctypes.byref(out[4]), ctypes.byref(out[5]))
            if rc != 0:
                raise RuntimeError(f"step {k}: {B.last_error()}")
            if record:
                log += _decisions(k, out, out[4].value)
        st = B.lora_stats(ctx)
        # warm-set adapters stay resident once bound (pinned slots are never
        # evicted): the pinned count is the number of them resident now
        pinned = sum(1 for a in range(min(pin_top, n)) if B.lora_lookup(ctx, a) >= 0)
    finally:
        B.lora_destroy(ctx)
    st["hit_rate"] = st["hits"] / max(1, st["hits"] + st["misses"])
    st["thrash_ratio"] = st["reloads_after_eviction"] / st["evictions"] if st["evictions"] else 0.0
    st["pinned"] = pinned
    if record:
        st["log"] = log
    return st


@dataclass
class ChurnResult:
    steps: int
    wall_s: float
    stats: dict
    decisions: list = field(default_factory=list)   # (step, adapter, status, slot, needs_load, evicted)
    tokens: int = 0


class ChurnRunner:
    """The churn workload on the GPU: 512 rank-16 adapters in pinned host
    memory registered once as the library's host store, 64 slots, q_proj and
    v_proj 4096 -> 4096; one lora_serve_step per decode step."""

    def __init__(self, n_adapters=512, max_loras=64, rank=16, d=4096, tokens=256, seed=0,
                 device="cuda:0", alpha=32.0, policy=0, weights=None, pin_top=0, overlap=False,
                 window=None):
        self.dev = torch.device(device)
        self.S, self.R, self.d, self.T = max_loras, rank, d, tokens
        self.n_adapters = n_adapters
        self.alpha = alpha
        host = wl.churn_adapters(seed, n_adapters, d, rank)
        # pinned host adapter store: per adapter, per layer A [r, d], B [d, r]
        self.A = {k: to_torch(v[0], wl.DTYPE_BF16).pin_memory() for k, v in host.items()}
        self.B = {k: to_torch(v[1], wl.DTYPE_BF16).pin_memory() for k, v in host.items()}
        self.host_np = host
        self.layers = ["q_proj", "v_proj"]
        self.slots = LoraSlots([(d, d), (d, d)], max_loras, rank, tokens, dtype=torch.bfloat16,
                               device=self.dev)
        ctx = self.slots.ctx
        B.lora_set_policy(ctx, policy)
        if weights is not None:
            B.lora_set_keep_score_weights(ctx, weights)
        if window is not None:
            B.lora_set_thrash_window(ctx, window)
        # the host store (adapter-major pointers, one per layer) and the warm set
        A_ptr = [self.A[l][a].data_ptr() for a in range(n_adapters) for l in self.layers]
        B_ptr = [self.B[l][a].data_ptr() for a in range(n_adapters) for l in self.layers]
        B.lora_register_host_adapters(ctx, list(range(n_adapters)), [rank] * n_adapters,
                                      [alpha] * n_adapters, A_ptr, B_ptr)
        B.lora_set_warm_set(ctx, list(range(min(pin_top, n_adapters))))
        # overlap: uploads wait only for the applies that used their slot, and
        # the host runs ahead of the GPU (slot-id buffers rotate over 4 steps)
        self.overlap = overlap
        if overlap:
            B.lora_set_slot_tracking(ctx, True)
        self.ring = 4 if overlap else 1
        rng = np.random.default_rng(seed + 7)
        xf = rng.standard_normal((tokens, d), dtype=np.float32)
        self.x_np = wl.f32_to_bf16_bits(xf)
        self.y_np = [wl.f32_to_bf16_bits(rng.standard_normal((tokens, d), dtype=np.float32)
                                         * np.float32(0.02 * np.sqrt(d))) for _ in self.layers]
        self.x = to_torch(self.x_np, wl.DTYPE_BF16).to(self.dev)
        self.y0 = [to_torch(v, wl.DTYPE_BF16).to(self.dev) for v in self.y_np]
        self.y = [t.clone() for t in self.y0]
        # slot-id buffers of a step: one per adapter group (a step has at most
        # ceil(tokens / evictable slots) groups), pinned host memory the
        # kernels read; a ring slot is reused only after its step has finished
        self.max_groups = (tokens + max(1, max_loras - pin_top) - 1) // max(1, max_loras - pin_top)
        self.idx_host = torch.empty((self.ring, self.max_groups, tokens), dtype=torch.int32).pin_memory()
        self.step_done = [False] * self.ring     # ring slot's event recorded and not yet waited for
        self._lay = B._i32_array([0, 1])
        self._xs = B._vp_array([self.x.data_ptr()] * 2)
        self._ys = B._vp_array([t.data_ptr() for t in self.y])
        self._out = _serve_outputs(tokens)
        # per ring slot: the step's adapter ids as the ABI takes them, the
        # address of its slot-id buffers, and an event marking its kernels
        self._ids = [(ctypes.c_uint64 * tokens)() for _ in range(self.ring)]
        self._ids_np = [np.frombuffer(b, dtype=np.uint64) for b in self._ids]
        self._idx_ptr = [self.idx_host[rb].data_ptr() for rb in range(self.ring)]
        self._events = [torch.cuda.Event() for _ in range(self.ring)]

    def run(self, trace: wl.ChurnTrace, record=False, reset_y=True, check_step=None):
        """Run every step of the trace; returns ChurnResult. With check_step=k
        the outputs of step k (y after that step, starting from the base
        outputs) are kept in self.checked = (ids, slot_of_token, y_q, y_v)."""
        decisions = []
        ctx = self.slots.ctx
        serve = B.load().lora_serve_step
        out = self._out
        n_dist, n_grp = ctypes.byref(out[4]), ctypes.byref(out[5])
        compute = self.slots.compute
        # adapter tokens of the trace (the metric's count, not work of a step)
        no_id = np.uint64(B.NO_ID)
        tokens = sum(int(np.count_nonzero(np.asarray(ids, dtype=np.uint64) != no_id)) for ids in trace.steps)
        torch.cuda.synchronize(self.dev)
        t0 = time.perf_counter()
        for k, ids in enumerate(trace.steps):
            rb = k % self.ring
            if self.step_done[rb]:
                self._events[rb].synchronize()          # this step's slot-id buffers are free
                self.step_done[rb] = False
            if reset_y or k == check_step:
                with torch.cuda.stream(compute):
                    for y, y0 in zip(self.y, self.y0):
                        y.copy_(y0)
            n_ids = len(ids)
            self._ids_np[rb][:n_ids] = ids
            rc = serve(ctx, n_ids, self._ids[rb], 2, self._lay, self._xs, self._ys, self._idx_ptr[rb],
                       self.max_groups, self.T, out[0], out[1], out[2], out[3], n_dist, n_grp)
            if rc != 0:
                raise RuntimeError(f"step {k}: {B.last_error()}")
            n = out[4].value
            if record:
                decisions += _decisions(k, out, n)
            ev = self._events[rb]
            ev.record(compute)
            if not self.overlap or k == check_step:
                ev.synchronize()                    # slot-id buffers are reused next step
            else:
                self.step_done[rb] = True
            if k == check_step:
                slot_of = {int(out[0][i]): int(out[1][i]) for i in range(n)}
                slot_tok = np.array([slot_of.get(int(a), -1) for a in ids], np.int32)
                self.checked = (ids.copy(), slot_tok, [y.clone().cpu() for y in self.y])
        self.slots.compute.synchronize()
        self.slots.sync_uploads()
        wall = time.perf_counter() - t0
        st = self.slots.stats()
        return ChurnResult(len(trace.steps), wall, st, decisions, tokens)

    def close(self):
        self.slots.close()
