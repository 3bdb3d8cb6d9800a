"""Slot-churn driver: decode steps whose adapters come and go.

Each step takes a batch of tokens with adapter ids, and for every group of at
most max_loras distinct adapters (first-appearance order; max_loras bounds the
adapters one batch may use, "Multi-LoRA 适配器缓存生产实战" page, section
核心原理, parameter table):
  1. assigns each adapter a slot (hit: touch; miss: free slot or LRU victim
     that is not in flight) and takes an in-flight reference,
  2. uploads the missing adapters from pinned host memory (tier L1, CPU hit ->
     H2D upload, section 冷加载延迟),
  3. applies the delta to q_proj and v_proj for the group's tokens,
  4. releases the references.
The epoch advances once per step (the thrash window counts epochs). Every
decision goes through the C ABI; this module only moves data.

`admission_stats` replays the same admission on a host-only context (no GPU)
to compare the eviction policies of the section 为什么纯 LRU 在多租户场景下容易
失效: pure LRU, a pinned warm set of the most popular adapters, and keep_score.
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


def plan_groups(order, pinned_resident, capacity):
    """Split a step's distinct adapters (first-appearance order) into groups:
    every adapter not already resident in a pinned slot needs one of
    `capacity` evictable slots (max_loras minus the pinned ones)."""
    groups, cur, cost = [], [], 0
    for a in order:
        c = 0 if a in pinned_resident else 1
        if cur and cost + c > capacity:
            groups.append(cur)
            cur, cost = [], 0
        cur.append(a)
        cost += c
    if cur:
        groups.append(cur)
    return groups


def plan_step(ids, pinned_resident, capacity):
    """A step's distinct adapters in first-appearance order, cut into groups by
    plan_groups, and the group of every token (numpy int32 per token). Plain
    dict passes over the few hundred tokens of a step: cheaper than sorting
    them with numpy."""
    ids_l = np.asarray(ids).tolist()
    groups = plan_groups(list(dict.fromkeys(ids_l)), pinned_resident, capacity)
    group_of = {a: gi for gi, g in enumerate(groups) for a in g}
    return groups, np.fromiter(map(group_of.__getitem__, ids_l), dtype=np.int32, count=len(ids_l))


def admission_stats(trace, max_loras=64, rank=16, policy=0, weights=None, pin_top=0,
                    min_residency=0, window=10, record=False):
    """Host-only replay of the churn admission: per step, groups of adapters are
    assigned (hit: touch; miss: free slot or policy victim), acquired, then
    released; adapters with id < pin_top are pinned when first bound (the warm
    set). Returns the slot-table statistics (and the decision log if record)."""
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
        pinned = {}
        for k, ids in enumerate(trace.steps):
            order = list(dict.fromkeys(int(a) for a in ids))
            for group in plan_groups(order, pinned, max_loras - len(pinned)):
                held = []
                for a in group:
                    st, slot, need, ev = B.lora_assign(ctx, a, rank)
                    if record:
                        log.append((k, a, st, slot, need, ev))
                    if st != 0:
                        raise RuntimeError(f"assign failed for adapter {a}: {st}")
                    if a < pin_top and a not in pinned:
                        B.check(B.lora_pin(ctx, slot, True))
                        pinned[a] = slot
                    lib.lora_acquire(ctx, slot)
                    held.append(slot)
                for sl in held:
                    lib.lora_release(ctx, sl)
            B.lora_tick(ctx)
        st = B.lora_stats(ctx)
    finally:
        B.lora_destroy(ctx)
    st["hit_rate"] = st["hits"] / max(1, st["hits"] + st["misses"])
    st["thrash_ratio"] = st["reloads_after_eviction"] / st["evictions"] if st["evictions"] else 0.0
    st["pinned"] = len(pinned)
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
    def __init__(self, n_adapters=512, max_loras=64, rank=16, d=4096, tokens=256, seed=0,
                 device="cuda:0", alpha=32.0, policy=0, weights=None, pin_top=0, overlap=False,
                 batched_upload=True, window=None):
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
        B.lora_set_policy(self.slots.ctx, policy)
        if weights is not None:
            B.lora_set_keep_score_weights(self.slots.ctx, weights)
        if window is not None:
            B.lora_set_thrash_window(self.slots.ctx, window)
        self.pin_top = pin_top
        self.pinned = {}
        # overlap: uploads wait only for the applies that used their slot, and
        # the host runs ahead of the GPU (slot-id buffers rotate over 4 steps)
        self.overlap = overlap
        # batched: one lora_load_slots per group (one kernel reads the host
        # adapters); otherwise one lora_load_slot (copy engine) per adapter
        self.batched_upload = batched_upload
        if overlap:
            B.lora_set_slot_tracking(self.slots.ctx, True)
        self.ring = 4 if overlap else 1
        rng = np.random.default_rng(seed + 7)
        xf = rng.standard_normal((tokens, d), dtype=np.float32)
        self.x_np = wl.f32_to_bf16_bits(xf)
        self.y_np = [wl.f32_to_bf16_bits(rng.standard_normal((tokens, d), dtype=np.float32)
                                         * np.float32(0.02 * np.sqrt(d))) for _ in self.layers]
        self.x = to_torch(self.x_np, wl.DTYPE_BF16).to(self.dev)
        self.y0 = [to_torch(v, wl.DTYPE_BF16).to(self.dev) for v in self.y_np]
        self.y = [t.clone() for t in self.y0]
        # one slot-id buffer per adapter group of a step (a step has at most
        # ceil(tokens / evictable slots) groups); reused only after the step's sync
        self.max_groups = (tokens + max(1, max_loras - pin_top) - 1) // max(1, max_loras - pin_top)
        self.idx_host = torch.empty((self.ring, self.max_groups, tokens), dtype=torch.int32).pin_memory()
        self.step_done = [None] * self.ring
        # call arguments built once: host pointers of every adapter's A and B
        # per layer (adapter-major rows), the layer list and x / y pointers
        self.A_ptr = np.array([[self.A[l][a].data_ptr() for l in self.layers] for a in range(n_adapters)],
                              dtype=np.uint64)
        self.B_ptr = np.array([[self.B[l][a].data_ptr() for l in self.layers] for a in range(n_adapters)],
                              dtype=np.uint64)
        self._lay = B._i32_array([0, 1])
        self._xs = B._vp_array([self.x.data_ptr()] * 2)
        self._ys = B._vp_array([t.data_ptr() for t in self.y])
        S = max_loras
        self._dids = np.zeros(S, np.uint64)
        self._slots = np.zeros(S, np.int32)
        self._need = np.zeros(S, np.int32)
        self._ev = np.zeros(S, np.uint64)
        P = ctypes.POINTER
        self._dids_p = self._dids.ctypes.data_as(P(ctypes.c_uint64))
        self._slots_p = self._slots.ctypes.data_as(P(ctypes.c_int))
        self._need_p = self._need.ctypes.data_as(P(ctypes.c_int))
        self._ev_p = self._ev.ctypes.data_as(P(ctypes.c_uint64))
        self._ranks = np.full(tokens, rank, np.int32)
        self._ranks_p = self._ranks.ctypes.data_as(P(ctypes.c_int))
        self._alphas = np.full(S, alpha, np.float32)
        self._alphas_p = self._alphas.ctypes.data_as(P(ctypes.c_float))
        # per-call buffers as ctypes arrays with numpy views over them (filled
        # through the views, handed to the library as they are)
        nl = len(self.layers)
        self._gids_c = (ctypes.c_uint64 * tokens)()
        self._gids = np.frombuffer(self._gids_c, dtype=np.uint64)
        self._sl_c = (ctypes.c_int * S)()
        self._sl = np.frombuffer(self._sl_c, dtype=np.int32)
        self._ap_c = (ctypes.c_void_p * (S * nl))()
        self._ap = np.frombuffer(self._ap_c, dtype=np.uint64)
        self._bp_c = (ctypes.c_void_p * (S * nl))()
        self._bp = np.frombuffer(self._bp_c, dtype=np.uint64)
        self._nd, self._done = ctypes.c_int(0), ctypes.c_int(0)
        self._nd_r, self._done_r = ctypes.byref(self._nd), ctypes.byref(self._done)
        self._idx_np = [[self.idx_host[rb, gi].numpy() for gi in range(self.max_groups)] for rb in range(self.ring)]
        self._idx_p = [[ctypes.cast(self.idx_host[rb, gi].data_ptr(), P(ctypes.c_int)) for gi in range(self.max_groups)]
                       for rb in range(self.ring)]
        self._idx_addr = [[self.idx_host[rb, gi].data_ptr() for gi in range(self.max_groups)] for rb in range(self.ring)]

    def upload(self, slot, adapter):
        a = [self.A[l][adapter] for l in self.layers]
        b = [self.B[l][adapter] for l in self.layers]
        self.slots.load_slot(slot, a, b, self.R, self.alpha)

    def run(self, trace: wl.ChurnTrace, record=False, reset_y=True, check_step=None):
        """Run every step of the trace; returns ChurnResult. With check_step=k
        the outputs of step k (y after that step's groups, starting from the
        base outputs) are kept in self.checked = (ids, slot_of_token, y_q, y_v)."""
        decisions = []
        tokens = 0
        ctx = self.slots.ctx
        lib = B.load()
        torch.cuda.synchronize(self.dev)
        t0 = time.perf_counter()
        for k, ids in enumerate(trace.steps):
            rb = k % self.ring
            if self.step_done[rb] is not None:
                self.step_done[rb].synchronize()          # this step's slot-id buffers are free
            if reset_y or k == check_step:
                with torch.cuda.stream(self.slots.compute):
                    for y, y0 in zip(self.y, self.y0):
                        y.copy_(y0)
            groups, tok_group = plan_step(ids, self.pinned, self.S - len(self.pinned))
            ids_u = ids.astype(np.uint64)
            slot_tok = np.full(self.T, -1, np.int32)
            for gi, group in enumerate(groups):
                # admit the group's adapters and map its tokens in one call:
                # assign (hit: touch; miss: free slot or policy victim), take an
                # in-flight reference, write every token's slot id (-1: not in
                # this group) straight into the pinned slot-id buffer
                np.copyto(self._gids, np.where(tok_group == gi, ids_u, np.uint64(B.NO_ID)))
                idx_h = self._idx_np[rb][gi]
                rc = lib.lora_assign_tokens(ctx, self.T, self._gids_c, self._ranks_p, 1, self._idx_p[rb][gi],
                                            self.S, self._dids_p, self._slots_p, self._need_p, self._ev_p,
                                            self._nd_r, self._done_r)
                n = self._nd.value
                if rc != 0:
                    raise RuntimeError(f"assign failed for adapter {group[self._done.value]}: {rc}")
                slots, need = self._slots[:n], self._need[:n]
                if record:
                    decisions += [(k, a, 0, int(sl), int(nd_), -1 if ev_ == np.uint64(B.NO_ID) else int(ev_))
                                  for a, sl, nd_, ev_ in zip(group, slots, need, self._ev[:n])]
                if self.pin_top:
                    for a, sl in zip(group, slots):
                        if a < self.pin_top and a not in self.pinned:
                            B.check(B.lora_pin(ctx, int(sl), True))
                            self.pinned[a] = int(sl)
                miss = np.nonzero(need)[0]
                if len(miss) and self.batched_upload:
                    ad = np.asarray(group, dtype=np.int64)[miss]
                    m = len(miss)
                    nl = len(self.layers)
                    self._sl[:m] = slots[miss]
                    self._ap[:m * nl] = self.A_ptr[ad].ravel()
                    self._bp[:m * nl] = self.B_ptr[ad].ravel()
                    B.check(lib.lora_load_slots(ctx, m, self._sl_c, self._ap_c, self._bp_c, self._ranks_p,
                                                self._alphas_p))
                else:
                    for i in miss:
                        self.upload(int(slots[i]), group[i])
                sel = idx_h >= 0
                slot_tok[sel] = idx_h[sel]
                # the kernels read the slot ids straight from the pinned buffer
                # (same address on the device; it is rewritten only after the
                # step that used it has finished)
                B.check(lib.lora_apply_multi(ctx, 2, self._lay, self._xs, self._ys, self._idx_addr[rb][gi], self.T))
                B.check(lib.lora_release_batch(ctx, n, self._slots_p))
                tokens += int(sel.sum())
            ev = torch.cuda.Event()
            ev.record(self.slots.compute)
            self.step_done[rb] = ev
            if not self.overlap or k == check_step:
                ev.synchronize()                    # slot-id buffers are reused next step
            if k == check_step:
                self.checked = (ids.copy(), slot_tok, [y.clone().cpu() for y in self.y])
            B.lora_tick(ctx)
        self.slots.compute.synchronize()
        self.slots.sync_uploads()
        wall = time.perf_counter() - t0
        st = self.slots.stats()
        return ChurnResult(len(trace.steps), wall, st, decisions, tokens)

    def close(self):
        self.slots.close()
