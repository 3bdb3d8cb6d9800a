"""Thin ctypes binding of the C ABI (include/rank_adapter_apply.h).

Functions keep the C names and only marshal arguments; every step of the path
runs in the compiled library. ``LoraSlots`` is a convenience owner of the
device memory the ABI asks the caller for (slot pools, scale/rank arrays,
workspace) and of the two streams, all allocated through PyTorch.

Loading raises ``RuntimeError`` when the library has not been built: there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# RANK_ADAPTER_APPLY_LIB selects another build of the same library (for
# example the sanitizer build of build.py); the default is the in-tree build.
LIB_PATH = os.environ.get("RANK_ADAPTER_APPLY_LIB") or os.path.join(HERE, "_build", "librank_adapter_apply.so")

LORA_OK = 0
LORA_ERR_ARG = -1
LORA_ERR_RANK = -2
LORA_ERR_NO_SLOT = -3
LORA_ERR_CUDA = -4
LORA_ERR_STATE = -5
LORA_DTYPE_F32 = 0
LORA_DTYPE_BF16 = 1
NO_ID = (1 << 64) - 1

EXPORTED = [
    "lora_workspace_bytes", "lora_slots_init", "lora_destroy", "lora_load_slot", "lora_apply",
    "lora_apply_multi", "lora_apply_multi_host", "lora_lookup", "lora_assign", "lora_acquire",
    "lora_release", "lora_evict_lru", "lora_tick", "lora_set_thrash_window",
    "lora_set_prefill_min_tokens", "lora_set_small_batch_tokens", "lora_set_inputs_ready", "lora_sync_uploads", "lora_stats", "lora_adapter_bytes",
    "lora_last_error", "lora_apply_static_scratch", "lora_pin", "lora_set_min_residency",
    "lora_set_policy", "lora_set_keep_score_weights", "lora_set_adapter_priority",
    "lora_set_slot_tracking", "lora_load_slots", "lora_assign_batch", "lora_release_batch",
    "lora_selftest_wait_timeout", "lora_assign_tokens", "lora_sync_host", "lora_abort_load",
    "lora_register_host_adapters", "lora_set_warm_set", "lora_serve_step",
]


class LoraLayerDesc(ctypes.Structure):
    _fields_ = [("d_in", ctypes.c_int), ("d_out", ctypes.c_int),
                ("A_pool", ctypes.c_void_p), ("B_pool", ctypes.c_void_p)]


class LoraStats(ctypes.Structure):
    _fields_ = [("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64),
                ("evictions", ctypes.c_uint64), ("reloads_after_eviction", ctypes.c_uint64),
                ("rejected", ctypes.c_uint64), ("uploads", ctypes.c_uint64),
                ("upload_bytes", ctypes.c_uint64), ("invalid_token_index", ctypes.c_uint64),
                ("upload_seconds", ctypes.c_double), ("epoch", ctypes.c_int64),
                ("device_wait_timeouts", ctypes.c_uint64), ("cluster_applies", ctypes.c_uint64),
                ("grouped_applies", ctypes.c_uint64), ("kernel_launches", ctypes.c_uint64),
                ("aborted_loads", ctypes.c_uint64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class LoraError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"[{code}] {msg}")
        self.code = code


_lib = None


def load(path: str = LIB_PATH):
    """Load the compiled library (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"rank_adapter_apply library not built: {path} is missing "
                           "(run `python -m rank_adapter_apply_gb300.build`)")
    lib = ctypes.CDLL(path)
    vp, i32, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "lora_workspace_bytes": (sz, [i32, i32, i32, i32]),
        "lora_slots_init": (i32, [P(vp), i32, i32, i32, i32, i32, i32, P(LoraLayerDesc), vp, vp,
                                  vp, sz, vp, vp]),
        "lora_destroy": (None, [vp]),
        "lora_load_slot": (i32, [vp, i32, P(vp), P(vp), i32, ctypes.c_float]),
        "lora_apply": (i32, [vp, i32, vp, vp, vp, i32]),
        "lora_apply_multi": (i32, [vp, i32, P(i32), P(vp), P(vp), vp, i32]),
        "lora_apply_multi_host": (i32, [vp, i32, P(i32), P(vp), P(vp), vp, i32, P(vp), P(vp), vp]),
        "lora_lookup": (i32, [vp, u64, P(i32)]),
        "lora_assign": (i32, [vp, u64, i32, P(i32), P(i32), P(u64)]),
        "lora_acquire": (i32, [vp, i32]),
        "lora_release": (i32, [vp, i32]),
        "lora_evict_lru": (i32, [vp, P(i32), P(u64)]),
        "lora_abort_load": (i32, [vp, i32, P(u64)]),
        "lora_tick": (i32, [vp]),
        "lora_set_thrash_window": (i32, [vp, i32]),
        "lora_pin": (i32, [vp, i32, i32]),
        "lora_set_slot_tracking": (i32, [vp, i32]),
        "lora_selftest_wait_timeout": (i32, [vp, P(i32)]),
        "lora_assign_batch": (i32, [vp, i32, P(u64), P(i32), i32, P(i32), P(i32), P(u64), P(i32)]),
        "lora_release_batch": (i32, [vp, i32, P(i32)]),
        "lora_assign_tokens": (i32, [vp, i32, P(u64), P(i32), i32, P(i32), i32, P(u64), P(i32), P(i32), P(u64),
                                     P(i32), P(i32)]),
        "lora_load_slots": (i32, [vp, i32, P(i32), P(vp), P(vp), P(i32), P(ctypes.c_float)]),
        "lora_set_min_residency": (i32, [vp, i32]),
        "lora_set_policy": (i32, [vp, i32]),
        "lora_set_keep_score_weights": (i32, [vp, P(ctypes.c_double)]),
        "lora_set_adapter_priority": (i32, [vp, u64, ctypes.c_double]),
        "lora_set_prefill_min_tokens": (i32, [vp, i32]),
        "lora_set_small_batch_tokens": (i32, [vp, i32]),
        "lora_set_inputs_ready": (i32, [vp, i32]),
        "lora_sync_uploads": (i32, [vp]),
        "lora_sync_host": (i32, [vp]),
        "lora_stats": (i32, [vp, P(LoraStats)]),
        "lora_adapter_bytes": (u64, [i32, P(i32), P(i32), i32, i32]),
        "lora_last_error": (ctypes.c_char_p, []),
        "lora_apply_static_scratch": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                            vp]),
        "lora_register_host_adapters": (i32, [vp, i32, P(u64), P(i32), P(ctypes.c_float), P(vp), P(vp)]),
        "lora_set_warm_set": (i32, [vp, i32, P(u64)]),
        "lora_serve_step": (i32, [vp, i32, P(u64), i32, P(i32), P(vp), P(vp), vp, i32, i32, P(u64), P(i32),
                                  P(i32), P(u64), P(i32), P(i32)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def last_error() -> str:
    return load().lora_last_error().decode()


def check(rc: int) -> int:
    if rc != LORA_OK:
        raise LoraError(rc, last_error())
    return rc


def _vp_array(ptrs):
    return (ctypes.c_void_p * len(ptrs))(*[ctypes.c_void_p(p) for p in ptrs])


def _i32_array(vals):
    return (ctypes.c_int * len(vals))(*vals)


# --- C-named wrappers (argument marshalling only) --------------------------------

def lora_workspace_bytes(max_loras, max_lora_rank, max_tokens, max_layers_per_call):
    return int(load().lora_workspace_bytes(max_loras, max_lora_rank, max_tokens, max_layers_per_call))


def lora_slots_init(max_loras, max_lora_rank, max_tokens, max_layers_per_call, dtype, layers,
                    scale_dev, rank_dev, workspace, workspace_bytes, compute_stream, upload_stream):
    """layers: list of (d_in, d_out, A_pool_ptr, B_pool_ptr). Returns the context handle."""
    descs = (LoraLayerDesc * max(1, len(layers)))(
        *[LoraLayerDesc(di, do, a, b) for di, do, a, b in layers])
    h = ctypes.c_void_p()
    check(load().lora_slots_init(ctypes.byref(h), max_loras, max_lora_rank, max_tokens,
                                 max_layers_per_call, dtype, len(layers), descs, scale_dev,
                                 rank_dev, workspace, workspace_bytes, compute_stream,
                                 upload_stream))
    return h


def lora_destroy(ctx):
    load().lora_destroy(ctx)


def lora_load_slot(ctx, slot, A_ptrs, B_ptrs, rank, alpha):
    return check(load().lora_load_slot(ctx, slot, _vp_array(A_ptrs), _vp_array(B_ptrs), rank,
                                       float(alpha)))


def lora_load_slots(ctx, slots, A_ptrs, B_ptrs, ranks, alphas):
    """A_ptrs / B_ptrs: n * n_layers host pointers, adapter-major."""
    n = len(slots)
    return check(load().lora_load_slots(ctx, n, _i32_array(list(slots)), _vp_array(A_ptrs),
                                        _vp_array(B_ptrs), _i32_array(list(ranks)),
                                        (ctypes.c_float * n)(*[float(a) for a in alphas])))


def lora_apply(ctx, layer, x_ptr, y_ptr, idx_ptr, n_tokens):
    return check(load().lora_apply(ctx, layer, x_ptr, y_ptr, idx_ptr, n_tokens))


def lora_apply_multi(ctx, layers, x_ptrs, y_ptrs, idx_ptr, n_tokens):
    return check(load().lora_apply_multi(ctx, len(layers), _i32_array(layers), _vp_array(x_ptrs),
                                         _vp_array(y_ptrs), idx_ptr, n_tokens))


def lora_apply_multi_host(ctx, layers, xs_host, ys_host, idx_host, n_tokens, xs_dev, ys_dev,
                          idx_dev):
    return check(load().lora_apply_multi_host(
        ctx, len(layers), _i32_array(layers), _vp_array(xs_host), _vp_array(ys_host), idx_host,
        n_tokens, _vp_array(xs_dev), _vp_array(ys_dev), idx_dev))


def lora_lookup(ctx, adapter_id):
    s = ctypes.c_int()
    check(load().lora_lookup(ctx, adapter_id, ctypes.byref(s)))
    return s.value


def lora_assign(ctx, adapter_id, rank):
    """Returns (status, slot, needs_load, evicted_id or -1); status is not raised."""
    s, nl, ev = ctypes.c_int(-1), ctypes.c_int(0), ctypes.c_uint64(NO_ID)
    rc = load().lora_assign(ctx, adapter_id, rank, ctypes.byref(s), ctypes.byref(nl),
                            ctypes.byref(ev))
    return rc, s.value, nl.value, (-1 if ev.value == NO_ID else ev.value)


def lora_assign_batch(ctx, ids, ranks, acquire=True):
    """Returns (status, n_done, slots, needs_load, evicted ids (-1: none)) as numpy arrays."""
    import numpy as np
    n = len(ids)
    ida = np.ascontiguousarray(np.asarray(ids, dtype=np.uint64))
    rka = np.ascontiguousarray(np.asarray(ranks, dtype=np.int32))
    slots = np.full(n, -1, np.int32)
    need = np.zeros(n, np.int32)
    ev = np.zeros(n, np.uint64)
    done = ctypes.c_int(0)
    P = ctypes.POINTER
    rc = load().lora_assign_batch(ctx, n, ida.ctypes.data_as(P(ctypes.c_uint64)),
                                  rka.ctypes.data_as(P(ctypes.c_int)), 1 if acquire else 0,
                                  slots.ctypes.data_as(P(ctypes.c_int)), need.ctypes.data_as(P(ctypes.c_int)),
                                  ev.ctypes.data_as(P(ctypes.c_uint64)), ctypes.byref(done))
    evi = np.where(ev == np.uint64(NO_ID), -1, ev.astype(np.int64))
    return rc, done.value, slots, need, evi


def lora_assign_tokens(ctx, adapter_ids, ranks, acquire=True, max_distinct=None):
    """Per-token admission. adapter_ids: int64 per token (-1 = base model only),
    ranks: per token. Returns (status, token_slot_idx int32[T], distinct ids,
    slots, needs_load, evicted ids (-1: none), n_done) as numpy arrays."""
    import numpy as np
    ids = np.asarray(adapter_ids, dtype=np.int64)
    T = ids.shape[0]
    ida = np.ascontiguousarray(np.where(ids < 0, np.uint64(NO_ID), ids.astype(np.uint64)))
    rka = np.ascontiguousarray(np.asarray(ranks, dtype=np.int32))
    m = T if max_distinct is None else int(max_distinct)
    tsi = np.full(T, -1, np.int32)
    dids = np.zeros(max(m, 1), np.uint64)
    slots = np.full(max(m, 1), -1, np.int32)
    need = np.zeros(max(m, 1), np.int32)
    ev = np.zeros(max(m, 1), np.uint64)
    nd, done = ctypes.c_int(0), ctypes.c_int(0)
    P = ctypes.POINTER
    rc = load().lora_assign_tokens(ctx, T, ida.ctypes.data_as(P(ctypes.c_uint64)), rka.ctypes.data_as(P(ctypes.c_int)),
                                   1 if acquire else 0, tsi.ctypes.data_as(P(ctypes.c_int)), m,
                                   dids.ctypes.data_as(P(ctypes.c_uint64)), slots.ctypes.data_as(P(ctypes.c_int)),
                                   need.ctypes.data_as(P(ctypes.c_int)), ev.ctypes.data_as(P(ctypes.c_uint64)),
                                   ctypes.byref(nd), ctypes.byref(done))
    k = nd.value
    evi = np.where(ev[:k] == np.uint64(NO_ID), -1, ev[:k].astype(np.int64))
    return rc, tsi, dids[:k].astype(np.int64), slots[:k], need[:k], evi, done.value


def lora_release_batch(ctx, slots):
    import numpy as np
    sa = np.ascontiguousarray(np.asarray(slots, dtype=np.int32))
    return load().lora_release_batch(ctx, len(sa), sa.ctypes.data_as(ctypes.POINTER(ctypes.c_int)))


def lora_acquire(ctx, slot):
    return load().lora_acquire(ctx, slot)


def lora_release(ctx, slot):
    return load().lora_release(ctx, slot)


def lora_evict_lru(ctx):
    """Returns (status, slot or -1, evicted id or -1)."""
    s, ev = ctypes.c_int(-1), ctypes.c_uint64(NO_ID)
    rc = load().lora_evict_lru(ctx, ctypes.byref(s), ctypes.byref(ev))
    return rc, s.value, (-1 if ev.value == NO_ID else ev.value)


def lora_abort_load(ctx, slot):
    """Returns (status, id that was bound or -1)."""
    ev = ctypes.c_uint64(NO_ID)
    rc = load().lora_abort_load(ctx, int(slot), ctypes.byref(ev))
    return rc, (-1 if ev.value == NO_ID else ev.value)


def lora_tick(ctx):
    return check(load().lora_tick(ctx))


def lora_set_thrash_window(ctx, epochs):
    return check(load().lora_set_thrash_window(ctx, epochs))


LORA_POLICY_LRU, LORA_POLICY_KEEP_SCORE = 0, 1


def lora_selftest_wait_timeout(ctx):
    """Returns 1 when the bounded wait gave up and set the device error word."""
    g = ctypes.c_int(0)
    check(load().lora_selftest_wait_timeout(ctx, ctypes.byref(g)))
    return g.value


def lora_set_slot_tracking(ctx, on=True):
    return check(load().lora_set_slot_tracking(ctx, 1 if on else 0))


def lora_pin(ctx, slot, pinned=True):
    """Returns the status (LORA_ERR_STATE for an empty slot)."""
    return load().lora_pin(ctx, slot, 1 if pinned else 0)


def lora_set_min_residency(ctx, epochs):
    return check(load().lora_set_min_residency(ctx, epochs))


def lora_set_policy(ctx, policy):
    return check(load().lora_set_policy(ctx, policy))


def lora_set_keep_score_weights(ctx, w):
    arr = (ctypes.c_double * 5)(*[float(v) for v in w])
    return check(load().lora_set_keep_score_weights(ctx, arr))


def lora_set_adapter_priority(ctx, adapter_id, priority):
    return check(load().lora_set_adapter_priority(ctx, int(adapter_id), float(priority)))


def lora_set_prefill_min_tokens(ctx, n):
    return check(load().lora_set_prefill_min_tokens(ctx, n))


def lora_set_small_batch_tokens(ctx, n):
    return check(load().lora_set_small_batch_tokens(ctx, n))


def lora_set_inputs_ready(ctx, on):
    return check(load().lora_set_inputs_ready(ctx, 1 if on else 0))


def lora_sync_host(ctx):
    return check(load().lora_sync_host(ctx))


def lora_sync_uploads(ctx):
    return check(load().lora_sync_uploads(ctx))


def lora_stats(ctx) -> dict:
    st = LoraStats()
    check(load().lora_stats(ctx, ctypes.byref(st)))
    return st.as_dict()


def lora_adapter_bytes(layers, rank, bytes_per_param):
    di = _i32_array([a for a, _ in layers])
    do = _i32_array([b for _, b in layers])
    return int(load().lora_adapter_bytes(len(layers), di, do, rank, bytes_per_param))


def lora_apply_static_scratch(x_ptr, y_ptr, idx_ptr, n_tokens, d_in, d_out, max_loras,
                              max_lora_rank, dtype, A_pool, B_pool, scale_dev, rank_dev, stream):
    """One layer without a context or workspace (scratch in the library's static array)."""
    return check(load().lora_apply_static_scratch(x_ptr, y_ptr, idx_ptr, n_tokens, d_in, d_out,
                                                  max_loras, max_lora_rank, dtype, A_pool, B_pool,
                                                  scale_dev, rank_dev, stream))


def lora_register_host_adapters(ctx, ids, ranks, alphas, A_ptrs=None, B_ptrs=None):
    """ids / ranks / alphas per adapter; A_ptrs / B_ptrs: n * n_layers host
    pointers, adapter-major (None on a host-only context)."""
    n = len(ids)
    A = _vp_array(A_ptrs) if A_ptrs is not None else None
    Bp = _vp_array(B_ptrs) if B_ptrs is not None else None
    return check(load().lora_register_host_adapters(
        ctx, n, (ctypes.c_uint64 * n)(*[int(i) for i in ids]), _i32_array(list(ranks)),
        (ctypes.c_float * n)(*[float(a) for a in alphas]), A, Bp))


def lora_set_warm_set(ctx, ids):
    n = len(ids)
    return check(load().lora_set_warm_set(ctx, n, (ctypes.c_uint64 * n)(*[int(i) for i in ids])))


def lora_serve_step(ctx, adapter_ids, layers=(), x_ptrs=(), y_ptrs=(), idx_bufs=0, max_groups=0):
    """One serving step (lora_serve_step). adapter_ids: one adapter id per token
    (NO_ID for base-model tokens); layers / x_ptrs / y_ptrs: the layer indices
    and device pointers of the call; idx_bufs: address of max_groups x
    n_tokens int32 that the host writes and the GPU reads (pinned memory).
    Returns (decisions, n_groups), decisions = per distinct adapter in order
    (id, slot, uploaded, evicted id or -1)."""
    import numpy as np
    ids = np.ascontiguousarray(adapter_ids, dtype=np.uint64)
    T = int(ids.shape[0])
    n = len(layers)
    md = max(1, T)
    o_ids = (ctypes.c_uint64 * md)()
    o_sl = (ctypes.c_int * md)()
    o_nd = (ctypes.c_int * md)()
    o_ev = (ctypes.c_uint64 * md)()
    nd, ng = ctypes.c_int(0), ctypes.c_int(0)
    check(load().lora_serve_step(
        ctx, T, ids.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), n,
        _i32_array(list(layers)) if n else None, _vp_array(x_ptrs) if n else None,
        _vp_array(y_ptrs) if n else None, idx_bufs or None, int(max_groups), md, o_ids, o_sl, o_nd, o_ev,
        ctypes.byref(nd), ctypes.byref(ng)))
    dec = [(int(o_ids[i]), int(o_sl[i]), int(o_nd[i]), -1 if o_ev[i] == NO_ID else int(o_ev[i]))
           for i in range(nd.value)]
    return dec, ng.value
