#!/usr/bin/env python
"""Benchmark of the multi-LoRA delta path on one GB300 (or N replicas).

Workload: the decode batch of Llama-7B-shaped q_proj and v_proj (4096 -> 4096,
bf16), max_loras = 8 slots of rank 16 (alpha 32), 256 tokens per batch with
Zipf(1.1) slot ids and 10% base-only tokens.

One step = one batch through the whole path: slot lookup (every adapter is
resident after warm-up, so no upload is queued), token grouping, shrink and
expand-add for both layers.

* value: delta tokens per second per layer set with inputs resident in HBM,
  from CUDA-graph replays on CUDA events. Every step uses its own x, y, slot
  ids and its own copy of the slot pools, cycling over enough sets to exceed
  twice the L2 size, so no step finds its operands in L2.
* e2e: the same metric through lora_apply_multi_host with pinned HOST buffers:
  H2D of x, y and slot ids, apply, D2H of y, plus host slot admission
  (assign/acquire/release), wall clock.
* cpu_baseline / --impl reference: the fp64 CPU oracle on host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from rank_adapter_apply_gb300 import workloads as wl  # noqa: E402

METRIC = "LoRA-delta tokens/s per layer set; achieved HBM GB/s and % roofline (1xGB300)"
UNIT = "delta-tokens/s"
WORKLOAD = "decode_qv_4096"
T_TOKENS, N_SLOTS, RANK, ALPHA, D = 256, 8, 16, 32.0, 4096
E2E_HOST_SETS, E2E_STAGING_SETS = 32, 3     # e2e: pinned host sets (a sync per cycle), device staging sets


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_traffic(kernel_file: str):
    """DRAM bytes per launch of the decode kernel from the committed ncu summary,
    if that summary was taken on the current kernel source (else None)."""
    import hashlib
    src = os.path.join(ROOT, "rank_adapter_apply_gb300", "csrc", kernel_file)
    summ = os.path.join(ROOT, "profiles", "decode_cluster_qv4096_traffic.json")
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        rec = json.load(open(summ))
        if rec.get("kernel_source_sha256") == sha:
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def algorithmic_bytes(idx: np.ndarray, ranks, layers, e=2) -> int:
    """Per layer set: the x rows of adapter tokens read once per distinct input
    (q/k/v, or gate/up, read the same activations), y rows read and written per
    layer, each used slot's true-rank A and B read once per layer, the slot ids
    read once."""
    T = idx.shape[0]
    act = idx[idx >= 0]
    used = np.unique(act)
    total = T * 4
    seen = set()
    for ly in layers:
        if ly.x_key not in seen:
            seen.add(ly.x_key)
            total += act.size * ly.d_in * e
        total += act.size * 2 * ly.d_out * e
        total += sum((ly.d_in + ly.d_out) * int(ranks[s]) * e for s in used)
    return total


def algorithmic_flops(idx, ranks, layers) -> int:
    act = idx[idx >= 0]
    return sum(2 * int(ranks[s]) * (ly.d_in + ly.d_out) for ly in layers for s in act)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        rows = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.file.flush()
            self.file.seek(0)
            for line in self.file:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        try:
            os.unlink(self.file.name)
        except Exception:
            pass
        return rows

    @staticmethod
    def summary(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def reduce_over_ranks(ms: float, tokens: int, device=None):
    """Job-wide figures of a weak-scaled run (one replica per rank, no data
    exchange between ranks): the slowest rank's time and every rank's tokens.
    Returns (ms, tokens) unchanged when no process group is running."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms, tokens
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(round(n.item()))


def make_batches(n_sets: int, seed0: int = 0):
    """Set 0 is the decode workload itself; sets 1.. draw new x, base outputs
    and slot ids with the same recipe (base output drawn directly)."""
    w = wl.decode_qv_4096(seed0)
    batches = [(w.xs["x"], w.ys, w.token_slot_idx)]
    for i in range(1, n_sets):
        rng = np.random.default_rng(seed0 + 7919 * i)
        batches.append(wl.decode_batch(rng, T_TOKENS, N_SLOTS, True))
    return w, batches


def cpu_oracle_run(w, batches, budget_s: float = 10.0, max_batches=None, threads=None):
    """Time the fp64 oracle over whole batches (both layers) until the budget
    is spent, on `threads` host threads (default: all cores). Returns
    (delta tokens/s, batches done, threads used, seconds)."""
    import oracle
    all_cores = oracle.threads()
    if threads is not None:
        oracle.set_threads(threads)
    try:
        return _time_oracle(oracle, w, batches, budget_s, max_batches)
    finally:
        oracle.set_threads(all_cores)


def _time_oracle(oracle, w, batches, budget_s, max_batches):
    pools = {ly.name: w.padded_pools(ly.name) for ly in w.layers}
    oracle.lora_apply_ref(batches[0][0][:1], batches[0][1]["q_proj"][:1], *pools["q_proj"],
                          w.ranks, w.alphas, batches[0][2][:1])        # build + load outside timing
    tokens, done = 0, 0
    t0 = time.perf_counter()
    while True:
        x, ys, idx = batches[done % len(batches)]
        for ly in w.layers:
            oracle.lora_apply_ref(x, ys[ly.name], *pools[ly.name], w.ranks, w.alphas, idx)
        tokens += int((idx >= 0).sum())
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_batches and done >= max_batches):
            break
    return tokens / el, done, oracle.threads(), el


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w, batches = make_batches(4)
    import oracle
    pools = {ly.name: w.padded_pools(ly.name) for ly in w.layers}
    n_tok = [T_TOKENS]

    # each step: the oracle over a bounded sample of one batch (the first n_tok
    # tokens, both layers), sized so that the K timed steps take about a minute
    def step(i):
        x, ys, idx = batches[i % len(batches)]
        tok = np.arange(n_tok[0])
        for ly in w.layers:
            oracle.lora_apply_ref(x, ys[ly.name], *pools[ly.name], w.ranks, w.alphas, idx, tokens=tok)
        return int((idx[tok] >= 0).sum())
    n_tok[0] = 16
    t0 = time.perf_counter()
    step(0)
    per_tok = (time.perf_counter() - t0) / 16
    n_tok[0] = int(max(1, min(T_TOKENS, 60.0 / max(1, args.steps) / max(per_tok, 1e-9))))
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    toks = sum(step(i) for i in range(args.steps))
    el = time.perf_counter() - t0
    v = toks / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens_per_batch": T_TOKENS, "layers": ["q_proj", "v_proj"],
                       "d": D, "max_loras": N_SLOTS, "rank": RANK, "alpha": ALPHA},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                             "sample": f"first {n_tok[0]} tokens of a 256-token batch, q_proj and v_proj, per step"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300 import build as build_mod
    from rank_adapter_apply_gb300.harness import to_torch
    from rank_adapter_apply_gb300.slots import LoraSlots

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(B.LIB_PATH):
        build_mod.build()
    if world > 1:
        dist.barrier()
    B.load()

    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 129 * 2 ** 20) or 129 * 2 ** 20
    per_set = T_TOKENS * D * 2 * 3 + 2 * N_SLOTS * RANK * D * 2 * 2 + T_TOKENS * 4
    n_sets = int(max(8, -(-2.5 * l2 // per_set)))
    w, batches = make_batches(n_sets)
    layers = [(ly.d_in, ly.d_out) for ly in w.layers]
    stream = torch.cuda.Stream(device=dev)
    upload = torch.cuda.Stream(device=dev)
    host_ad = []
    for s in range(N_SLOTS):
        A = [to_torch(w.adapters[s][ly.name][0], w.dtype).pin_memory() for ly in w.layers]
        Bm = [to_torch(w.adapters[s][ly.name][1], w.dtype).pin_memory() for ly in w.layers]
        host_ad.append((A, Bm))

    class DevSet:
        pass

    sets = []
    for i, (x, ys, idx) in enumerate(batches):
        d = DevSet()
        d.slots = LoraSlots(layers, N_SLOTS, RANK, T_TOKENS, dtype=torch.bfloat16, device=dev,
                            compute_stream=stream, upload_stream=upload)
        # every step's x, slot ids and pools are its own: the kernel before never writes them
        B.lora_set_inputs_ready(d.slots.ctx, not args.no_early)
        for s in range(N_SLOTS):
            # admission: adapter id s -> slot (all misses on first sight), then upload
            rc, slot, need, _ = d.slots.assign(s, RANK)
            assert rc == 0 and need == 1
            d.slots.load_slot(slot, host_ad[s][0], host_ad[s][1], RANK, ALPHA)
        d.x = to_torch(x, w.dtype).to(dev)
        d.ys = [to_torch(ys[ly.name], w.dtype).to(dev) for ly in w.layers]
        d.idx = torch.from_numpy(idx).to(dev)
        d.t_act = int((idx >= 0).sum())
        d.bytes = algorithmic_bytes(idx, w.ranks, w.layers)
        d.flops = algorithmic_flops(idx, w.ranks, w.layers)
        sets.append(d)
    torch.cuda.synchronize(dev)
    for d in sets:
        d.slots.sync_uploads()

    def step_apply(d):
        d.slots.apply_multi([0, 1], [d.x, d.x], d.ys, d.idx)

    # eager warm-up (clears pending-upload waits; sets kernel attributes)
    with torch.cuda.stream(stream):
        for d in sets:
            step_apply(d)
    torch.cuda.synchronize(dev)

    # graphs: one over all sets, and one per set for the remainder of K
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all, stream=stream):
        for d in sets:
            step_apply(d)
    g_one, per_step = [], set()
    for d in sets:
        k0 = d.slots.stats()["kernel_launches"]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step_apply(d)
        g_one.append(g)
        per_step.add(d.slots.stats()["kernel_launches"] - k0)   # kernels in one step, counted by the library
    torch.cuda.synchronize(dev)
    if len(per_step) != 1:
        raise RuntimeError(f"steps of different sets queue different kernel counts: {sorted(per_step)}")
    launches_per_step = per_step.pop()

    def run_steps(k):
        full, rem = divmod(k, len(sets))
        with torch.cuda.stream(stream):
            for _ in range(full):
                g_all.replay()
            for i in range(rem):
                g_one[i].replay()
        return full, rem

    run_steps(max(3, args.warmup))
    torch.cuda.synchronize(dev)
    # keep the GPU busy ~1 s before timing so the clocks settle (untimed)
    t_probe = time.perf_counter()
    while not args.quick and time.perf_counter() - t_probe < 1.0:
        run_steps(len(sets) * 20)
        torch.cuda.synchronize(dev)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.12)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    full, rem = run_steps(args.steps)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    clock_rows = sampler.stop()

    order = [i % len(sets) for i in range(full * len(sets))] + list(range(rem))
    tokens = sum(sets[i].t_act for i in order)
    bytes_ = sum(sets[i].bytes for i in order)
    flops = sum(sets[i].flops for i in order)
    ms, job_tokens = reduce_over_ranks(ms, tokens, dev)
    value = job_tokens / (ms * 1e-3)
    hbm, peak_kind = peaks()
    achieved = bytes_ / (ms * 1e-3) / 1e9

    # --- context: a plain copy of the same bytes per graph-replayed launch ---
    floor = None if args.quick else copy_floor(bytes_ / max(1, args.steps), stream, dev, l2)

    # --- end to end through the C ABI with host buffers --------------------
    e2e = None if args.quick else run_e2e(args, w, batches, sets[0], stream, dev, world)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded numpy: x~N(0,1), A~U(+-1/64), B~N(0,0.02), Zipf(1.1) slots, 10% base-only)",
        "config": {"workload": WORKLOAD, "tokens_per_batch": T_TOKENS, "layers": ["q_proj", "v_proj"],
                   "d": D, "max_loras": N_SLOTS, "rank": RANK, "alpha": ALPHA,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {len(sets)} distinct x/y/idx/pool sets, "
                         f"{len(sets) * per_set / 2**20:.0f} MiB per cycle vs L2 {l2 / 2**20:.0f} MiB",
                   "timing": "CUDA-graph replay, CUDA events on the launch stream",
                   "inputs_ready": not args.no_early},
        "roofline": {"bound": "hbm",
                     "kernel": "decode_cluster_kernel (one launch per step: grouping, shrink and "
                               "expand of q_proj and v_proj)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_kind": peak_kind, "traffic": kernel_traffic("decode_cluster.cu"),
                     "copy_floor": floor,
                     "algorithmic_bytes_per_step": bytes_ / max(1, args.steps),
                     "tflops": flops / (ms * 1e-3) / 1e12},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": ClockSampler.summary(clock_rows),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quick:
        v, n, cores, el = cpu_oracle_run(w, batches, budget_s=args.cpu_seconds)
        # the same oracle on one thread, over a shorter sample
        v1, n1, _, el1 = cpu_oracle_run(w, batches, budget_s=max(1.0, args.cpu_seconds / 3),
                                        threads=1)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{n} whole batches (256 tokens, q_proj+v_proj) in {el:.1f} s",
                                "single_thread": {"value": v1, "cores": 1,
                                                  "sample": f"{n1} whole batches in {el1:.1f} s"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    for d in sets:
        d.slots.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def copy_floor(step_bytes, stream, dev, l2):
    """GB/s of a plain device-to-device copy that moves as many bytes per
    launch as one step (half read, half written), graph-replayed over buffers
    larger than L2 in total: what a single launch of this size reaches on this
    GPU, for comparison with the step's achieved GB/s."""
    import torch
    # bf16 elements per buffer (bytes/2 each), rounded up to whole 64 KiB: the
    # driver's copy runs a slower path on sizes that are not (6.82 MB copies
    # measured 6.05 us against 4.1 us for 6.5 MiB).
    n = max(1, -(-int(step_bytes // 4) // 32768) * 32768)
    sets = int(max(8, -(-2.5 * l2 // (2 * n * 2))))
    bufs = [(torch.empty(n, dtype=torch.bfloat16, device=dev), torch.empty(n, dtype=torch.bfloat16, device=dev))
            for _ in range(sets)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for a, b in bufs:
            b.copy_(a)
    with torch.cuda.stream(stream):
        for _ in range(5):
            g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 50
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    e1.record(stream)
    stream.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * sets)
    del bufs
    return {"GBps": 4.0 * n / us / 1e3, "us_per_launch": us, "bytes_per_launch": 4 * n,
            "note": "torch device-to-device copy of the step's byte count per launch, CUDA-graph replayed"}


def run_e2e(args, w, batches, d0, stream, dev, world):
    """Whole-job throughput through lora_apply_multi_host with pinned host
    buffers: per step admission of every token's adapter (lora_assign_tokens:
    lookup hit, acquire, slot id per token), H2D of slot ids / x / y (one packed
    copy), apply, D2H of both y (one packed copy), release."""
    import torch
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300.harness import to_torch

    ctx = d0.slots.ctx
    nh = min(E2E_HOST_SETS, len(batches))      # host buffer sets, reused after a sync
    nd_sets = args.e2e_staging_sets
    lib = B.load()
    import ctypes
    # One pinned block per host set and one device block per staging set, each
    # laid out idx | x | y_q | y_v, so the library copies each way in one piece.
    off_x = T_TOKENS * 4
    off_y = [off_x + T_TOKENS * D * 2 * (1 + li) for li in range(len(w.layers))]
    blk = off_y[-1] + T_TOKENS * D * 2

    def views(buf):
        idx = buf[:off_x].view(torch.int32)
        x = buf[off_x:off_x + T_TOKENS * D * 2].view(torch.bfloat16).view(T_TOKENS, D)
        ys = [buf[o:o + T_TOKENS * D * 2].view(torch.bfloat16).view(T_TOKENS, D) for o in off_y]
        return idx, x, ys

    hblk = [torch.empty(blk, dtype=torch.uint8).pin_memory() for _ in range(nh)]
    hv = [views(hb) for hb in hblk]
    for i in range(nh):
        hv[i][1].copy_(to_torch(batches[i][0], w.dtype))
        for li, ly in enumerate(w.layers):
            hv[i][2][li].copy_(to_torch(batches[i][1][ly.name], w.dtype))
    # device staging sets, rotated: one call's copies in overlap the
    # previous call's apply and copies back
    dblk = [torch.empty(blk, dtype=torch.uint8, device=dev) for _ in range(nd_sets)]
    dv = [views(db) for db in dblk]
    lay = (ctypes.c_int * 2)(0, 1)
    xs_dev = [B._vp_array([dv[k][1].data_ptr()] * 2) for k in range(nd_sets)]
    ys_dev = [B._vp_array([t.data_ptr() for t in dv[k][2]]) for k in range(nd_sets)]
    host_x = [B._vp_array([hv[i][1].data_ptr()] * 2) for i in range(nh)]
    host_y = [B._vp_array([t.data_ptr() for t in hv[i][2]]) for i in range(nh)]
    idx_h = [ctypes.cast(hv[i][0].data_ptr(), ctypes.POINTER(ctypes.c_int)) for i in range(nh)]
    idx_hp = [hv[i][0].data_ptr() for i in range(nh)]
    idx_dp = [dv[k][0].data_ptr() for k in range(nd_sets)]
    # the adapter of every token (base-only: the no-adapter id) and its rank
    ids_np = [np.ascontiguousarray(np.where(batches[i][2] >= 0, batches[i][2], -1).astype(np.int64)
                                   .astype(np.uint64)) for i in range(nh)]
    ids_p = [a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)) for a in ids_np]
    ranks_np = np.full(T_TOKENS, RANK, np.int32)
    ranks_p = ranks_np.ctypes.data_as(ctypes.POINTER(ctypes.c_int))
    dids = np.zeros(N_SLOTS, np.uint64)
    slots = np.zeros(N_SLOTS, np.int32)
    need = np.zeros(N_SLOTS, np.int32)
    evi = np.zeros(N_SLOTS, np.uint64)
    P = ctypes.POINTER
    dids_p, slots_p = dids.ctypes.data_as(P(ctypes.c_uint64)), slots.ctypes.data_as(P(ctypes.c_int))
    need_p, evi_p = need.ctypes.data_as(P(ctypes.c_int)), evi.ctypes.data_as(P(ctypes.c_uint64))
    nd, ndone = ctypes.c_int(0), ctypes.c_int(0)
    nd_r, ndone_r = ctypes.byref(nd), ctypes.byref(ndone)
    act = [int((batches[i][2] >= 0).sum()) for i in range(nh)]

    def step(i):
        j = i % nh
        # admission of the batch's adapters and the slot id of every token, in
        # one call (all hits here), written straight into the pinned idx block
        rc = lib.lora_assign_tokens(ctx, T_TOKENS, ids_p[j], ranks_p, 1, idx_h[j], N_SLOTS, dids_p, slots_p,
                                    need_p, evi_p, nd_r, ndone_r)
        if rc != 0 or need[:nd.value].any():
            raise RuntimeError("adapter unexpectedly not resident")
        b = i % nd_sets
        B.check(lib.lora_apply_multi_host(ctx, 2, lay, host_x[j], host_y[j], idx_hp[j], T_TOKENS,
                                          xs_dev[b], ys_dev[b], idx_dp[b]))
        B.check(lib.lora_release_batch(ctx, nd.value, slots_p))
        return act[j]

    for i in range(max(3, args.warmup)):
        step(i)
    B.check(lib.lora_sync_host(ctx))
    k = min(args.steps, 20000)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    toks = 0
    for i in range(k):
        if i % nh == 0 and i > 0:
            B.check(lib.lora_sync_host(ctx))   # host buffers of a set are reused every nh steps
        toks += step(i)
    B.check(lib.lora_sync_host(ctx))
    el = time.perf_counter() - t0
    el_ms, job_toks = reduce_over_ranks(el * 1e3, toks, dev)
    el = el_ms * 1e-3
    h2d = T_TOKENS * D * 2 + 2 * T_TOKENS * D * 2 + T_TOKENS * 4
    d2h = 2 * T_TOKENS * D * 2
    floor = link_floor(hblk, dblk, blk - off_y[0], off_y[0], dev)
    return {"value": job_toks / el, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": k, "us_per_step": el / k * 1e6,
            "link_floor": floor, "host_sets": nh, "staging_sets": nd_sets,
            "timing": "wall clock, host admission + H2D + apply + D2H per step"}


def link_floor(hblk, dblk, out_bytes, out_off, dev, reps=200):
    """Time per step of the host link alone: each step's whole block copied in
    on one stream while the previous step's y bytes are copied back on another,
    rotating the same pinned host sets and device staging sets as the e2e loop
    (no kernels, no admission)."""
    import torch
    si, so = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    nh, nd = len(hblk), len(dblk)
    ev = [torch.cuda.Event() for _ in range(nd)]

    def run(n):
        for i in range(n):
            b = i % nd
            with torch.cuda.stream(si):
                si.wait_event(ev[b])
                dblk[b].copy_(hblk[i % nh], non_blocking=True)
            so.wait_stream(si)
            with torch.cuda.stream(so):
                hblk[i % nh][out_off:out_off + out_bytes].copy_(dblk[b][out_off:out_off + out_bytes],
                                                                non_blocking=True)
                ev[b].record(so)
    for e in ev:
        e.record(so)
    run(10)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    run(reps)
    torch.cuda.synchronize(dev)
    us = (time.perf_counter() - t0) / reps * 1e6
    return {"us_per_step": us, "note": "the step's bytes copied in and out concurrently on two streams, "
                                       "same buffer rotation, no kernels"}


def run_big(args, name):
    """Prefill-style workloads (one large batch per step, every layer of the set)."""
    import torch
    from rank_adapter_apply_gb300 import build as build_mod
    from rank_adapter_apply_gb300.harness import DeviceWorkload
    build_mod.build()
    w = (wl.prefill_5120(0, n_seqs=args.prefill_seqs) if name == "prefill_5120"
         else wl.BY_NAME[name](0))
    dw = DeviceWorkload(w, max_tokens=w.n_tokens)
    lys = list(range(len(w.layers)))
    xs = [dw.xs[ly.x_key] for ly in w.layers]
    ys = [dw.ys[ly.name] for ly in w.layers]
    st = dw.slots.compute
    with torch.cuda.stream(st):
        for _ in range(max(3, args.warmup)):
            dw.slots.apply_multi(lys, xs, ys, dw.idx)
    st.synchronize()
    k0 = dw.slots.stats()["kernel_launches"]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        dw.slots.apply_multi(lys, xs, ys, dw.idx)
    per_step = dw.slots.stats()["kernel_launches"] - k0      # kernels in one replay of the step
    with torch.cuda.stream(st):
        for _ in range(3):
            g.replay()
    st.synchronize()
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.12)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    with torch.cuda.stream(st):
        for _ in range(args.steps):
            g.replay()
    e1.record(st)
    st.synchronize()
    ms = e0.elapsed_time(e1)
    clocks = ClockSampler.summary(sampler.stop())
    act = int((w.token_slot_idx >= 0).sum())
    bytes_ = algorithmic_bytes(w.token_slot_idx, w.ranks, w.layers)
    flops = algorithmic_flops(w.token_slot_idx, w.ranks, w.layers)
    hbm, kind = peaks()
    ach = bytes_ * args.steps / (ms * 1e-3) / 1e9
    line = {"metric": METRIC, "value": act * args.steps / (ms * 1e-3), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded numpy, shapes and slot structure of the workload)",
            "config": {"workload": name, "tokens": w.n_tokens, "layers": [l.name for l in w.layers],
                       "max_loras": w.max_loras, "max_lora_rank": w.max_lora_rank,
                       "l2": f"inputs larger than L2 ({bytes_ / 2**20:.0f} MiB per step)",
                       "timing": "CUDA-graph replay, CUDA events on the launch stream"},
            "roofline": {"bound": "hbm", "kernel": "whole step: group_tokens, prefill_shrink, [prefill_reduce], prefill_expand, decode shrink + expand (every layer)",
                         "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "peak_kind": kind,
                         "traffic": None, "algorithmic_bytes_per_step": bytes_,
                         "tflops": flops * args.steps / (ms * 1e-3) / 1e12},
            # grouping, prefill shrink, [chunk sums at rank 64], prefill expand, decode shrink + expand,
            # as counted by the library while the step was captured
            "gpu_launches": per_step * args.steps, "clocks": clocks}
    print(json.dumps(line), flush=True)
    dw.close()
    return 0


def run_churn(args):
    """Slot churn: 64 GPU slots, 512 rank-16 adapters in pinned host memory,
    Zipf(1.2) adapter ids with a burst of 20 cold adapters every 50 steps."""
    from rank_adapter_apply_gb300 import build as build_mod
    from rank_adapter_apply_gb300.churn import KEEP_PIN32, ChurnRunner
    build_mod.build()
    steps = args.steps if args.steps <= 1000 else 200
    trace = wl.churn_trace(0, n_steps=steps)
    warm = wl.churn_trace(99, n_steps=max(3, min(args.warmup, 20)))
    pol = {"lru": {}, "pin16": {"pin_top": 16},
           "keep": {"policy": 1, "weights": (1.0, 1.0, 0.0, 0.0, 0.0)},
           "keep_pin32": dict(KEEP_PIN32)}[args.churn_policy]
    r = ChurnRunner(overlap=args.churn_overlap, batched_upload=args.churn_upload == "batched", **pol)
    r.run(warm)
    base = r.slots.stats()
    res = r.run(trace)
    st = res.stats
    d = {k: st[k] - base[k] for k in ("hits", "misses", "evictions", "reloads_after_eviction",
                                      "uploads", "upload_bytes")}
    up_s = st["upload_seconds"] - base["upload_seconds"]
    line = {"metric": "slot-churn decode steps/s (LRU lookup, H2D uploads, q_proj+v_proj delta)",
            "value": res.steps / res.wall_s, "unit": "steps/s", "n_gpus": 1, "steps": res.steps,
            "warmup": len(warm.steps), "ms_per_step": res.wall_s * 1e3 / res.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded Zipf(1.2) adapter ids over 512 with cold bursts)",
            "config": {"workload": "churn_4096", "max_loras": 64, "host_adapters": 512, "rank": 16,
                       "eviction_policy": args.churn_policy, "upload_overlap": args.churn_overlap,
                       "upload": args.churn_upload,
                       "tokens_per_step": 256, "timing": "wall clock, host bookkeeping included"},
            "churn": {**d, "thrash_ratio": (d["reloads_after_eviction"] / d["evictions"]) if d["evictions"] else 0.0,
                      "hit_rate": d["hits"] / max(1, d["hits"] + d["misses"]),
                      "h2d_GBps": d["upload_bytes"] / up_s / 1e9 if up_s > 0 else None,
                      "delta_tokens_per_s": res.tokens / res.wall_s},
            "gpu_launches": st["kernel_launches"] - base["kernel_launches"]}
    print(json.dumps(line), flush=True)
    r.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=[WORKLOAD, "prefill_5120", "mixed_ranks_8b", "churn_4096"])
    ap.add_argument("--no-early", action="store_true",
                    help="decode: do not declare inputs independent of the preceding kernel")
    ap.add_argument("--prefill-seqs", type=int, default=32,
                    help="sequences in the prefill workload (32 = the full workload)")
    ap.add_argument("--churn-policy", choices=["lru", "pin16", "keep", "keep_pin32"], default="lru",
                    help="churn: pure LRU, LRU with the 16 most popular adapters pinned, keep_score, "
                         "or keep_score (40-epoch window) with the 32 most popular pinned")
    ap.add_argument("--churn-upload", choices=["batched", "copy"], default="batched",
                    help="churn: one upload kernel per group (default) or copy-engine copies per adapter")
    ap.add_argument("--churn-overlap", action="store_true",
                    help="churn: per-slot upload ordering, host runs ahead of the GPU")
    ap.add_argument("--e2e-staging-sets", type=int, default=E2E_STAGING_SETS,
                    help="e2e: device staging sets rotated by the host-buffer calls")
    ap.add_argument("--quick", action="store_true",
                    help="profiling runs: no clock settling, no e2e, no CPU baseline")
    args = ap.parse_args()
    if args.e2e_staging_sets < 1:
        ap.error("--e2e-staging-sets must be >= 1")
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload in ("prefill_5120", "mixed_ranks_8b"):
        return run_big(args, args.workload)
    if args.workload == "churn_4096":
        return run_churn(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
