#!/usr/bin/env python
"""Benchmark of the multi-LoRA delta path on one GB300 (or N replicas).

Headline (the largest workload that fits one GPU): ``prefill_5120`` -- 32
contiguous sequences of 128..1024 tokens (18,167 tokens with seed 0), hidden
5120, q_proj 5120->8192, k_proj / v_proj 5120->1024, o_proj 8192->5120, bf16,
16 slots of rank 32 (alpha 64), every sequence on one slot. One step = one
batch through the whole path for the whole layer set: token grouping, the
tensor-core shrink and expand of the long runs, the decode kernels for the
rest (none here).

* value: delta tokens per second per layer set, inputs resident in HBM (a
  step moves 1.6 GB, far above L2). The timed region is one CUDA-graph replay
  of exactly --steps steps, CUDA events on the launch stream, barrier and
  synchronize on both sides; it is repeated (at least 3 times, until about a
  second has passed) so that nvidia-smi can sample the clocks during it, and
  the median is reported.
* e2e: the same metric through lora_apply_multi_host with pinned HOST
  buffers: per step host admission of the batch's adapters, host-to-device
  copies of slot ids, activations and base outputs, the apply, device-to-host
  copies of every output; wall clock.
* cpu_baseline / --impl reference: the fp64 CPU oracle on the host cores over
  sampled tokens of the same workload.
* sub-records (same JSON line, key "workloads"), each with its own roofline:
  decode_qv_4096 (one step at a time and overlapped through programmatic
  dependent launch), mixed_ranks_8b, churn_4096 (LRU, and keep_score with a
  pinned warm set and overlapped uploads). Their timed regions have fixed
  sizes, independent of --steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
       [--workload prefill_5120|decode_qv_4096|mixed_ranks_8b|churn_4096]
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
HEADLINE = "prefill_5120"
DECODE = "decode_qv_4096"
T_TOKENS, N_SLOTS, RANK, ALPHA, D = 256, 8, 16, 32.0, 4096     # decode_qv_4096
E2E_HOST_SETS, E2E_STAGING_SETS = 32, 3     # decode e2e: pinned host sets (a sync per cycle), device staging sets
DECODE_CYCLES = 30                          # decode sub-record: graph of 30 cycles over the L2-defeating sets
BIG_STEPS = 40                              # mixed-rank sub-record: steps per timed graph
GRAPH_CHUNK = 512                           # steps captured per CUDA graph (a timed region may span several)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_traffic(record: str):
    """DRAM bytes per launch (or per step) from a committed ncu summary, if
    that summary was taken on the current sources of its kernels (else None)."""
    import hashlib
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", record)))
        for f, want in rec["kernel_sources"].items():
            src = os.path.join(ROOT, "rank_adapter_apply_gb300", "csrc", f)
            if hashlib.sha256(open(src, "rb").read()).hexdigest() != want:
                return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
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


def graph_chunks(n_steps: int, chunk: int = GRAPH_CHUNK):
    """Sizes of the CUDA graphs that together hold exactly n_steps steps."""
    full, rem = divmod(n_steps, chunk)
    return [chunk] * full + ([rem] if rem else [])


def capture_steps(stream, step, n_steps: int, first: int = 0):
    """CUDA graphs holding exactly n_steps calls of step(i), i = first, first+1, ..."""
    import torch
    graphs, i = [], first
    for size in graph_chunks(n_steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(size):
                step(i)
                i += 1
        graphs.append(g)
    return graphs


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def time_region(graphs, stream, dev, world, min_reps=3, min_total_ms=1000.0, max_reps=50):
    """Replay `graphs` (one timed region) repeatedly: each replay bracketed by a
    barrier and a device synchronize, timed by CUDA events on the launch
    stream. Returns the per-replay milliseconds."""
    import torch
    out = []
    while len(out) < max_reps and (len(out) < min_reps or sum(out) < min_total_ms):
        barrier(world)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for g in graphs:
                g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        out.append(e0.elapsed_time(e1))
    return out


# --------------------------------------------------------------------------
# CPU oracle timing (the only place besides the reference arm that runs it)
# --------------------------------------------------------------------------

def sample_tokens(idx: np.ndarray, n: int, seed: int = 5) -> np.ndarray:
    """A seeded sample of n adapter tokens of a batch, spread over all of it."""
    act = np.nonzero(idx >= 0)[0]
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(act, size=min(n, act.size), replace=False))


def oracle_tokens_per_s(w, tokens, budget_s: float, threads=None, max_passes=None):
    """The fp64 oracle over the sampled tokens of every layer of the workload,
    repeated until the budget is spent. Returns (delta tokens/s, passes,
    threads, seconds)."""
    import oracle
    all_cores = oracle.threads()
    if threads is not None:
        oracle.set_threads(threads)
    try:
        pools = {ly.name: w.padded_pools(ly.name) for ly in w.layers}
        oracle.lora_apply_ref(w.xs[w.layers[0].x_key], w.ys[w.layers[0].name], *pools[w.layers[0].name],
                              w.ranks, w.alphas, w.token_slot_idx, tokens=tokens[:1], dtype=w.dtype)
        t0 = time.perf_counter()
        passes = 0
        while True:
            for ly in w.layers:
                oracle.lora_apply_ref(w.xs[ly.x_key], w.ys[ly.name], *pools[ly.name], w.ranks, w.alphas,
                                      w.token_slot_idx, tokens=tokens, dtype=w.dtype)
            passes += 1
            el = time.perf_counter() - t0
            if el >= budget_s or (max_passes and passes >= max_passes):
                break
        return passes * len(tokens) / el, passes, oracle.threads(), el
    finally:
        oracle.set_threads(all_cores)


def run_reference(args):
    """The reference arm: the fp64 oracle, as it stands, on the host cores, on
    the workload and metric of our arm. Each step is a bounded sample of the
    batch (seeded adapter tokens, every layer), sized so the whole run takes
    about a minute."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    w = load_workload(args.workload)
    if args.workload == "churn_4096":
        print(json.dumps({"impl": "reference", "unavailable": "churn is timed on the GPU only"}), flush=True)
        return 0
    pools = {ly.name: w.padded_pools(ly.name) for ly in w.layers}
    probe = sample_tokens(w.token_slot_idx, 16)

    def step(i, toks):
        for ly in w.layers:
            oracle.lora_apply_ref(w.xs[ly.x_key], w.ys[ly.name], *pools[ly.name], w.ranks, w.alphas,
                                  w.token_slot_idx, tokens=toks, dtype=w.dtype)
        return len(toks)
    t0 = time.perf_counter()
    step(0, probe)
    per_tok = (time.perf_counter() - t0) / len(probe)
    n_tok = int(max(1, min(int((w.token_slot_idx >= 0).sum()),
                           60.0 / max(1, args.steps + args.warmup) / max(per_tok, 1e-9))))
    samples = [sample_tokens(w.token_slot_idx, n_tok, seed=11 + i) for i in range(4)]
    for i in range(args.warmup):
        step(i, samples[i % 4])
    t0 = time.perf_counter()
    toks = sum(step(i, samples[i % 4]) for i in range(args.steps))
    el = time.perf_counter() - t0
    v = toks / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                             "sample": f"{n_tok} seeded adapter tokens of the {w.n_tokens}-token batch, "
                                       f"every layer ({', '.join(l.name for l in w.layers)}), per step"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def load_workload(name, prefill_seqs=32):
    if name == DECODE:
        return wl.decode_qv_4096(0)
    if name == HEADLINE and prefill_seqs != 32:
        return wl.prefill_5120(0, n_seqs=prefill_seqs)      # smaller case for profiler captures
    return wl.BY_NAME[name](0)


def workload_config(w):
    return {"workload": w.name, "tokens": w.n_tokens,
            "adapter_tokens": int((w.token_slot_idx >= 0).sum()),
            "layers": [f"{l.name} {l.d_in}->{l.d_out}" for l in w.layers],
            "max_loras": w.max_loras, "max_lora_rank": w.max_lora_rank,
            "ranks": sorted({int(r) for r in w.ranks}), "parallelism": "replicas"}


# --------------------------------------------------------------------------
# Our arm
# --------------------------------------------------------------------------

def run_ours(args):
    import torch
    import torch.distributed as dist
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300 import build as build_mod

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(B.LIB_PATH):
        build_mod.build()
    barrier(world)
    B.load()
    ctx = {"dev": dev, "world": world, "rank": rank, "local": local}

    if args.workload == "churn_4096":
        line = run_churn(args, ctx, args.churn_policy, args.churn_overlap)
    elif args.workload == DECODE:
        line = run_decode(args, ctx)
    else:
        line = run_big(args, ctx, args.workload, headline=True)
        if not args.quick and not args.no_subrecords:
            line["workloads"] = subrecords(args, ctx)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def subrecords(args, ctx):
    """The other workloads, each timed on its own fixed-size region."""
    out = {}
    jobs = [(DECODE, lambda: run_decode(args, ctx, sub=True)),
            ("mixed_ranks_8b", lambda: run_big(args, ctx, "mixed_ranks_8b", headline=False)),
            ("churn_4096 lru", lambda: run_churn(args, ctx, "lru", False, sub=True)),
            ("churn_4096 lru overlap", lambda: run_churn(args, ctx, "lru", True, sub=True)),
            ("churn_4096 keep_pin32 overlap", lambda: run_churn(args, ctx, "keep_pin32", True, sub=True))]
    for name, job in jobs:
        try:
            out[name] = job()
        except Exception as e:          # a sub-record never takes the headline down
            out[name] = {"error": f"{type(e).__name__}: {e}"}
    return out


def run_big(args, ctx, name, headline):
    """One large batch per step through every layer of the set (prefill_5120,
    mixed_ranks_8b). Headline: exactly --steps steps per timed region, plus
    e2e and the CPU oracle. Sub-record: BIG_STEPS steps per timed region."""
    import torch
    from rank_adapter_apply_gb300.harness import DeviceWorkload
    dev, world, rank = ctx["dev"], ctx["world"], ctx["rank"]
    w = load_workload(name, args.prefill_seqs if headline else 32)
    dw = DeviceWorkload(w, device=dev, max_tokens=w.n_tokens)
    lys = list(range(len(w.layers)))
    xs = [dw.xs[ly.x_key] for ly in w.layers]
    ys = [dw.ys[ly.name] for ly in w.layers]
    st = dw.slots.compute
    n_steps = args.steps if headline else BIG_STEPS

    def step(_):
        dw.slots.apply_multi(lys, xs, ys, dw.idx)

    with torch.cuda.stream(st):
        step(0)                                  # eager: kernel attributes, pending uploads
    st.synchronize()
    warm = capture_steps(st, step, 1)
    k0 = dw.slots.stats()["kernel_launches"]
    graphs = capture_steps(st, step, n_steps)
    launches = dw.slots.stats()["kernel_launches"] - k0     # kernels of one timed region
    with torch.cuda.stream(st):
        for _ in range(max(3, args.warmup)):
            warm[0].replay()
    st.synchronize()

    sampler = ClockSampler(ctx["local"])
    sampler.start()
    time.sleep(0.12)
    reps = time_region(graphs, st, dev, world)
    clocks = ClockSampler.summary(sampler.stop())
    ms = statistics.median(reps)
    act = int((w.token_slot_idx >= 0).sum())
    ms_job, job_tokens = reduce_over_ranks(ms, act * n_steps, dev)
    bytes_ = algorithmic_bytes(w.token_slot_idx, w.ranks, w.layers)
    flops = algorithmic_flops(w.token_slot_idx, w.ranks, w.layers)
    hbm, kind = peaks()
    ach = bytes_ * n_steps / (ms * 1e-3) / 1e9
    roof = {"bound": "hbm",
            "kernel": "whole step (one launch sequence per step: group_tokens, prefill_shrink, "
                      "[prefill_reduce], prefill_expand, decode shrink + expand; every layer of the set)",
            "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "peak_kind": kind,
            "frac_of_8TBps": ach / 8000.0,
            "traffic": kernel_traffic(f"{name}_traffic.json"),
            "algorithmic_bytes_per_step": bytes_,
            "tflops": flops * n_steps / (ms * 1e-3) / 1e12}
    line = {"metric": METRIC, "value": job_tokens / (ms_job * 1e-3), "unit": UNIT, "n_gpus": world,
            "steps": n_steps, "warmup": args.warmup, "ms_per_step": ms_job / n_steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded numpy, shapes and slot structure of the workload)",
            "config": {**workload_config(w),
                       "l2": f"inputs larger than L2 ({bytes_ / 2**20:.0f} MiB per step)",
                       "timing": f"one CUDA-graph replay of exactly {n_steps} steps per timed region, "
                                 f"CUDA events on the launch stream; median of {len(reps)} regions "
                                 f"(min {min(reps) / n_steps:.4f}, max {max(reps) / n_steps:.4f} ms per step)"},
            "roofline": roof, "gpu_launches": launches, "clocks": clocks}
    if headline and not args.quick:
        line["e2e"] = big_e2e(args, w, dw, dev, world)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            tok = sample_tokens(w.token_slot_idx, 256)
            v, n, cores, el = oracle_tokens_per_s(w, tok, args.cpu_seconds)
            tok1 = sample_tokens(w.token_slot_idx, 16, seed=6)
            v1, n1, _, el1 = oracle_tokens_per_s(w, tok1, max(1.0, args.cpu_seconds / 3), threads=1)
            line["cpu_baseline"] = {
                "value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample": f"{n} passes over {len(tok)} seeded adapter tokens of the {w.n_tokens}-token batch, "
                          f"every layer, in {el:.1f} s",
                "single_thread": {"value": v1, "cores": 1,
                                  "sample": f"{n1} passes over {len(tok1)} tokens in {el1:.1f} s"}}
    dw.close()
    return line


def big_e2e(args, w, dw, dev, world, host_idx_ring=64):
    """Whole-job throughput through lora_apply_multi_host with pinned host
    buffers, for a large batch: per step the admission of every token's
    adapter (lora_assign_tokens, written into a pinned slot-id buffer), the
    copies in (slot ids; one packed block of activations and base outputs),
    the apply, the copies back of every output, the release. Two host blocks
    are paired with two device staging blocks, so a call's copies in wait for
    the copies back of the call two steps earlier that used the same blocks;
    slot-id buffers rotate over a ring and are reused after a host sync."""
    import ctypes
    import torch
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300.harness import to_torch
    lib = B.load()
    c = dw.slots.ctx
    T = w.n_tokens
    # admission: adapter id s bound to slot s (the pools already hold adapter s)
    for s in range(w.max_loras):
        rc, slot, _, _ = B.lora_assign(c, s, int(w.ranks[s]))
        if rc != 0 or slot != s:
            raise RuntimeError("unexpected slot binding")
    # block layout, in the library's copy order (x once per distinct input, then y)
    order, offs, off = [], {}, 0
    for ly in w.layers:
        if ly.x_key not in offs:
            offs[ly.x_key] = off
            order.append(("x", ly.x_key))
            off += T * ly.d_in * 2
        offs["y:" + ly.name] = off
        order.append(("y", ly.name))
        off += T * ly.d_out * 2
    blk = off
    n_sets = 2
    hblk = [torch.empty(blk, dtype=torch.uint8).pin_memory() for _ in range(n_sets)]
    dblk = [torch.empty(blk, dtype=torch.uint8, device=dev) for _ in range(n_sets)]
    for hb in hblk:
        for kind, key in order:
            src = w.xs[key] if kind == "x" else w.ys[key]
            o = offs[key] if kind == "x" else offs["y:" + key]
            hb[o:o + src.nbytes].copy_(to_torch(src, w.dtype).view(torch.uint8).reshape(-1))
    nl = len(w.layers)
    lay = B._i32_array(list(range(nl)))
    xs_h = [B._vp_array([hb.data_ptr() + offs[ly.x_key] for ly in w.layers]) for hb in hblk]
    ys_h = [B._vp_array([hb.data_ptr() + offs["y:" + ly.name] for ly in w.layers]) for hb in hblk]
    xs_d = [B._vp_array([db.data_ptr() + offs[ly.x_key] for ly in w.layers]) for db in dblk]
    ys_d = [B._vp_array([db.data_ptr() + offs["y:" + ly.name] for ly in w.layers]) for db in dblk]
    idx_h = torch.empty((host_idx_ring, T), dtype=torch.int32).pin_memory()
    idx_d = [torch.empty(T, dtype=torch.int32, device=dev) for _ in range(n_sets)]
    ids = np.ascontiguousarray(np.where(w.token_slot_idx >= 0, w.token_slot_idx, -1).astype(np.int64)
                               .astype(np.uint64))
    P = ctypes.POINTER
    ids_p = ids.ctypes.data_as(P(ctypes.c_uint64))
    ranks = np.ascontiguousarray(np.where(w.token_slot_idx >= 0, w.ranks[np.clip(w.token_slot_idx, 0, None)],
                                          1).astype(np.int32))
    ranks_p = ranks.ctypes.data_as(P(ctypes.c_int))
    S = w.max_loras
    dids, slots = np.zeros(S, np.uint64), np.zeros(S, np.int32)
    need, evi = np.zeros(S, np.int32), np.zeros(S, np.uint64)
    dids_p, slots_p = dids.ctypes.data_as(P(ctypes.c_uint64)), slots.ctypes.data_as(P(ctypes.c_int))
    need_p, evi_p = need.ctypes.data_as(P(ctypes.c_int)), evi.ctypes.data_as(P(ctypes.c_uint64))
    nd, ndone = ctypes.c_int(0), ctypes.c_int(0)
    act = int((w.token_slot_idx >= 0).sum())

    def step(i):
        r = i % host_idx_ring
        if r == 0 and i > 0:
            B.check(lib.lora_sync_host(c))        # the slot-id ring is reused from here
        ip = ctypes.cast(idx_h[r].data_ptr(), P(ctypes.c_int))
        rc = lib.lora_assign_tokens(c, T, ids_p, ranks_p, 1, ip, S, dids_p, slots_p, need_p, evi_p,
                                    ctypes.byref(nd), ctypes.byref(ndone))
        if rc != 0 or need[:nd.value].any():
            raise RuntimeError("adapter unexpectedly not resident")
        b = i % n_sets
        B.check(lib.lora_apply_multi_host(c, nl, lay, xs_h[b], ys_h[b], idx_h[r].data_ptr(), T,
                                          xs_d[b], ys_d[b], idx_d[b].data_ptr()))
        B.check(lib.lora_release_batch(c, nd.value, slots_p))
        return act

    for i in range(max(2, min(args.warmup, 4))):
        step(i)
    B.check(lib.lora_sync_host(c))
    k = max(4, min(args.steps, 40))
    # three timed regions of k steps each; the median region is reported (the
    # host link's speed varies from one region to the next)
    regions = []
    i0 = 0
    for _ in range(3):
        barrier(world)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        toks = sum(step(i0 + i) for i in range(k))
        B.check(lib.lora_sync_host(c))
        el = time.perf_counter() - t0
        i0 += k
        regions.append(reduce_over_ranks(el * 1e3, toks, dev))
    regions.sort(key=lambda r: r[0])
    el_ms, job_toks = regions[1]
    h2d = T * 4 + blk
    d2h = sum(T * ly.d_out * 2 for ly in w.layers)
    floor = big_link_floor(hblk, dblk, [(offs["y:" + ly.name], T * ly.d_out * 2) for ly in w.layers], dev)
    del hblk, dblk
    return {"value": job_toks / (el_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": k, "ms_per_step": el_ms / k, "link_floor": floor,
            "regions_ms_per_step": [round(r[0] / k, 4) for r in regions],
            "timing": "wall clock, host admission + H2D + apply + D2H per step, two buffer sets rotated; "
                      "median of three regions of `steps` steps"}


def big_link_floor(hblk, dblk, outs, dev, reps=8):
    """Time per step of the host link alone for the e2e loop: the whole block
    copied in on one stream while the previous step's outputs are copied back
    on another, same two buffer sets, no kernels and no admission."""
    import torch
    si, so = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = [torch.cuda.Event() for _ in dblk]
    for e in ev:
        e.record(so)

    def run(n):
        for i in range(n):
            b = i % len(dblk)
            with torch.cuda.stream(si):
                si.wait_event(ev[b])
                dblk[b].copy_(hblk[b], non_blocking=True)
            so.wait_stream(si)
            with torch.cuda.stream(so):
                for o, nb in outs:
                    hblk[b][o:o + nb].copy_(dblk[b][o:o + nb], non_blocking=True)
                ev[b].record(so)
    run(2)
    times = []
    for _ in range(3):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        run(reps)
        torch.cuda.synchronize(dev)
        times.append((time.perf_counter() - t0) / reps * 1e3)
    times.sort()
    return {"ms_per_step": times[1],
            "note": "the step's bytes copied in and out concurrently on two streams, same buffers, no kernels; "
                    "median of three regions"}


# --------------------------------------------------------------------------
# Decode workload (256 tokens, q_proj + v_proj)
# --------------------------------------------------------------------------

def make_batches(n_sets: int, seed0: int = 0):
    """Set 0 is the decode workload itself; sets 1.. draw new x, base outputs
    and slot ids with the same recipe (base output drawn directly)."""
    w = wl.decode_qv_4096(seed0)
    batches = [(w.xs["x"], w.ys, w.token_slot_idx)]
    for i in range(1, n_sets):
        rng = np.random.default_rng(seed0 + 7919 * i)
        batches.append(wl.decode_batch(rng, T_TOKENS, N_SLOTS, True))
    return w, batches


def run_decode(args, ctx, sub=False):
    """Decode steps cycling over enough distinct sets (x, y, slot ids and slot
    pools each) to exceed 2.5 x L2. Two timed graphs of the same fixed number
    of steps: one step at a time (each kernel waits for the one before), and
    overlapped (inputs declared ready: a step's kernel starts under the
    previous one and waits for it only before touching y)."""
    import torch
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300.harness import to_torch
    from rank_adapter_apply_gb300.slots import LoraSlots
    dev, world, rank = ctx["dev"], ctx["world"], ctx["rank"]
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
    for x, ys, idx in batches:
        d = DevSet()
        d.slots = LoraSlots(layers, N_SLOTS, RANK, T_TOKENS, dtype=torch.bfloat16, device=dev,
                            compute_stream=stream, upload_stream=upload)
        for s in range(N_SLOTS):
            rc, slot, need, _ = d.slots.assign(s, RANK)     # adapter id s -> slot, a miss on first sight
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

    def step(i):
        d = sets[i % len(sets)]
        d.slots.apply_multi([0, 1], [d.x, d.x], d.ys, d.idx)

    with torch.cuda.stream(stream):
        for i in range(len(sets)):
            step(i)                                   # eager: clears pending-upload waits
    torch.cuda.synchronize(dev)
    n_steps = len(sets) * (DECODE_CYCLES if not args.quick else 3)
    modes = {}
    for mode, ready in (("one_at_a_time", False), ("overlapped", True)):
        for d in sets:
            B.lora_set_inputs_ready(d.slots.ctx, ready)
        k0 = sum(d.slots.stats()["kernel_launches"] for d in sets)
        graphs = capture_steps(stream, step, n_steps)
        launches = sum(d.slots.stats()["kernel_launches"] for d in sets) - k0
        with torch.cuda.stream(stream):
            for g in graphs:
                g.replay()
        torch.cuda.synchronize(dev)
        modes[mode] = (graphs, launches)
    sampler = ClockSampler(ctx["local"])
    sampler.start()
    time.sleep(0.12)
    res = {}
    for mode, (graphs, launches) in modes.items():
        reps = time_region(graphs, stream, dev, world, min_reps=5, min_total_ms=300.0)
        res[mode] = (statistics.median(reps), launches, len(reps))
    clocks = ClockSampler.summary(sampler.stop())
    tokens = sum(sets[i % len(sets)].t_act for i in range(n_steps))
    bytes_ = sum(sets[i % len(sets)].bytes for i in range(n_steps))
    flops = sum(sets[i % len(sets)].flops for i in range(n_steps))
    hbm, kind = peaks()
    out = {}
    for mode, (ms, launches, nrep) in res.items():
        ms_job, job_tokens = reduce_over_ranks(ms, tokens, dev)
        ach = bytes_ / (ms * 1e-3) / 1e9
        out[mode] = {"value": job_tokens / (ms_job * 1e-3), "us_per_step": ms_job * 1e3 / n_steps,
                     "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                                  "frac": ach / hbm, "peak_kind": kind, "frac_of_8TBps": ach / 8000.0,
                                  "tflops": flops / (ms * 1e-3) / 1e12},
                     "gpu_launches": launches, "timed_regions": nrep}
    floor = copy_floor(bytes_ / n_steps, stream, dev, l2)
    e2e = None if args.quick else run_e2e(args, w, batches, sets[0], stream, dev, world)
    line = {"metric": METRIC, "unit": UNIT, "steps": n_steps, "n_gpus": world,
            "value": out["overlapped"]["value"], "ms_per_step": out["overlapped"]["us_per_step"] * 1e-3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded numpy: x~N(0,1), A~U(+-1/64), B~N(0,0.02), Zipf(1.1) slots, 10% base-only)",
            "config": {"workload": DECODE, "tokens_per_batch": T_TOKENS, "layers": ["q_proj", "v_proj"],
                       "d": D, "max_loras": N_SLOTS, "rank": RANK, "alpha": ALPHA,
                       "l2": f"inputs larger than L2: {len(sets)} distinct x/y/idx/pool sets, "
                             f"{len(sets) * per_set / 2**20:.0f} MiB per cycle vs L2 {l2 / 2**20:.0f} MiB",
                       "timing": f"one timed region = CUDA-graph replays of exactly {n_steps} steps "
                                 f"({len(sets)} sets x {n_steps // len(sets)} cycles), independent of --steps; "
                                 "CUDA events on the launch stream; median over regions"},
            "one_at_a_time": out["one_at_a_time"], "overlapped": out["overlapped"],
            "roofline": {**out["overlapped"]["roofline"],
                         "kernel": "decode_cluster_kernel (one launch per step: grouping, shrink and "
                                   "expand of q_proj and v_proj)",
                         "traffic": kernel_traffic("decode_cluster_qv4096_traffic.json"),
                         "copy_floor": floor, "algorithmic_bytes_per_step": bytes_ / n_steps},
            "e2e": e2e, "gpu_launches": out["overlapped"]["gpu_launches"], "clocks": clocks}
    if not sub and rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quick:
        tok = np.arange(T_TOKENS)[w.token_slot_idx >= 0]
        v, n, cores, el = oracle_tokens_per_s(w, tok, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{n} passes over the batch's adapter tokens in {el:.1f} s"}
    for d in sets:
        d.slots.close()
    return line


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
    import ctypes
    import torch
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300.harness import to_torch

    ctx = d0.slots.ctx
    B.lora_set_inputs_ready(ctx, True)
    nh = min(E2E_HOST_SETS, len(batches))      # host buffer sets, reused after a sync
    nd_sets = args.e2e_staging_sets
    lib = B.load()
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
    k = nh * 30                                 # fixed: 30 cycles over the host sets
    barrier(world)
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


# --------------------------------------------------------------------------
# Slot churn
# --------------------------------------------------------------------------

def run_churn(args, ctx, policy, overlap, sub=False):
    """Slot churn: 64 GPU slots, 512 rank-16 adapters in pinned host memory,
    Zipf(1.2) adapter ids with a burst of 20 cold adapters every 50 steps; all
    200 steps of the trace (fewer if --steps is smaller and this is not a
    sub-record)."""
    from rank_adapter_apply_gb300.churn import KEEP_PIN32, ChurnRunner
    steps = 200 if (sub or args.steps >= 200) else args.steps
    trace = wl.churn_trace(0, n_steps=steps)
    warm = wl.churn_trace(99, n_steps=20)
    pol = {"lru": {}, "pin16": {"pin_top": 16},
           "keep": {"policy": 1, "weights": (1.0, 1.0, 0.0, 0.0, 0.0)},
           "keep_pin32": dict(KEEP_PIN32)}[policy]
    r = ChurnRunner(overlap=overlap, device=ctx["dev"], **pol)
    try:
        r.run(warm, reset_y=False)
        base = r.slots.stats()
        res = r.run(trace, reset_y=False)
        st = res.stats
    finally:
        r.close()
    d = {k: st[k] - base[k] for k in ("hits", "misses", "evictions", "reloads_after_eviction",
                                      "uploads", "upload_bytes")}
    up_s = st["upload_seconds"] - base["upload_seconds"]
    return {"metric": "slot-churn decode steps/s (admission, H2D uploads, q_proj+v_proj delta)",
            "value": res.steps / res.wall_s, "unit": "steps/s", "n_gpus": 1, "steps": res.steps,
            "warmup": len(warm.steps), "ms_per_step": res.wall_s * 1e3 / res.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded Zipf(1.2) adapter ids over 512 with cold bursts)",
            "config": {"workload": "churn_4096", "max_loras": 64, "host_adapters": 512, "rank": 16,
                       "eviction_policy": policy, "upload_overlap": overlap,
                       "host_calls_per_step": "one lora_serve_step",
                       "tokens_per_step": 256, "timing": "wall clock over every step of the trace, "
                                                         "host bookkeeping included"},
            "churn": {**d, "thrash_ratio": (d["reloads_after_eviction"] / d["evictions"]) if d["evictions"] else 0.0,
                      "hit_rate": d["hits"] / max(1, d["hits"] + d["misses"]),
                      "h2d_GBps": d["upload_bytes"] / up_s / 1e9 if up_s > 0 else None,
                      "delta_tokens_per_s": res.tokens / res.wall_s},
            "gpu_launches": st["kernel_launches"] - base["kernel_launches"]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-subrecords", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload", default=HEADLINE,
                    choices=[HEADLINE, DECODE, "mixed_ranks_8b", "churn_4096"])
    ap.add_argument("--churn-policy", choices=["lru", "pin16", "keep", "keep_pin32"], default="lru",
                    help="churn: pure LRU, LRU with the 16 most popular adapters pinned, keep_score, "
                         "or keep_score (40-epoch window) with the 32 most popular pinned")
    ap.add_argument("--churn-overlap", action="store_true",
                    help="churn: per-slot upload ordering, host runs ahead of the GPU")
    ap.add_argument("--e2e-staging-sets", type=int, default=E2E_STAGING_SETS,
                    help="decode e2e: device staging sets rotated by the host-buffer calls")
    ap.add_argument("--prefill-seqs", type=int, default=32,
                    help="sequences of the prefill workload (32 = the full workload; fewer only for "
                         "profiler captures)")
    ap.add_argument("--quick", action="store_true",
                    help="profiling runs: no e2e, no CPU baseline, no sub-records, short decode graphs")
    args = ap.parse_args()
    if args.e2e_staging_sets < 1:
        ap.error("--e2e-staging-sets must be >= 1")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
