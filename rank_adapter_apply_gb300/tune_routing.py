"""Measure where the cluster decode kernel stops beating the grouped kernels.

    python -m rank_adapter_apply_gb300.tune_routing [--ranks 16,32,64] [--tokens 256,512,768,1024]

For every (max_lora_rank, batch size) it builds the decode batch of q_proj and
v_proj (4096 -> 4096, bf16, 8 slots of that rank, 10 % base-only tokens, Zipf
slot ids), runs the same lora_apply_multi call once with every batch sent to the
cluster kernel (lora_set_small_batch_tokens 1024) and once with none (0), and
prints one JSON line per point with the time per call of each path (CUDA-graph
replays timed with CUDA events on the library's compute stream; operands stay
in L2 for both paths alike). The last line gives, per rank, the largest batch
size at which the cluster kernel was faster: the value to pass to
lora_set_small_batch_tokens for layer shapes like these.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import binding as B
from . import build as build_mod
from . import workloads as wl
from .harness import DeviceWorkload

CLUSTER_ALL = 1024      # every batch of up to 1024 tokens to the cluster kernel
CLUSTER_NONE = 0        # every batch to the grouped kernels


def time_apply(dw: DeviceWorkload, calls_per_graph: int = 10, reps: int = 50) -> float:
    """Microseconds per lora_apply_multi call over both layers."""
    w = dw.w
    lys = list(range(len(w.layers)))
    xs = [dw.xs[w.layers[i].x_key] for i in lys]
    ys = [dw.ys[w.layers[i].name] for i in lys]
    st = dw.slots.compute
    with torch.cuda.stream(st):
        for _ in range(3):
            dw.slots.apply_multi(lys, xs, ys, dw.idx)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for _ in range(calls_per_graph):
            dw.slots.apply_multi(lys, xs, ys, dw.idx)
    with torch.cuda.stream(st):
        g.replay()
    st.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    with torch.cuda.stream(st):
        for _ in range(reps):
            g.replay()
    e1.record(st)
    st.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * calls_per_graph)


def measure(rank: int, tokens: int, seed: int = 0) -> dict:
    w = wl.decode_qv_4096(seed, direct_base=True, n_tokens=tokens, rank=rank)
    out = {"max_lora_rank": rank, "tokens": tokens}
    for name, limit in (("cluster_us", CLUSTER_ALL), ("grouped_us", CLUSTER_NONE)):
        dw = DeviceWorkload(w, small_batch_tokens=limit)
        try:
            out[name] = round(time_apply(dw), 2)
            st = dw.slots.stats()
            served = st["cluster_applies"] if limit else st["grouped_applies"]
            if served == 0:
                raise RuntimeError(f"{name}: no call took the requested path ({st})")
        finally:
            dw.close()
    out["faster"] = "cluster" if out["cluster_us"] < out["grouped_us"] else "grouped"
    return out


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--ranks", default="16,32,64")
    ap.add_argument("--tokens", default="256,512,768,1024")
    ap.add_argument("--seed", type=int, default=0)
    a = ap.parse_args(argv)
    if not torch.cuda.is_available():
        raise SystemExit("tune_routing needs a CUDA device")
    build_mod.build()
    B.load()
    ranks = [int(v) for v in a.ranks.split(",")]
    tokens = sorted(int(v) for v in a.tokens.split(","))
    if any(t < 1 or t > CLUSTER_ALL for t in tokens):
        raise SystemExit(f"token counts must be in 1..{CLUSTER_ALL}")
    largest = {}
    for r in ranks:
        # the largest measured size up to which the cluster kernel won every point
        largest[str(r)] = 0
        still_winning = True
        for t in tokens:
            res = measure(r, t, a.seed)
            print(json.dumps(res), flush=True)
            still_winning = still_winning and res["faster"] == "cluster"
            if still_winning:
                largest[str(r)] = t
    print(json.dumps({"largest_cluster_batch": largest}), flush=True)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
