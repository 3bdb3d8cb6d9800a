"""CPU tests of the benchmark's host-side arithmetic: the algorithmic bytes and
flops that form the roofline numerators, and the job-wide figures."""
import numpy as np

import bench
import oracle
from rank_adapter_apply_gb300 import workloads as wl


def _layers():
    # two layers reading one input (as q_proj / v_proj do), d_in 8, d_out 16 and 4
    return [wl.Layer("a", 8, 16, "x"), wl.Layer("b", 8, 4, "x")]


def test_bytes_and_flops_by_hand():
    """4 tokens, slot ids [0, -1, 1, 0], ranks 2 and 3, bf16 (2 bytes):
    slot ids 4 x 4 = 16; x once for the shared input, 3 adapter rows x 8 x 2 = 48;
    layer a: y read + written 3 x 2 x 16 x 2 = 192, weights (8 + 16) x (2 + 3) x 2 = 240;
    layer b: y 3 x 2 x 4 x 2 = 48, weights (8 + 4) x 5 x 2 = 120.  Total 664.
    Flops: 2 r (d_in + d_out) per adapter token and layer:
    layer a 2 x 2 x 24 x 2 + 2 x 3 x 24 = 336, layer b 2 x 2 x 12 x 2 + 2 x 3 x 12 = 168."""
    idx = np.array([0, -1, 1, 0], np.int32)
    ranks = np.array([2, 3], np.int32)
    assert bench.algorithmic_bytes(idx, ranks, _layers()) == 664
    assert bench.algorithmic_flops(idx, ranks, _layers()) == 504


def test_distinct_inputs_are_counted_once_each():
    """A layer with its own input adds its x rows; one sharing an input does not."""
    idx = np.array([1, 1, -1], np.int32)
    ranks = np.array([4, 8], np.int32)
    shared = [wl.Layer("a", 8, 16, "x"), wl.Layer("b", 8, 16, "x")]
    own = [wl.Layer("a", 8, 16, "x"), wl.Layer("b", 8, 16, "z")]
    assert bench.algorithmic_bytes(idx, ranks, own) - bench.algorithmic_bytes(idx, ranks, shared) == 2 * 8 * 2


def test_weight_term_matches_the_capacity_formula():
    """At the decode headline shapes, the weight part of the byte count equals
    the capacity formula (the oracle's, written from the LRU page) summed over
    the slots the batch uses; the rest is x, y and the slot ids."""
    w, batches = bench.make_batches(2)
    for x, ys, idx in batches:
        act = idx[idx >= 0]
        used = np.unique(act)
        dims = [(ly.d_in, ly.d_out) for ly in w.layers]
        weights = sum(oracle.adapter_bytes(dims, int(w.ranks[s]), 2) for s in used)
        rest = idx.shape[0] * 4 + act.size * bench.D * 2 + len(w.layers) * act.size * 2 * bench.D * 2
        assert bench.algorithmic_bytes(idx, w.ranks, w.layers) == weights + rest
        # 230-odd adapter tokens of 256 and up to 8 rank-16 slots: about 13.6 MB
        assert 12.5e6 < weights + rest < 14.7e6


def test_job_wide_reduction_single_rank():
    """One process: the job-wide time and tokens are its own."""
    ms, toks = bench.reduce_over_ranks(12.5, 1000, None)
    assert (ms, toks) == (12.5, 1000)
