"""Element-wise comparison of the CUDA path with the fp64 oracle.

Tolerances:
* bf16 storage, fp32 accumulation: per element |g - o| <= 2e-3 + 1e-2 * |o|
  (the stated bounds max-abs 2e-3 and max-rel 1e-2 read as one allclose bound;
  a bf16 output alone carries up to half an ulp, 2**-9 relative, so a strict
  conjunction of the two maxima cannot hold for |o| > ~1).
* fp32: |g - o| <= 1e-5 + 1e-5 * |o| (fp32 rounding of 512-term sums).
Tokens whose slot index is -1, out of range or empty must be bit-identical to
the input.
"""
import numpy as np

import oracle
from rank_adapter_apply_gb300 import workloads as wl

TOL = {wl.DTYPE_BF16: (2e-3, 1e-2), wl.DTYPE_F32: (1e-5, 1e-5)}


def decode(arr, dtype):
    return (wl.bf16_bits_to_f32(arr) if dtype == wl.DTYPE_BF16 else arr).astype(np.float64)


def check_layer(w, layer, y_gpu, tokens=None, y_in=None, idx=None):
    """Compare GPU output of one layer with the oracle on `tokens` (all if None).
    Returns a dict of error statistics; raises AssertionError on a violation."""
    ly = next(l for l in w.layers if l.name == layer)
    A, B = w.padded_pools(layer)
    y_in = w.ys[layer] if y_in is None else y_in
    idx = w.token_slot_idx if idx is None else idx
    tok = np.arange(w.n_tokens) if tokens is None else np.asarray(tokens)
    ref = oracle.lora_apply_ref(w.xs[ly.x_key], y_in, A, B, w.ranks, w.alphas, idx,
                                tokens=tok, dtype=w.dtype)
    got = decode(y_gpu[tok], w.dtype)
    atol, rtol = TOL[w.dtype]
    s = idx[tok]
    active = (s >= 0) & (s < w.max_loras)
    active &= np.where(active, w.ranks[np.clip(s, 0, w.max_loras - 1)] > 0, False)
    # untouched rows: bit-identical
    if (~active).any():
        assert np.array_equal(y_gpu[tok][~active].view(np.uint8),
                              y_in[tok][~active].view(np.uint8)), f"{layer}: base-only row changed"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    stats = {"layer": layer, "n": int(active.sum()), "max_abs": float(err.max(initial=0.0)),
             "max_rel": float((err / np.maximum(np.abs(ref), 1e-30))[active].max(initial=0.0)),
             "worst_ratio": float((err / bound).max(initial=0.0))}
    assert not bad.any(), f"{layer}: {int(bad.sum())} elements out of tolerance, {stats}"
    return stats
