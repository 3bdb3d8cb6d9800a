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


# Delta-only comparison (base output y_in = 0, bf16): the output is then the
# rounded delta itself, so the error measures the delta's own precision rather
# than the rounding of y_in + delta.  Bound per element of token t:
#     |g - o| <= 2**-8 |o| + 2**-12 rms_t(o)
# 2**-8 is the unit roundoff of bf16 (8 significant bits, round to nearest):
# the one final rounding of the fp32 result.  The second term covers the fp32
# arithmetic before it, relative to the size of the token's delta: splitting
# the fp32 intermediate v into bf16 high and low parts keeps ~16 bits
# (|v - hi - lo| <= 2**-16 |v|), which over r products B_ik v_k is at most
# 2**-16 sum_k |B_ik v_k| ~ 2**-16 sqrt(r) rms_t(o) (about 2**-13 at r = 64);
# the fp32 sums of the shrink (d_in terms) and the expand (r terms) add
# ~2**-24 sqrt(n) relative.  Elements whose delta cancels to near zero are
# held to the absolute part only.
DELTA_RTOL = 2.0 ** -8
DELTA_ROW_ATOL = 2.0 ** -12


def zero_base(w):
    """The same workload with every base output y_in = 0 (bit pattern 0)."""
    for k in list(w.ys):
        w.ys[k] = np.zeros_like(w.ys[k])
    return w


def check_delta(w, layer, y_gpu, tokens=None):
    """y_gpu from a run with y_in = 0 against the oracle's delta (bf16 only).
    Returns error statistics; raises AssertionError past the bound above."""
    assert w.dtype == wl.DTYPE_BF16
    ly = next(l for l in w.layers if l.name == layer)
    A, B = w.padded_pools(layer)
    assert not w.ys[layer].any(), "check_delta needs y_in = 0"
    tok = np.arange(w.n_tokens) if tokens is None else np.asarray(tokens)
    ref = oracle.lora_apply_ref(w.xs[ly.x_key], w.ys[layer], A, B, w.ranks, w.alphas,
                                w.token_slot_idx, tokens=tok, dtype=w.dtype)
    got = decode(y_gpu[tok], w.dtype)
    s = w.token_slot_idx[tok]
    active = (s >= 0) & (s < w.max_loras)
    active &= np.where(active, w.ranks[np.clip(s, 0, w.max_loras - 1)] > 0, False)
    if (~active).any():
        assert not y_gpu[tok][~active].any(), f"{layer}: base-only row changed"
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    err = np.abs(got - ref)
    bound = DELTA_RTOL * np.abs(ref) + DELTA_ROW_ATOL * rms
    act = active[:, None] & np.ones_like(err, dtype=bool)
    ratio = np.where(act, err / np.maximum(bound, 1e-300), 0.0)
    big = act & (np.abs(ref) > 1e-3 * rms)
    stats = {"layer": layer, "n": int(active.sum()), "max_abs": float(err[act].max(initial=0.0)),
             "max_rel": float((err / np.maximum(np.abs(ref), 1e-300))[big].max(initial=0.0)),
             "max_abs_over_rms": float((err / np.maximum(rms, 1e-300))[act].max(initial=0.0)),
             "worst_ratio": float(ratio.max(initial=0.0))}
    assert stats["worst_ratio"] <= 1.0, f"{layer}: delta out of bound, {stats}"
    return stats
