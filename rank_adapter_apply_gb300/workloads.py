"""Seeded synthetic workloads for the multi-LoRA delta path.

This module only draws random numbers and lays them out. It holds none of the
method's arithmetic: no shrink, no expand, no scaling by alpha/r. Both the CUDA
path (through the binding) and the fp64 CPU oracle are fed from here, so that
the two sides see the same bits.

Shapes and distributions follow the five workloads the method is measured on:

* ``tiny_fp32``        one 512x512 layer, fp32, 4 slots of rank 16, alpha 32.
* ``decode_qv_4096``   q_proj and v_proj 4096->4096, bf16, 8 slots rank 16,
                       256 decode tokens, Zipf(1.1) slot ids, 10% base-only.
* ``prefill_5120``     32 contiguous sequences of 128..1024 tokens, hidden 5120,
                       q 5120->8192, k/v 5120->1024, o 8192->5120, bf16,
                       16 slots of rank 32, alpha 64.
* ``mixed_ranks_8b``   Llama-8B shapes (q, k, v, o, gate, up, down), bf16,
                       32 slots with ranks drawn from {8,16,32,64} padded to 64,
                       6 prefill segments of 640 tokens + 256 decode tokens.
* ``churn_4096``       decode_qv_4096 shapes, 64 GPU slots, 512 rank-16
                       adapters on the host, Zipf(1.2) ids with cold bursts.

Adapter weights use the PEFT convention (the adapter_config.json example on
the "vLLM LoRA Resolver 插件详解" page, section 3.2: fields ``r`` and
``lora_alpha``): A is [r, d_in] and B is [d_out, r], row-major.

bf16 tensors are carried as uint16 bit patterns (round-to-nearest-even of an
fp32 draw); fp32 tensors as float32.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

DTYPE_F32 = 0
DTYPE_BF16 = 1


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Decode uint16 bf16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def zipf_probs(n: int, s: float) -> np.ndarray:
    """Finite-support Zipf: P(k) proportional to k**-s for k = 1..n (id k-1)."""
    w = np.arange(1, n + 1, dtype=np.float64) ** (-s)
    return w / w.sum()


@dataclass
class Layer:
    name: str
    d_in: int
    d_out: int
    x_key: str          # which activation tensor feeds this layer


@dataclass
class Workload:
    """One batch of the path: activations, base outputs, adapters, slot ids."""
    name: str
    dtype: int                      # DTYPE_F32 or DTYPE_BF16
    max_loras: int                  # S
    max_lora_rank: int              # R
    layers: list[Layer]
    token_slot_idx: np.ndarray      # int32 [T]; -1 = base model only
    xs: dict[str, np.ndarray]       # activation name -> [T, d_in] (uint16 bits or f32)
    ys: dict[str, np.ndarray]       # layer name -> base output y_in [T, d_out]
    # per-slot adapters (true rank), one entry per slot: dict layer -> (A [r,d_in], B [d_out,r])
    adapters: list[dict[str, tuple[np.ndarray, np.ndarray]]]
    ranks: np.ndarray               # int32 [S] true rank per slot
    alphas: np.ndarray              # float64 [S]
    meta: dict = field(default_factory=dict)

    @property
    def n_tokens(self) -> int:
        return int(self.token_slot_idx.shape[0])

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == DTYPE_F32 else 2

    def padded_pools(self, layer: str) -> tuple[np.ndarray, np.ndarray]:
        """Slot pools for one layer with ranks zero-padded to max_lora_rank:
        A_pool [S, R, d_in] and B_pool [S, d_out, R] (same element type)."""
        ly = next(l for l in self.layers if l.name == layer)
        S, R = self.max_loras, self.max_lora_rank
        et = np.float32 if self.dtype == DTYPE_F32 else np.uint16
        A = np.zeros((S, R, ly.d_in), dtype=et)
        B = np.zeros((S, ly.d_out, R), dtype=et)
        for s, ad in enumerate(self.adapters):
            if ad is None:
                continue
            a, b = ad[layer]
            r = a.shape[0]
            A[s, :r, :] = a
            B[s, :, :r] = b
        return A, B


def _mat(rng, shape, kind, scale, dtype):
    if kind == "uniform":
        v = rng.uniform(-scale, scale, size=shape).astype(np.float32)
    else:
        v = (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale))
    return v if dtype == DTYPE_F32 else f32_to_bf16_bits(v)


def _adapter(rng, layers, r, dtype):
    """A ~ U(+-1/sqrt(d_in)), B ~ N(0, 0.02), per injected layer."""
    out = {}
    for ly in layers:
        a = _mat(rng, (r, ly.d_in), "uniform", 1.0 / np.sqrt(ly.d_in), dtype)
        b = _mat(rng, (ly.d_out, r), "normal", 0.02, dtype)
        out[ly.name] = (a, b)
    return out


def _base_out_direct(rng, T, ly, dtype):
    """Base output drawn as N(0, 0.02^2 * d_in): the distribution of x.W^T for
    x ~ N(0,1) and W ~ N(0, 0.02) without materialising W."""
    return _mat(rng, (T, ly.d_out), "normal", 0.02 * np.sqrt(ly.d_in), dtype)


def _base_out_matmul(rng, x, ly, dtype):
    """Base output y_in = x . W^T with W ~ N(0, 0.02) (the frozen base layer)."""
    w = rng.standard_normal(size=(ly.d_out, ly.d_in), dtype=np.float32) * np.float32(0.02)
    xf = x if dtype == DTYPE_F32 else bf16_bits_to_f32(x)
    y = (xf.astype(np.float64) @ w.astype(np.float64).T).astype(np.float32)
    return y if dtype == DTYPE_F32 else f32_to_bf16_bits(y)


def tiny_fp32(seed: int = 0) -> Workload:
    rng = np.random.default_rng(seed)
    S, R, r, alpha, T, d = 4, 16, 16, 32.0, 64, 512
    layers = [Layer("proj", d, d, "x")]
    adapters = [_adapter(rng, layers, r, DTYPE_F32) for _ in range(S)]
    x = _mat(rng, (T, d), "normal", 1.0, DTYPE_F32)
    y = _base_out_matmul(rng, x, layers[0], DTYPE_F32)
    idx = rng.integers(-1, S, size=T).astype(np.int32)
    return Workload("tiny_fp32", DTYPE_F32, S, R, layers, idx, {"x": x}, {"proj": y},
                    adapters, np.full(S, r, np.int32), np.full(S, alpha))


DECODE_LAYERS = [Layer("q_proj", 4096, 4096, "x"), Layer("v_proj", 4096, 4096, "x")]


def decode_batch(rng, T: int, S: int, direct_base: bool, layers=DECODE_LAYERS,
                 base_only_p: float = 0.1, zipf_s: float = 1.1):
    """One decode batch: x ~ N(0,1) bf16, base outputs, slot ids (-1 with
    probability base_only_p, else Zipf(zipf_s) over S slots)."""
    d = layers[0].d_in
    x = _mat(rng, (T, d), "normal", 1.0, DTYPE_BF16)
    ys = {}
    for ly in layers:
        ys[ly.name] = (_base_out_direct(rng, T, ly, DTYPE_BF16) if direct_base
                       else _base_out_matmul(rng, x, ly, DTYPE_BF16))
    base_only = rng.random(T) < base_only_p
    slots = rng.choice(S, size=T, p=zipf_probs(S, zipf_s)).astype(np.int32)
    idx = np.where(base_only, -1, slots).astype(np.int32)
    return x, ys, idx


def decode_qv_4096(seed: int = 0, direct_base: bool = False, n_tokens: int = 256,
                   rank: int = 16) -> Workload:
    """Decode batch on q_proj and v_proj (4096 -> 4096, bf16), 8 slots of one
    rank (16 by default; max_lora_rank the same), alpha = 2 x rank."""
    rng = np.random.default_rng(seed)
    S, R, r, alpha, T = 8, rank, rank, 2.0 * rank, n_tokens
    layers = list(DECODE_LAYERS)
    adapters = [_adapter(rng, layers, r, DTYPE_BF16) for _ in range(S)]
    x, ys, idx = decode_batch(rng, T, S, direct_base, layers)
    return Workload("decode_qv_4096", DTYPE_BF16, S, R, layers, idx, {"x": x}, ys,
                    adapters, np.full(S, r, np.int32), np.full(S, alpha))


def prefill_5120(seed: int = 0, n_seqs: int = 32, len_range=(128, 1024)) -> Workload:
    rng = np.random.default_rng(seed)
    S, R, r, alpha = 16, 32, 32, 64.0
    layers = [Layer("q_proj", 5120, 8192, "x"), Layer("k_proj", 5120, 1024, "x"),
              Layer("v_proj", 5120, 1024, "x"), Layer("o_proj", 8192, 5120, "attn")]
    adapters = [_adapter(rng, layers, r, DTYPE_BF16) for _ in range(S)]
    lens = rng.integers(len_range[0], len_range[1] + 1, size=n_seqs)
    seq_slot = rng.integers(0, S, size=n_seqs)
    idx = np.repeat(seq_slot, lens).astype(np.int32)
    T = int(lens.sum())
    xs = {"x": _mat(rng, (T, 5120), "normal", 1.0, DTYPE_BF16),
          "attn": _mat(rng, (T, 8192), "normal", 1.0, DTYPE_BF16)}
    ys = {ly.name: _base_out_direct(rng, T, ly, DTYPE_BF16) for ly in layers}
    return Workload("prefill_5120", DTYPE_BF16, S, R, layers, idx, xs, ys, adapters,
                    np.full(S, r, np.int32), np.full(S, alpha),
                    meta={"seq_lens": lens.tolist(), "seq_slots": seq_slot.tolist()})


def mixed_ranks_8b(seed: int = 0, n_segments: int = 6, seg_len: int = 640,
                   n_decode: int = 256) -> Workload:
    rng = np.random.default_rng(seed)
    S, R = 32, 64
    layers = [Layer("q_proj", 4096, 4096, "x"), Layer("k_proj", 4096, 1024, "x"),
              Layer("v_proj", 4096, 1024, "x"), Layer("o_proj", 4096, 4096, "attn"),
              Layer("gate_proj", 4096, 14336, "x"), Layer("up_proj", 4096, 14336, "x"),
              Layer("down_proj", 14336, 4096, "mlp")]
    ranks = rng.choice(np.array([8, 16, 32, 64]), size=S).astype(np.int32)
    alphas = 2.0 * ranks.astype(np.float64)
    adapters = [_adapter(rng, layers, int(ranks[s]), DTYPE_BF16) for s in range(S)]
    p = zipf_probs(S, 1.0)
    seg_slots = rng.choice(S, size=n_segments, p=p)
    dec_slots = rng.choice(S, size=n_decode, p=p)
    idx = np.concatenate([np.repeat(seg_slots, seg_len), dec_slots]).astype(np.int32)
    T = idx.shape[0]
    xs = {"x": _mat(rng, (T, 4096), "normal", 1.0, DTYPE_BF16),
          "attn": _mat(rng, (T, 4096), "normal", 1.0, DTYPE_BF16),
          "mlp": _mat(rng, (T, 14336), "normal", 1.0, DTYPE_BF16)}
    ys = {ly.name: _base_out_direct(rng, T, ly, DTYPE_BF16) for ly in layers}
    return Workload("mixed_ranks_8b", DTYPE_BF16, S, R, layers, idx, xs, ys, adapters,
                    ranks, alphas, meta={"seg_slots": seg_slots.tolist(), "seg_len": seg_len})


# ---------------------------------------------------------------------------
# Slot churn: adapter id streams (host-side), adapters drawn lazily per id.
# ---------------------------------------------------------------------------

@dataclass
class ChurnTrace:
    n_adapters: int
    steps: list[np.ndarray]         # per step: int64 adapter id per token


def churn_trace(seed: int = 0, n_adapters: int = 512, n_steps: int = 200,
                tokens: int = 256, zipf_s: float = 1.2, burst_every: int = 50,
                burst_len: int = 20) -> ChurnTrace:
    """Adapter ids per decode step. Zipf(zipf_s) over n_adapters (id = rank-1).
    At steps k with k % burst_every == 0 and k > 0 the last burst_len tokens take
    burst_len distinct cold ids: ids not used in the burst_every steps before,
    taken from the tail (highest id downward). (Ids never used at all run out:
    with Zipf(1.2) over 512 ids one is left before step 100 and none before
    step 150.)"""
    rng = np.random.default_rng(seed)
    p = zipf_probs(n_adapters, zipf_s)
    last_use = np.full(n_adapters, -(1 << 30), np.int64)    # step of each id's last use
    steps = []
    for k in range(n_steps):
        ids = rng.choice(n_adapters, size=tokens, p=p).astype(np.int64)
        if burst_every and k > 0 and k % burst_every == 0:
            cold = []
            cand = n_adapters - 1
            while len(cold) < burst_len and cand >= 0:
                if last_use[cand] < k - burst_every:
                    cold.append(cand)
                cand -= 1
            ids[tokens - len(cold):] = np.array(cold, dtype=np.int64)
        last_use[np.unique(ids)] = k
        steps.append(ids)
    return ChurnTrace(n_adapters, steps)


def churn_adapters(seed: int = 0, n_adapters: int = 512, d: int = 4096, r: int = 16):
    """Host adapter store for the churn workload: per layer (q_proj, v_proj)
    A [n, r, d] and B [n, d, r] as bf16 bits."""
    rng = np.random.default_rng(seed + 1000)
    out = {}
    for name in ("q_proj", "v_proj"):
        a = f32_to_bf16_bits(rng.uniform(-1 / np.sqrt(d), 1 / np.sqrt(d),
                                         size=(n_adapters, r, d)).astype(np.float32))
        b = f32_to_bf16_bits(rng.standard_normal(size=(n_adapters, d, r), dtype=np.float32)
                             * np.float32(0.02))
        out[name] = (a, b)
    return out


BY_NAME = {
    "tiny_fp32": tiny_fp32,
    "decode_qv_4096": decode_qv_4096,
    "prefill_5120": prefill_5120,
    "mixed_ranks_8b": mixed_ranks_8b,
}
