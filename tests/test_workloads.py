"""CPU tests of the seeded input recipes: the shapes, ranks, slot-id structure
and value distributions each synthetic workload is meant to have."""
import numpy as np

from rank_adapter_apply_gb300 import workloads as wl


def _f32(w, a):
    return wl.bf16_bits_to_f32(a) if w.dtype == wl.DTYPE_BF16 else a


def test_zipf_probs():
    """Finite support: P(k) proportional to k^-s for k = 1..N (id k - 1)."""
    for n, s in ((8, 1.1), (32, 1.0), (512, 1.2)):
        p = wl.zipf_probs(n, s)
        assert p.shape == (n,) and abs(p.sum() - 1.0) < 1e-12
        k = np.arange(1, n + 1, dtype=np.float64)
        assert np.allclose(p / p[0], k ** -s, rtol=1e-12)


def test_tiny_fp32_recipe():
    w = wl.tiny_fp32(0)
    assert w.dtype == wl.DTYPE_F32 and (w.max_loras, w.max_lora_rank) == (4, 16)
    assert w.token_slot_idx.shape == (64,)
    assert set(np.unique(w.token_slot_idx)) <= {-1, 0, 1, 2, 3}
    assert np.all(w.ranks == 16) and np.all(w.alphas == 32.0)
    A, B = w.adapters[0]["proj"]
    assert A.shape == (16, 512) and B.shape == (512, 16)
    assert np.abs(A).max() <= 1 / np.sqrt(512)


def test_decode_recipe():
    w = wl.decode_qv_4096(0)
    idx = w.token_slot_idx
    assert idx.shape == (256,) and idx.min() >= -1 and idx.max() < 8
    base = float((idx < 0).mean())
    assert 0.03 < base < 0.2                          # 10 % base-only tokens
    counts = np.bincount(idx[idx >= 0], minlength=8)
    assert counts[0] == counts.max()                  # Zipf: slot 0 the most used
    assert [ly.name for ly in w.layers] == ["q_proj", "v_proj"]
    assert all(ly.d_in == 4096 and ly.d_out == 4096 and ly.x_key == "x" for ly in w.layers)
    assert np.all(w.ranks == 16) and np.all(w.alphas == 32.0)
    x = _f32(w, w.xs["x"])
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    A, B = w.adapters[3]["q_proj"]
    A, B = _f32(w, A), _f32(w, B)
    assert A.shape == (16, 4096) and B.shape == (4096, 16)
    assert np.abs(A).max() <= (1 / 64) * (1 + 2 ** -8)   # U(+-1/sqrt(d)), bf16 rounding
    assert abs(B.std() - 0.02) < 0.001


def test_prefill_recipe():
    w = wl.prefill_5120(0)
    lens, slots = w.meta["seq_lens"], w.meta["seq_slots"]
    assert len(lens) == 32 and min(lens) >= 128 and max(lens) <= 1024
    assert w.n_tokens == sum(lens)
    # tokens of a sequence are contiguous and share its slot
    assert np.array_equal(w.token_slot_idx, np.repeat(slots, lens))
    assert all(0 <= s < 16 for s in slots)
    assert [(ly.name, ly.d_in, ly.d_out, ly.x_key) for ly in w.layers] == [
        ("q_proj", 5120, 8192, "x"), ("k_proj", 5120, 1024, "x"), ("v_proj", 5120, 1024, "x"),
        ("o_proj", 8192, 5120, "attn")]
    assert np.all(w.ranks == 32) and np.all(w.alphas == 64.0) and w.max_lora_rank == 32


def test_mixed_ranks_recipe():
    w = wl.mixed_ranks_8b(0)
    idx = w.token_slot_idx
    assert idx.shape == (6 * 640 + 256,) and (w.max_loras, w.max_lora_rank) == (32, 64)
    for k, s in enumerate(w.meta["seg_slots"]):      # six prefill segments of 640 tokens
        assert np.all(idx[k * 640:(k + 1) * 640] == s)
    assert set(np.unique(w.ranks)) <= {8, 16, 32, 64}
    assert np.array_equal(w.alphas, 2.0 * w.ranks)   # alpha = 2r: scale 2
    names = [ly.name for ly in w.layers]
    assert names == ["q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj"]
    assert w.adapters[0]["down_proj"][0].shape == (int(w.ranks[0]), 14336)


def test_churn_trace_bursts():
    """Zipf(1.2) ids over 512 adapters; at steps 50, 100, 150 the last 20 tokens
    take 20 distinct ids not used in the 50 steps before, from the highest id
    down (at step 50 these are ids never used at all)."""
    t = wl.churn_trace(0)
    assert len(t.steps) == 200 and all(s.shape == (256,) for s in t.steps)
    for k in (50, 100, 150):
        recent = set(int(a) for ids in t.steps[k - 50:k] for a in ids)
        cold = [int(a) for a in t.steps[k][-20:]]
        assert len(set(cold)) == 20 and not (set(cold) & recent)
        assert cold == [a for a in range(511, -1, -1) if a not in recent][:20]
    never = set(int(a) for ids in t.steps[:50] for a in ids)
    assert not (set(int(a) for a in t.steps[50][-20:]) & never)
    first = np.concatenate(t.steps[:40])
    assert np.bincount(first, minlength=512)[0] == np.bincount(first, minlength=512).max()


def test_decode_recipe_other_ranks():
    """The decode recipe at another rank: every slot and max_lora_rank take it,
    alpha = 2 x rank (scale 2), the batch keeps its 256 tokens."""
    w16, w32 = wl.decode_qv_4096(0, direct_base=True), wl.decode_qv_4096(0, direct_base=True, rank=32)
    assert w32.max_lora_rank == 32 and np.all(w32.ranks == 32) and np.all(w32.alphas == 64.0)
    A, B = w32.adapters[5]["v_proj"]
    assert A.shape == (32, 4096) and B.shape == (4096, 32)
    assert w16.token_slot_idx.shape == w32.token_slot_idx.shape == (256,)
