"""Pins for the fp64 oracle: each test checks it against something other than
itself (a worked example, exact integer arithmetic, a library matmul, a closed
form or an invariant), chosen so that a dropped term, a wrong sign or index, or
a transposed operand fails at least one of them."""
import os

import numpy as np
import pytest

import oracle
from oracle import lora_apply_ref, F32, BF16
from rank_adapter_apply_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            vals[k] = [float(a) for a in v]
    return vals


def _int_case(rng, T, d_in, d_out, S, R, ranks, lo=-3, hi=4):
    """Small-integer fp32 inputs: every product and partial sum is exact."""
    x = rng.integers(lo, hi, size=(T, d_in)).astype(np.float32)
    A = np.zeros((S, R, d_in), np.float32)
    B = np.zeros((S, d_out, R), np.float32)
    for s in range(S):
        r = ranks[s]
        A[s, :r] = rng.integers(lo, hi, size=(r, d_in))
        B[s, :, :r] = rng.integers(lo, hi, size=(d_out, r))
    return x, A, B


def test_golden_peft_example():
    g = _read_golden("peft_example_scale.txt")
    r, alpha = int(g["r"][0]), g["lora_alpha"][0]
    d_in, d_out = int(g["d_in"][0]), int(g["d_out"][0])
    A = np.zeros((1, r, d_in), np.float32)
    B = np.zeros((1, d_out, r), np.float32)
    A[0, 0], A[0, 1] = g["A0"], g["A1"]
    B[0, :, 0], B[0, :, 1] = g["Bcol0"], g["Bcol1"]
    x = np.array([g["x"]], np.float32)
    y = np.array([g["y_in"]], np.float32)
    out = lora_apply_ref(x, y, A, B, [r], [alpha], [0], dtype=F32)
    assert out[0].tolist() == g["y_out"]


def test_merged_weight_identity_exact():
    """y = W x and the delta path equal (W + (alpha/r) B A) x exactly when all
    values are small integers and alpha/r is a power of two."""
    rng = np.random.default_rng(1)
    T, d_in, d_out, S, R = 9, 13, 7, 3, 8
    ranks = [4, 2, 8]
    alphas = np.array([8.0, 1.0, 32.0])         # scales 2, 0.5, 4
    x, A, B = _int_case(rng, T, d_in, d_out, S, R, ranks)
    W = rng.integers(-3, 4, size=(d_out, d_in)).astype(np.float64)
    y_in = (x.astype(np.float64) @ W.T).astype(np.float32)
    idx = np.array([0, 1, 2, -1, 2, 0, 1, 1, -1], np.int32)
    out = lora_apply_ref(x, y_in, A, B, ranks, alphas, idx, dtype=F32)
    for t in range(T):
        s = idx[t]
        if s < 0:
            W_eff = W
        else:
            r = ranks[s]
            W_eff = W + (alphas[s] / r) * (B[s, :, :r].astype(np.float64) @ A[s, :r].astype(np.float64))
        np.testing.assert_array_equal(out[t], W_eff @ x[t].astype(np.float64))


def test_merged_weight_identity_random_bf16():
    rng = np.random.default_rng(2)
    T, d_in, d_out, S, R, r, alpha = 6, 40, 24, 2, 16, 16, 32.0
    x = wl.f32_to_bf16_bits(rng.standard_normal((T, d_in)).astype(np.float32))
    A = wl.f32_to_bf16_bits(rng.uniform(-0.2, 0.2, (S, R, d_in)).astype(np.float32))
    B = wl.f32_to_bf16_bits(rng.normal(0, 0.02, (S, d_out, R)).astype(np.float32))
    W = rng.normal(0, 0.02, (d_out, d_in))
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    y_in = wl.f32_to_bf16_bits((xf @ W.T).astype(np.float32))
    idx = np.array([0, 1, 1, 0, 1, 0], np.int32)
    out = lora_apply_ref(x, y_in, A, B, [r, r], [alpha, alpha], idx, dtype=BF16)
    Af = wl.bf16_bits_to_f32(A).astype(np.float64)
    Bf = wl.bf16_bits_to_f32(B).astype(np.float64)
    yf = wl.bf16_bits_to_f32(y_in).astype(np.float64)
    for t in range(T):
        s = idx[t]
        merged = (alpha / r) * (Bf[s] @ Af[s])
        ref = yf[t] + merged @ xf[t]
        np.testing.assert_allclose(out[t], ref, rtol=1e-12, atol=1e-14)


def test_library_reduction_single_slot():
    """All tokens on one slot: the result is y_in + s (X A^T) B^T."""
    rng = np.random.default_rng(3)
    T, d_in, d_out, R, r, alpha = 17, 64, 48, 16, 12, 24.0
    x = rng.standard_normal((T, d_in)).astype(np.float32)
    y = rng.standard_normal((T, d_out)).astype(np.float32)
    A = np.zeros((1, R, d_in), np.float32)
    B = np.zeros((1, d_out, R), np.float32)
    A[0, :r] = rng.uniform(-0.1, 0.1, (r, d_in))
    B[0, :, :r] = rng.normal(0, 0.02, (d_out, r))
    out = lora_apply_ref(x, y, A, B, [r], [alpha], np.zeros(T, np.int32), dtype=F32)
    X = x.astype(np.float64)
    ref = y.astype(np.float64) + (alpha / r) * ((X @ A[0, :r].T.astype(np.float64)) @ B[0, :, :r].T.astype(np.float64))
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_zero_B_and_minus_one_reproduce_base():
    w = wl.tiny_fp32(0)
    A, B = w.padded_pools("proj")
    out0 = lora_apply_ref(w.xs["x"], w.ys["proj"], A, np.zeros_like(B), w.ranks, w.alphas,
                          w.token_slot_idx, dtype=F32)
    np.testing.assert_array_equal(out0, w.ys["proj"].astype(np.float64))
    idx = np.full(w.n_tokens, -1, np.int32)
    out1 = lora_apply_ref(w.xs["x"], w.ys["proj"], A, B, w.ranks, w.alphas, idx, dtype=F32)
    np.testing.assert_array_equal(out1, w.ys["proj"].astype(np.float64))
    # -0.0 in y_in survives a base-only token bit for bit
    y = w.ys["proj"].copy()
    y[0, :5] = -0.0
    out2 = lora_apply_ref(w.xs["x"], y, A, B, w.ranks, w.alphas, idx, dtype=F32)
    assert np.all(np.signbit(out2[0, :5]))


def test_invalid_and_empty_slots_are_noops():
    rng = np.random.default_rng(4)
    x, A, B = _int_case(rng, 4, 8, 6, 2, 4, [4, 4])
    y = rng.standard_normal((4, 6)).astype(np.float32)
    idx = np.array([2, -7, 1, 0], np.int32)             # out of range, invalid, empty, valid
    out = lora_apply_ref(x, y, A, B, [4, 0], [8.0, 8.0], idx, dtype=F32)
    np.testing.assert_array_equal(out[:3], y[:3].astype(np.float64))
    assert not np.array_equal(out[3], y[3].astype(np.float64))


def test_rank_one_one_hot():
    """r = 1, A = e_i^T, B = e_j: delta[t][j] = alpha * x[t][i], zero elsewhere."""
    rng = np.random.default_rng(5)
    T, d_in, d_out, i, j, alpha = 5, 11, 9, 7, 3, 3.0
    x = rng.standard_normal((T, d_in)).astype(np.float32)
    y = np.zeros((T, d_out), np.float32)
    A = np.zeros((1, 1, d_in), np.float32)
    B = np.zeros((1, d_out, 1), np.float32)
    A[0, 0, i] = 1.0
    B[0, j, 0] = 1.0
    out = lora_apply_ref(x, y, A, B, [1], [alpha], np.zeros(T, np.int32), dtype=F32)
    ref = np.zeros((T, d_out))
    ref[:, j] = alpha * x[:, i].astype(np.float64)
    np.testing.assert_array_equal(out, ref)


def test_zero_padding_is_bit_exact():
    """Pools padded from rank r to max_lora_rank with zeros give the same bits
    as unpadded pools, whether the loop stops at r or runs over the padding."""
    w = wl.mixed_ranks_8b(0, n_segments=1, seg_len=4, n_decode=12)
    ly = w.layers[1]                                     # k_proj 4096 -> 1024
    A, B = w.padded_pools(ly.name)
    xs = w.xs[ly.x_key]
    base = lora_apply_ref(xs, w.ys[ly.name], A, B, w.ranks, w.alphas, w.token_slot_idx)
    padded_loop = lora_apply_ref(xs, w.ys[ly.name], A, B, w.ranks, w.alphas, w.token_slot_idx,
                                 loop_padded=True)
    np.testing.assert_array_equal(base, padded_loop)
    for t in range(w.n_tokens):
        s = int(w.token_slot_idx[t])
        r = int(w.ranks[s])
        a1 = A[s:s + 1, :r]
        b1 = B[s:s + 1, :, :r]
        one = lora_apply_ref(xs[t:t + 1], w.ys[ly.name][t:t + 1], a1, b1, [r],
                             [w.alphas[s]], [0])
        np.testing.assert_array_equal(one[0], base[t])


def test_scale_uses_true_rank_and_is_linear_in_alpha():
    rng = np.random.default_rng(6)
    T, d_in, d_out, R, r = 8, 32, 16, 64, 8
    x = rng.standard_normal((T, d_in)).astype(np.float32)
    y0 = np.zeros((T, d_out), np.float32)
    A = np.zeros((1, R, d_in), np.float32)
    B = np.zeros((1, d_out, R), np.float32)
    A[0, :r] = rng.uniform(-0.2, 0.2, (r, d_in))
    B[0, :, :r] = rng.normal(0, 0.02, (d_out, r))
    idx = np.zeros(T, np.int32)
    d1 = lora_apply_ref(x, y0, A, B, [r], [16.0], idx, dtype=F32)
    d2 = lora_apply_ref(x, y0, A, B, [r], [32.0], idx, dtype=F32)
    np.testing.assert_array_equal(d2, 2.0 * d1)
    # alpha / r with r the adapter's rank (8), not max_lora_rank (64)
    X = x.astype(np.float64)
    ref = (16.0 / r) * (X @ A[0, :r].T.astype(np.float64)) @ B[0, :, :r].T.astype(np.float64)
    np.testing.assert_allclose(d1, ref, rtol=1e-12, atol=1e-14)


def test_token_list_matches_whole_batch():
    """Invariant: the rows computed for a list of tokens (any order, repeats
    allowed) are the rows of those tokens in the whole-batch result."""
    rng = np.random.default_rng(7)
    T, d_in, d_out, S, R = 12, 10, 6, 3, 8
    x, A, B = _int_case(rng, T, d_in, d_out, S, R, [8, 3, 5])
    y = rng.integers(-5, 6, size=(T, d_out)).astype(np.float32)
    idx = np.array([2, 0, -1, 1, 1, 2, 0, -1, 2, 1, 0, 0], np.int32)
    whole = lora_apply_ref(x, y, A, B, [8, 3, 5], [16.0, 6.0, 5.0], idx, dtype=F32)
    tok = [9, 3, 3, 0, 11, 2, 6]
    part = lora_apply_ref(x, y, A, B, [8, 3, 5], [16.0, 6.0, 5.0], idx, tokens=tok, dtype=F32)
    np.testing.assert_array_equal(part, whole[tok])


def test_bf16_decoding_is_exact():
    v = np.array([1.0, -2.5, 3.140625, 1e-3, -0.0, 65504.0], np.float32)
    bits = wl.f32_to_bf16_bits(v)
    back = wl.bf16_bits_to_f32(bits)
    # values already representable in bf16 round-trip; 1e-3 rounds to nearest
    assert back[0] == 1.0 and back[1] == -2.5 and back[2] == 3.140625
    assert abs(back[3] - 1e-3) <= 2.0 ** -9 * 1e-3 * 2
    assert np.signbit(back[4])
    # the oracle reads bf16 bits and fp32 values identically
    A = wl.f32_to_bf16_bits(np.ones((1, 1, 6), np.float32))
    B = wl.f32_to_bf16_bits(np.ones((1, 1, 1), np.float32))
    y = wl.f32_to_bf16_bits(np.zeros((1, 1), np.float32))
    out = lora_apply_ref(bits[None, :], y, A, B, [1], [1.0], [0], dtype=BF16)
    assert out[0, 0] == float(back.astype(np.float64).sum())


@pytest.mark.parametrize("layers,rank,bpp,expected", [
    ([(4096, 4096), (4096, 4096)], 16, 2, 524_288),                       # decode q+v adapter
    ([(5120, 8192)], 32, 2, 851_968),
    ([(5120, 8192), (5120, 1024), (5120, 1024), (8192, 5120)], 32, 2, 2_490_368),
    ([(4096, 4096), (4096, 1024), (4096, 1024), (4096, 4096),
      (4096, 14336), (4096, 14336), (14336, 4096)], 64, 2, 10_485_760),
])
def test_adapter_bytes_formula(layers, rank, bpp, expected):
    assert oracle.adapter_bytes(layers, rank, bpp) == expected
    # the same count as the element count of A [r, d_in] plus B [d_out, r]
    assert expected == sum(rank * di * bpp + do * rank * bpp for di, do in layers)


def test_delta_bound_of_the_parity_helper():
    """The delta-only comparison accepts the oracle's own delta rounded once to
    bf16 (the one rounding the bound allows) and rejects a delta 1 % off, a
    delta of the wrong sign, and a changed base-only row."""
    from tests.parity_util import check_delta, zero_base
    w = zero_base(wl.decode_qv_4096(0, n_tokens=24))
    for ly in w.layers:
        A, B = w.padded_pools(ly.name)
        ref = oracle.lora_apply_ref(w.xs["x"], w.ys[ly.name], A, B, w.ranks, w.alphas, w.token_slot_idx)
        good = wl.f32_to_bf16_bits(ref.astype(np.float32))
        assert check_delta(w, ly.name, good)["worst_ratio"] <= 1.0
        for bad in (wl.f32_to_bf16_bits((ref * 1.01).astype(np.float32)),
                    wl.f32_to_bf16_bits((-ref).astype(np.float32))):
            with pytest.raises(AssertionError):
                check_delta(w, ly.name, bad)
        off = np.nonzero(w.token_slot_idx < 0)[0]
        changed = good.copy()
        changed[off[0], 0] = 0x3F80
        with pytest.raises(AssertionError):
            check_delta(w, ly.name, changed)
