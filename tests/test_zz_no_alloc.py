"""lora_apply_static_scratch: the delta of one layer for callers that cannot
allocate device memory (the scratch is a fixed array inside the library).
Its output must match lora_apply on the same inputs, on two calls in a row
(the second call finds the previous call's leftovers in the shared array),
and the fp64 oracle: with the usual tolerance, delta-only (base output 0),
and near the largest problem the array holds."""
import numpy as np
import pytest

from rank_adapter_apply_gb300 import workloads as wl
from tests.parity_util import TOL, check_delta, check_layer, decode, zero_base

pytestmark = pytest.mark.gpu


def _reference_and_static(w, layer_name):
    import torch
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300 import build
    from rank_adapter_apply_gb300.harness import DeviceWorkload, from_torch
    build.build()
    dw = DeviceWorkload(w)
    try:
        li = dw.layer_index[layer_name]
        ly = w.layers[li]
        # existing entry point (context + workspace)
        ref = dw.run([layer_name], multi=False)[layer_name]
        outs = []
        for _ in range(2):
            y = dw.y_in[layer_name].clone()
            torch.cuda.synchronize()
            s = dw.slots
            B.lora_apply_static_scratch(
                dw.xs[ly.x_key].data_ptr(), y.data_ptr(), dw.idx.data_ptr(), w.n_tokens,
                ly.d_in, ly.d_out, w.max_loras, w.max_lora_rank, s.cdtype, s.A[li].data_ptr(),
                s.B[li].data_ptr(), s.scale.data_ptr(), s.rank.data_ptr(), s.compute.cuda_stream)
            s.compute.synchronize()
            outs.append(from_torch(y))
    finally:
        dw.close()
    return ref, outs


def _close(w, got, ref):
    atol, rtol = TOL[w.dtype]
    g, r = decode(got, w.dtype), decode(ref, w.dtype)
    assert np.all(np.abs(g - r) <= atol + rtol * np.abs(r))


@pytest.mark.parametrize("make,layer", [
    (lambda: wl.decode_qv_4096(0), "q_proj"),
    (lambda: wl.mixed_ranks_8b(0, n_segments=1, seg_len=90, n_decode=50), "k_proj"),
    (lambda: wl.tiny_fp32(0), "proj"),
])
def test_static_scratch_matches_context_path(make, layer):
    w = make()
    ref, outs = _reference_and_static(w, layer)
    for got in outs:
        _close(w, got, ref)
    # base-only rows are untouched, bit for bit
    off = w.token_slot_idx < 0
    for got in outs:
        assert np.array_equal(got[off].view(np.uint8), w.ys[layer][off].view(np.uint8))


def test_static_scratch_rejects_oversize():
    import torch
    from rank_adapter_apply_gb300 import binding as B
    B.load()
    dev = torch.device("cuda:0")
    T, d = 9000, 64
    x = torch.zeros((T, d), dtype=torch.bfloat16, device=dev)
    y = torch.zeros((T, d), dtype=torch.bfloat16, device=dev)
    idx = torch.zeros(T, dtype=torch.int32, device=dev)
    A = torch.zeros((4, 64, d), dtype=torch.bfloat16, device=dev)
    Bp = torch.zeros((4, d, 64), dtype=torch.bfloat16, device=dev)
    sc = torch.zeros(4, dtype=torch.float32, device=dev)
    rk = torch.zeros(4, dtype=torch.int32, device=dev)
    with pytest.raises(B.LoraError) as ei:
        B.lora_apply_static_scratch(x.data_ptr(), y.data_ptr(), idx.data_ptr(), T, d, d, 4, 64,
                                    B.LORA_DTYPE_BF16, A.data_ptr(), Bp.data_ptr(), sc.data_ptr(),
                                    rk.data_ptr(), 0)
    assert ei.value.code == B.LORA_ERR_ARG and "static scratch" in str(ei.value)


def _static_only(w, layer_name, calls=2):
    """Outputs of `calls` static-scratch calls in a row (each from y_in)."""
    import torch
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300 import build
    from rank_adapter_apply_gb300.harness import DeviceWorkload, from_torch
    build.build()
    dw = DeviceWorkload(w)
    try:
        li = dw.layer_index[layer_name]
        ly = w.layers[li]
        s = dw.slots
        outs = []
        for _ in range(calls):
            y = dw.y_in[layer_name].clone()
            torch.cuda.synchronize()
            B.lora_apply_static_scratch(
                dw.xs[ly.x_key].data_ptr(), y.data_ptr(), dw.idx.data_ptr(), w.n_tokens,
                ly.d_in, ly.d_out, w.max_loras, w.max_lora_rank, s.cdtype, s.A[li].data_ptr(),
                s.B[li].data_ptr(), s.scale.data_ptr(), s.rank.data_ptr(), s.compute.cuda_stream)
            s.compute.synchronize()
            outs.append(from_torch(y))
    finally:
        dw.close()
    return outs


@pytest.mark.parametrize("make,layer", [
    (lambda: wl.decode_qv_4096(0), "q_proj"),
    (lambda: wl.mixed_ranks_8b(0, n_segments=1, seg_len=90, n_decode=50), "down_proj"),
    (lambda: wl.tiny_fp32(0), "proj"),
])
def test_static_scratch_matches_oracle(make, layer):
    w = make()
    for got in _static_only(w, layer):
        check_layer(w, layer, got)


def test_static_scratch_delta_only():
    """Base output 0: the static path's delta against the oracle's delta."""
    w = zero_base(wl.decode_qv_4096(0))
    for got in _static_only(w, "v_proj"):
        st = check_delta(w, "v_proj", got)
    print(f"delta[static_scratch] max_abs={st['max_abs']:.3e} max_rel={st['max_rel']:.3e} "
          f"max_abs/rms={st['max_abs_over_rms']:.3e} worst_ratio={st['worst_ratio']:.3f}")


def _near_limit(T, seed=4):
    rng = np.random.default_rng(seed)
    S, R = 8, 64
    ranks = np.array([8, 16, 32, 64, 64, 24, 48, 8], np.int32)
    layers = [wl.Layer("l0", 2048, 1024, "x")]
    adapters = [wl._adapter(rng, layers, int(ranks[s]), wl.DTYPE_BF16) for s in range(S)]
    idx = rng.integers(-1, S, size=T).astype(np.int32)
    x = wl._mat(rng, (T, 2048), "normal", 1.0, wl.DTYPE_BF16)
    y = wl._mat(rng, (T, 1024), "normal", 1.0, wl.DTYPE_BF16)
    return wl.Workload("near_limit", wl.DTYPE_BF16, S, R, layers, idx, {"x": x}, {"l0": y},
                       adapters, ranks, 2.0 * ranks)


def test_static_scratch_near_its_limit():
    """8,090 tokens at max_lora_rank 64: the partial rows are cut to what the
    4 MiB array holds (one d_in chunk per tile). Sampled tokens against the
    oracle; base-only rows bit for bit; 8,100 tokens no longer fit."""
    from rank_adapter_apply_gb300 import binding as B
    w = _near_limit(8090)
    rng = np.random.default_rng(1)
    tok = np.unique(np.concatenate([rng.choice(w.n_tokens, 500, replace=False), [0, w.n_tokens - 1]]))
    for got in _static_only(w, "l0"):
        check_layer(w, "l0", got, tokens=tok)
        off = w.token_slot_idx < 0
        assert np.array_equal(got[off].view(np.uint8), w.ys["l0"][off].view(np.uint8))
    with pytest.raises(B.LoraError) as ei:
        _static_only(_near_limit(8100), "l0", calls=1)
    assert ei.value.code == B.LORA_ERR_ARG


@pytest.mark.parametrize("dtype,R,d_in", [(wl.DTYPE_BF16, 24, 2048), (wl.DTYPE_BF16, 8, 2056),
                                          (wl.DTYPE_F32, 40, 1100)])
def test_static_scratch_ranks_between_block_sizes(dtype, R, d_in):
    """max_lora_rank not a multiple of 16 with d_in split into chunks: the
    static array's partial rows are whole 16-rank blocks long, so the split is
    capped at what its rows of R floats hold; sampled against the oracle."""
    from tests.test_gpu_parity import _custom
    T = 75
    rng = np.random.default_rng(R + d_in)
    ranks = [R, max(1, R // 2), 1, max(1, R - 3), 5]
    idx = rng.integers(-1, 5, size=T)
    w = _custom(T, d_in, 392, 5, R, ranks, idx, dtype=dtype, seed=R)
    for got in _static_only(w, "l0"):
        check_layer(w, "l0", got)
