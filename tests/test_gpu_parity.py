"""GPU parity: the CUDA path through the C ABI against the fp64 oracle."""
import numpy as np
import pytest

from rank_adapter_apply_gb300 import workloads as wl
from tests.parity_util import check_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from rank_adapter_apply_gb300 import build
    build.build()


def _run(w, multi=True, layers=None, **kw):
    from rank_adapter_apply_gb300.harness import DeviceWorkload
    dw = DeviceWorkload(w, **kw)
    try:
        out = dw.run(layers, multi=multi)
        stats = dw.slots.stats()
    finally:
        dw.close()
    return out, stats


def _custom(T, d_in, d_out, S, R, ranks, idx, dtype=wl.DTYPE_BF16, seed=0, empty=()):
    rng = np.random.default_rng(seed)
    layers = [wl.Layer("l0", d_in, d_out, "x")]
    adapters = []
    for s in range(S):
        if s in empty:
            adapters.append(None)
            continue
        adapters.append(wl._adapter(rng, layers, int(ranks[s]), dtype))
    x = wl._mat(rng, (T, d_in), "normal", 1.0, dtype)
    y = wl._mat(rng, (T, d_out), "normal", 1.0, dtype)
    rk = np.array([0 if s in empty else ranks[s] for s in range(S)], np.int32)
    return wl.Workload("custom", dtype, S, R, layers, np.asarray(idx, np.int32), {"x": x},
                       {"l0": y}, adapters, rk, 2.0 * np.maximum(rk, 1))


def test_tiny_fp32_full():
    w = wl.tiny_fp32(0)
    out, _ = _run(w)
    check_layer(w, "proj", out["proj"])


@pytest.mark.parametrize("multi", [True, False])
def test_decode_qv_4096_full(multi):
    w = wl.decode_qv_4096(0)
    out, st = _run(w, multi=multi)
    for ly in w.layers:
        check_layer(w, ly.name, out[ly.name])
    assert st["invalid_token_index"] == 0
    assert st["device_wait_timeouts"] == 0
    assert st["upload_bytes"] == 8 * 524_288


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 37])
def test_small_and_ragged_token_counts(T):
    rng = np.random.default_rng(T)
    idx = rng.integers(-1, 4, size=T)
    w = _custom(T, 256, 128, 4, 16, [16, 16, 16, 16], idx)
    out, _ = _run(w)
    check_layer(w, "l0", out["l0"])


@pytest.mark.parametrize("d_in,d_out,R,early", [(1032, 1000, 16, True), (1032, 1000, 16, False),
                                                  (4096, 4104, 16, True), (512, 4096, 32, True),
                                                  (768, 2056, 64, True), (768, 2056, 48, False)])
def test_cluster_decode_partial_stages(d_in, d_out, R, early):
    """Small-batch cluster kernel with column slices that end inside a stage:
    d_out up to 4096 takes the short path (products before the wait on the
    previous kernel, y updated from registers), d_out above 4096 the staged
    path; both with and without inputs declared ready."""
    from rank_adapter_apply_gb300.harness import DeviceWorkload
    from rank_adapter_apply_gb300 import binding as B
    T = 53
    rng = np.random.default_rng(d_in + d_out + R)
    S = 5
    ranks = [R, max(1, R // 2), 8, R, 5]
    idx = rng.integers(-1, S, size=T)
    w = _custom(T, d_in, d_out, S, R, ranks, idx, seed=d_out)
    dw = DeviceWorkload(w, small_batch_tokens=1024)       # the cluster kernel at every rank
    try:
        B.lora_set_inputs_ready(dw.slots.ctx, early)
        out = dw.run(None, multi=True)
    finally:
        dw.close()
    check_layer(w, "l0", out["l0"])


@pytest.mark.parametrize("T,S,one_slot", [(1024, 40, False), (1025, 40, False), (1024, 8, True)])
def test_small_batch_limits(T, S, one_slot):
    """The cluster path at its largest batch (1024 tokens) and one token past it
    (general path), with more than 32 slots (the tile prefix runs through shared
    memory) or every token on one slot (64 tiles of one slot)."""
    rng = np.random.default_rng(T + S)
    R = 32
    ranks = [int(rng.choice([8, 16, 24, 32])) for _ in range(S)]
    if one_slot:
        idx = np.full(T, 3, np.int32)
    else:
        idx = rng.integers(-1, S, size=T).astype(np.int32)
    w = _custom(T, 512, 256, S, R, ranks, idx, seed=T + 1)
    out, st = _run(w, small_batch_tokens=1024)            # the cluster kernel up to 1024 tokens at rank 32
    check_layer(w, "l0", out["l0"])
    assert st["device_wait_timeouts"] == 0


def test_small_batch_limit_follows_rank():
    """Without an explicit limit, rank 64 pools send small batches to the
    grouped kernels, rank 32 pools batches up to 768 tokens and rank 16 pools
    batches up to 1024 tokens to the cluster kernel."""
    from rank_adapter_apply_gb300.harness import DeviceWorkload
    for R, T, grouped, prefill_min in ((16, 64, False, None), (64, 64, True, None), (32, 768, False, None),
                                       (32, 769, True, None), (64, 64, True, 0)):
        rng = np.random.default_rng(R + T)
        idx = rng.integers(0, 4, size=T)
        w = _custom(T, 512, 256, 4, R, [R] * 4, idx, seed=R)
        dw = DeviceWorkload(w, prefill_min_tokens=prefill_min)
        try:
            out = dw.run(None, multi=True)
            check_layer(w, "l0", out["l0"])
            st = dw.slots.stats()
        finally:
            dw.close()
        assert (st["grouped_applies"], st["cluster_applies"]) == ((1, 0) if grouped else (0, 1)), (R, T, st)
        # four slot uploads (one kernel each), then one cluster kernel, or the
        # grouping, decode shrink and decode expand kernels plus two or three
        # prefill kernels when the batch reaches the prefill threshold (64
        # tokens by default; 0 turns the prefill kernels off)
        if not grouped:
            expect = {1}
        elif prefill_min == 0:
            expect = {3}
        else:
            expect = {5, 6}
        assert st["kernel_launches"] - 4 in expect, (R, T, prefill_min, st)


def test_all_base_only_is_bitwise_noop():
    T = 64
    w = _custom(T, 512, 256, 4, 16, [16] * 4, np.full(T, -1))
    w.ys["l0"][0, :8] = 0x8000          # -0.0 in bf16
    out, _ = _run(w)
    assert np.array_equal(out["l0"], w.ys["l0"])


def test_unaligned_dims_and_small_ranks():
    """d_in, d_out not multiples of 8 (scalar tails), ranks below 8 and odd."""
    T = 45
    rng = np.random.default_rng(7)
    idx = rng.integers(-1, 3, size=T)
    w = _custom(T, 203, 37, 3, 16, [3, 1, 13], idx)
    out, _ = _run(w)
    check_layer(w, "l0", out["l0"])


def test_fp32_unaligned():
    T = 23
    rng = np.random.default_rng(8)
    idx = rng.integers(-1, 3, size=T)
    w = _custom(T, 77, 53, 3, 24, [24, 5, 17], idx, dtype=wl.DTYPE_F32)
    out, _ = _run(w)
    check_layer(w, "l0", out["l0"])


def test_empty_slot_and_invalid_indices():
    T = 40
    idx = np.array(([0, 1, 2, 3, 7, -5, -1, 1] * 5)[:T])   # slot 2 empty; 7 and -5 invalid
    w = _custom(T, 256, 256, 4, 16, [16, 8, 16, 16], idx, empty=(2,))
    out, st = _run(w)
    check_layer(w, "l0", out["l0"])
    assert st["invalid_token_index"] == 10


@pytest.mark.parametrize("how", ["evict", "abort"])
def test_emptied_slot_reads_as_empty_on_the_device(how):
    """A slot emptied after its upload -- lora_evict_lru of the least recently
    used slot, or lora_abort_load of a chosen one -- reads as empty on the
    device: its tokens come back bit for bit, and the others match the oracle
    given the same slot as empty."""
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300.harness import DeviceWorkload
    T = 40
    idx = np.array(([0, 1, 2, 3, -1] * 8)[:T])
    w = _custom(T, 256, 256, 4, 16, [16, 8, 16, 16], idx)
    dw = DeviceWorkload(w)
    try:
        ctx = dw.slots.ctx
        for a in range(4):                       # bind ids 100..103 to slots 0..3, in that order
            assert B.lora_assign(ctx, 100 + a, int(w.ranks[a])) == (0, a, 1, -1)
        if how == "evict":
            assert B.lora_evict_lru(ctx) == (0, 0, 100)
            gone = 0
        else:
            assert B.lora_abort_load(ctx, 2) == (0, 102)
            gone = 2
        out = dw.run(None, multi=True)
    finally:
        dw.close()
    adapters = [None if s == gone else a for s, a in enumerate(w.adapters)]
    ranks = np.where(np.arange(4) == gone, 0, w.ranks).astype(np.int32)
    w_gone = wl.Workload("custom", w.dtype, w.max_loras, w.max_lora_rank, w.layers, w.token_slot_idx,
                         w.xs, w.ys, adapters, ranks, w.alphas)
    check_layer(w_gone, "l0", out["l0"])
    assert np.array_equal(out["l0"][idx == gone].view(np.uint8), w.ys["l0"][idx == gone].view(np.uint8))


@pytest.mark.parametrize("small_batch", [None, 1024])
def test_max_rank_64_mixed(small_batch):
    """max_lora_rank 64: the grouped kernels by default, the cluster kernel
    when the caller asks for it."""
    T = 96
    rng = np.random.default_rng(9)
    ranks = [8, 16, 32, 64, 48, 24]
    idx = rng.integers(0, 6, size=T)
    w = _custom(T, 1024, 512, 6, 64, ranks, idx)
    out, _ = _run(w, small_batch_tokens=small_batch)
    check_layer(w, "l0", out["l0"])


@pytest.mark.parametrize("small_batch", [0, 1024])
@pytest.mark.parametrize("R", [8, 24, 56])
def test_bf16_max_ranks_between_block_sizes(R, small_batch):
    """bf16 max_lora_rank 8, 24 and 56: B pools in blocks of 8 ranks, decode
    rows padded to whole 16-rank blocks, and (cluster kernel) MMA rank blocks
    of 16, 32 and 64 that reach past max_lora_rank; slot ranks from 1 to R on
    the grouped kernels (small_batch 0, d_in split into 5-9 chunks whose
    partial rows hold R ranks) and on the cluster kernel. d_in 2048 takes the
    grouped shrink's loop for whole 32-column steps, 2056 the other one."""
    T = 75
    rng = np.random.default_rng(R * 7 + small_batch)
    ranks = [R, max(1, R // 2), 1, max(1, R - 3), 5]
    idx = rng.integers(-1, 5, size=T)
    d_in = {8: 2056, 24: 2048, 56: 2056}[R]
    w = _custom(T, d_in, 392, 5, R, ranks, idx, seed=R + 11)
    out, st = _run(w, small_batch_tokens=small_batch)
    check_layer(w, "l0", out["l0"])
    if small_batch:
        assert st["cluster_applies"] >= 1 and st["grouped_applies"] == 0
    else:
        assert st["cluster_applies"] == 0 and st["grouped_applies"] >= 1


@pytest.mark.parametrize("R", [256, 200])
def test_fp32_largest_ranks(R):
    """fp32 takes max_lora_rank up to 256: the grouped kernels at 256 (B in
    blocks of 32 ranks) and at 200 (blocks of 8), slot ranks from 1 to R,
    d_in split into several chunks, ragged tails of tokens and columns."""
    T = 70
    rng = np.random.default_rng(R + 1)
    ranks = [R, 1, 130, 17, 64]
    idx = rng.integers(-1, 5, size=T)
    w = _custom(T, 1100, 300, 5, R, ranks, idx, dtype=wl.DTYPE_F32, seed=R)
    out, _ = _run(w)
    check_layer(w, "l0", out["l0"])


def _runs_over_slots(rng, T, S, long_p):
    """Slot ids as runs: with probability long_p a run of 64-200 tokens, else
    1-8 tokens; slots uniform over S, one in ten runs base-only."""
    idx = []
    while len(idx) < T:
        n = int(rng.integers(64, 201)) if rng.random() < long_p else int(rng.integers(1, 9))
        s = -1 if rng.random() < 0.1 else int(rng.integers(0, S))
        idx += [s] * n
    return np.array(idx[:T], np.int32)


@pytest.mark.parametrize("T,long_p", [(600, 0.0), (5000, 0.05)])
def test_max_loras_256(T, long_p):
    """max_loras at its limit (256 slots, every one bound): the cluster decode
    kernel takes at most 255 slots, so even a small batch takes the grouped
    kernels; a batch of two grouping blocks adds tensor-core prefill runs."""
    S = 256
    rng = np.random.default_rng(T)
    ranks = rng.integers(1, 17, size=S)
    idx = _runs_over_slots(rng, T, S, long_p)
    w = _custom(T, 256, 192, S, 16, ranks, idx, seed=5)
    out, st = _run(w)
    check_layer(w, "l0", out["l0"])
    assert st["cluster_applies"] == 0 and st["grouped_applies"] >= 1


@pytest.mark.parametrize("R,small_batch", [(48, 0), (48, 1024), (40, 0)])
def test_rank_blocked_pools_of_16_and_8(R, small_batch):
    """max_lora_rank 48 keeps B in three blocks of 16 ranks and 40 in five blocks
    of 8: the grouped kernels (small_batch 0) and the cluster kernel read only
    the blocks a slot's rank covers, ranks of every size inside them."""
    T = 80
    rng = np.random.default_rng(R)
    ranks = [R, 20, 8, 33, 16, 1]
    idx = rng.integers(-1, 6, size=T)
    w = _custom(T, 640, 384, 6, R, ranks, idx, seed=R + 3)
    out, _ = _run(w, small_batch_tokens=small_batch)
    check_layer(w, "l0", out["l0"])


def test_prefill_small_full():
    w = wl.prefill_5120(0, n_seqs=4, len_range=(5, 150))
    out, _ = _run(w)
    for ly in w.layers:
        check_layer(w, ly.name, out[ly.name])


def test_mixed_ranks_small_full():
    w = wl.mixed_ranks_8b(0, n_segments=2, seg_len=70, n_decode=40)
    out, _ = _run(w)
    for ly in w.layers:
        check_layer(w, ly.name, out[ly.name])


def _sample(w, n, seed=0):
    rng = np.random.default_rng(seed)
    tok = rng.choice(w.n_tokens, size=min(n, w.n_tokens), replace=False)
    # always include both ends and some segment boundaries
    return np.unique(np.concatenate([tok, [0, w.n_tokens - 1]]))


def test_prefill_full_size_sampled():
    w = wl.prefill_5120(0)
    out, _ = _run(w)
    tok = _sample(w, 160)
    for ly in w.layers:
        check_layer(w, ly.name, out[ly.name], tokens=tok)


def test_mixed_ranks_full_size_sampled():
    w = wl.mixed_ranks_8b(0)
    out, _ = _run(w)
    tok = _sample(w, 120)
    for ly in w.layers:
        check_layer(w, ly.name, out[ly.name], tokens=tok)


def test_fused_repeated_calls_and_layer_subsets():
    """Many launches on one context (epoch-tagged flags), single layers and the
    pair, each checked against the oracle after applying once more."""
    from rank_adapter_apply_gb300.harness import DeviceWorkload
    w = wl.decode_qv_4096(3, n_tokens=200)
    dw = DeviceWorkload(w)
    try:
        for rep in range(5):
            dw.reset()
            out = dw.run(["v_proj"] if rep % 2 else None, multi=rep < 3)
            for name, y in out.items():
                check_layer(w, name, y)
        st = dw.slots.stats()
        assert st["device_wait_timeouts"] == 0
    finally:
        dw.close()


@pytest.mark.parametrize("R", [16, 32, 64])
def test_tensor_core_prefill_small(R):
    """Runs of >= 64 same-slot tokens through the tcgen05 prefill kernel (general
    path forced), ragged run ends, decode tokens mixed in, ranks below R."""
    rng = np.random.default_rng(R)
    runs = [(0, 200), (2, 64), (1, 63), (3, 130), (-1, 40), (2, 129), (0, 7), (1, 300)]
    idx = np.concatenate([np.full(n, s) for s, n in runs]).astype(np.int32)
    ranks = [R, max(1, R // 2), R, 8 if R > 8 else R]
    w = _custom(idx.shape[0], 512, 384, 4, R, ranks, idx, seed=R)
    out, st = _run(w, small_batch_tokens=0)
    check_layer(w, "l0", out["l0"])
    assert st["device_wait_timeouts"] == 0


@pytest.mark.parametrize("R", [32, 64])
def test_tensor_core_prefill_ragged_dims(R):
    """d_in not a multiple of the 64-column k-block (the last TMA box of x and A
    reaches past the row and reads zeros) and d_out a multiple of 64 but not of
    the 128-column n-block; decode tokens of the same batch take the general
    path with a d_in chunk that ends inside a 32-column step."""
    rng = np.random.default_rng(R + 1)
    runs = [(1, 150), (0, 64), (-1, 9), (2, 70), (3, 5), (0, 200), (1, 3)]
    idx = np.concatenate([np.full(n, s) for s, n in runs]).astype(np.int32)
    ranks = [R, 8, R // 2, 5]
    w = _custom(idx.shape[0], 1032, 448, 4, R, ranks, idx, seed=R + 7)
    out, st = _run(w, small_batch_tokens=0)
    check_layer(w, "l0", out["l0"])
    assert st["device_wait_timeouts"] == 0


@pytest.mark.parametrize("R", [16, 64])
def test_tensor_core_prefill_short_runs(R):
    """Threshold 32: runs of 32-63 tokens take the tensor-core prefill path
    (a single ragged tile each), shorter ones the decode kernels."""
    rng = np.random.default_rng(R + 3)
    runs = [(0, 32), (1, 33), (2, 31), (3, 47), (-1, 5), (1, 63), (0, 64), (2, 40), (3, 1), (1, 32)]
    idx = np.concatenate([np.full(n, s) for s, n in runs]).astype(np.int32)
    ranks = [R, max(8, R // 2), 8, R]
    w = _custom(idx.shape[0], 512, 384, 4, R, ranks, idx, seed=R + 5)
    out, st = _run(w, small_batch_tokens=0, prefill_min_tokens=32)
    check_layer(w, "l0", out["l0"])
    assert st["device_wait_timeouts"] == 0


def test_prefill_small_general_path_matches_oracle():
    w = wl.prefill_5120(1, n_seqs=5, len_range=(60, 300))
    out, st = _run(w, small_batch_tokens=0)
    for ly in w.layers:
        check_layer(w, ly.name, out[ly.name])
    assert st["device_wait_timeouts"] == 0


def test_prefill_disabled_matches_oracle():
    w = wl.prefill_5120(2, n_seqs=3, len_range=(100, 200))
    out, _ = _run(w, small_batch_tokens=0, prefill_min_tokens=0)
    for ly in w.layers:
        check_layer(w, ly.name, out[ly.name])


def test_inputs_ready_back_to_back():
    """Early input loads: several applies in a row on one context with
    lora_set_inputs_ready, the second layer's y depending on nothing else."""
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300.harness import DeviceWorkload
    w = wl.decode_qv_4096(5)
    dw = DeviceWorkload(w)
    try:
        B.lora_set_inputs_ready(dw.slots.ctx, True)
        for rep in range(3):
            dw.reset()
            out = dw.run(["q_proj"], multi=False)
            out.update(dw.run(["v_proj"], multi=False))
            for name, y in out.items():
                check_layer(w, name, y)
        assert dw.slots.stats()["device_wait_timeouts"] == 0
    finally:
        dw.close()


def test_graph_replay_in_bench_launch_configuration():
    """The decode step as the benchmark times it: inputs declared ready
    (programmatic dependent launch), three steps on their own x, y and slot ids
    captured back to back in one CUDA graph. After a replay every step matches
    the oracle, and a second replay from the same inputs gives the same bits."""
    import torch
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300.harness import DeviceWorkload, from_torch, to_torch
    w = wl.decode_qv_4096(21, direct_base=True)
    dw = DeviceWorkload(w)
    try:
        B.lora_set_inputs_ready(dw.slots.ctx, True)
        dev = dw.device
        steps = []
        for k in range(3):
            x, ys, idx = wl.decode_batch(np.random.default_rng(300 + k), w.n_tokens, w.max_loras, True)
            wk = wl.Workload("decode_qv_4096", w.dtype, w.max_loras, w.max_lora_rank, w.layers, idx,
                             {"x": x}, ys, w.adapters, w.ranks, w.alphas)
            steps.append((wk, to_torch(x, w.dtype).to(dev),
                          {n: to_torch(ys[n], w.dtype).to(dev) for n in ys},
                          {n: to_torch(ys[n], w.dtype).to(dev) for n in ys},
                          torch.from_numpy(idx).to(dev)))
        st = dw.slots.compute

        def apply(step):
            _, xd, _, yd, idd = step
            dw.slots.apply_multi([0, 1], [xd, xd], [yd["q_proj"], yd["v_proj"]], idd)

        def reset():
            for _, _, y0, yd, _ in steps:
                for n in yd:
                    yd[n].copy_(y0[n])
            torch.cuda.synchronize(dev)

        with torch.cuda.stream(st):
            apply(steps[0])                 # eager call first: uploads are waited for outside the graph
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for step in steps:
                apply(step)
        outs = []
        for _ in range(2):
            reset()
            with torch.cuda.stream(st):
                g.replay()
            st.synchronize()
            outs.append([{n: from_torch(yd[n]) for n in yd} for _, _, _, yd, _ in steps])
        for (wk, *_), out in zip(steps, outs[0]):
            for n, y in out.items():
                check_layer(wk, n, y)
        for a, b in zip(outs[0], outs[1]):
            for n in a:
                assert np.array_equal(a[n], b[n]), n
        assert dw.slots.stats()["device_wait_timeouts"] == 0
    finally:
        dw.close()


def test_mixed_ranks_small_general_path():
    """Five layers reading one input at max_lora_rank 64: the shrink splits
    them into input groups of at most four, each x tile read once per group."""
    w = wl.mixed_ranks_8b(1, n_segments=3, seg_len=150, n_decode=50)
    out, st = _run(w, small_batch_tokens=0)
    for ly in w.layers:
        check_layer(w, ly.name, out[ly.name])
    assert st["device_wait_timeouts"] == 0


@pytest.mark.parametrize("T,run", [(100, 100), (90, 70), (129, 129)])
def test_prefill_batch_shorter_than_a_tile(T, run):
    """Fewer tokens than one 128-row tile (the TMA boxes reach past the last
    row), and a run ending one row into a second tile."""
    idx = np.concatenate([np.full(run, 1), np.full(T - run, 0)]).astype(np.int32)
    w = _custom(T, 320, 192, 2, 32, [32, 16], idx, seed=T)
    out, st = _run(w, small_batch_tokens=0)
    check_layer(w, "l0", out["l0"])
    assert st["device_wait_timeouts"] == 0


@pytest.mark.parametrize("dtype", [wl.DTYPE_BF16, wl.DTYPE_F32])
def test_batched_upload_matches_oracle(dtype):
    """lora_load_slots: adapters of several ranks (zero padding up to R) in one
    call, pinned buffers read by the upload kernel plus one pageable adapter
    (read by the kernel too where the GPU walks the host's page tables, else
    taken by the copy-engine path); then the delta equals the oracle's,
    padding rows of a slot that held a larger rank before are zero again, and
    every slot's B sits in the pool's rank-blocked layout bit for bit."""
    import torch
    from rank_adapter_apply_gb300.harness import to_torch, from_torch
    from rank_adapter_apply_gb300.slots import LoraSlots
    rng = np.random.default_rng(11)
    T, d_in, d_out, S, R = 96, 512, 384, 5, 32
    ranks = [32, 8, 16, 24, 32]
    layers = [wl.Layer("l0", d_in, d_out, "x")]
    ads = [wl._adapter(rng, layers, r, dtype) for r in ranks]
    idx = rng.integers(-1, S, size=T).astype(np.int32)
    x = wl._mat(rng, (T, d_in), "normal", 1.0, dtype)
    y = wl._mat(rng, (T, d_out), "normal", 1.0, dtype)
    w = wl.Workload("custom", dtype, S, R, layers, idx, {"x": x}, {"l0": y}, ads,
                    np.array(ranks, np.int32), 2.0 * np.array(ranks, np.float64))
    tdt = torch.bfloat16 if dtype == wl.DTYPE_BF16 else torch.float32
    sl = LoraSlots([(d_in, d_out)], S, R, T, dtype=tdt, device="cuda:0")
    try:
        # slot 1 first holds a rank-32 adapter, so its padding must be cleared later
        big = wl._adapter(rng, layers, 32, dtype)
        sl.load_slot(1, [to_torch(big["l0"][0], dtype).pin_memory()],
                     [to_torch(big["l0"][1], dtype).pin_memory()], 32, 64.0)
        sl.sync_uploads()
        host = []
        for s in range(S):
            A = to_torch(ads[s]["l0"][0], dtype)
            Bm = to_torch(ads[s]["l0"][1], dtype)
            if s != 3:                                   # slot 3: pageable memory
                A, Bm = A.pin_memory(), Bm.pin_memory()
            host.append(([A], [Bm]))
        sl.load_slots(list(range(S)), host, ranks, [2.0 * r for r in ranks])
        sl.sync_uploads()
        st = sl.stats()
        assert st["uploads"] == S + 1
        assert st["upload_bytes"] == sum((d_in + d_out) * r for r in [32] + ranks) * (2 if dtype == wl.DTYPE_BF16 else 4)
        xd = to_torch(x, dtype).to("cuda:0")
        yd = to_torch(y, dtype).to("cuda:0")
        sl.apply(0, xd, yd, torch.from_numpy(idx).to("cuda:0"))
        torch.cuda.synchronize()
        check_layer(w, "l0", from_torch(yd))
        A_pool = from_torch(sl.A[0])
        B_pool = from_torch(sl.B[0])
        assert not A_pool[1, 8:].any()                   # rank 8 now: rows 8..31 zero again
        # B pool of a slot: blocks of kb ranks, each [d_out][kb] (kb = 32 at
        # max_lora_rank 32: the plain [d_out][R] layout)
        kb = 32 if R % 32 == 0 else (16 if R % 16 == 0 else 8)
        for s in range(S):
            Bs = B_pool[s].reshape(R // kb, d_out, kb).transpose(1, 0, 2).reshape(d_out, R)
            r = ranks[s]
            assert np.array_equal(Bs[:, :r].view(np.uint8), np.ascontiguousarray(ads[s]["l0"][1]).view(np.uint8))
            assert not Bs[:, r:].any()
    finally:
        sl.close()


@pytest.mark.parametrize("name", ["decode", "prefill", "mixed"])
def test_repeated_runs_are_bitwise_identical(name):
    """Every reduction (d_in chunks, cluster partials, prefill chunk sums) adds in
    a fixed order, so the same inputs give the same bits on every run."""
    from rank_adapter_apply_gb300.harness import DeviceWorkload
    w = {"decode": lambda: wl.decode_qv_4096(4),
         "prefill": lambda: wl.prefill_5120(3, n_seqs=6, len_range=(100, 700)),
         "mixed": lambda: wl.mixed_ranks_8b(2, n_segments=3, seg_len=300, n_decode=200)}[name]()
    dw = DeviceWorkload(w, small_batch_tokens=None if name == "decode" else 0)
    try:
        outs = []
        for _ in range(3):
            dw.reset()
            outs.append(dw.run())
        for ly in w.layers:
            for o in outs[1:]:
                assert np.array_equal(o[ly.name], outs[0][ly.name]), ly.name
        check_layer(w, w.layers[0].name, outs[0][w.layers[0].name])
    finally:
        dw.close()


def test_batched_upload_rejects_bad_arguments():
    import torch
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300.slots import LoraSlots
    sl = LoraSlots([(64, 64)], 4, 16, 8, dtype=torch.bfloat16, device="cuda:0")
    try:
        a = torch.zeros((16, 64), dtype=torch.bfloat16).pin_memory()
        b = torch.zeros((64, 16), dtype=torch.bfloat16).pin_memory()
        for slots, ranks in (([0, 0], [16, 16]), ([4], [16]), ([1], [32]), ([1], [0])):
            with pytest.raises(B.LoraError):
                sl.load_slots(slots, [([a], [b])] * len(slots), ranks, [32.0] * len(slots))
        assert sl.stats()["uploads"] == 0          # nothing was queued
    finally:
        sl.close()


def _packed_bytes(T, d, dv):
    return T * 4 + T * d * 2 * 2 + T * dv * 2


def _packed_views(buf, T, d, dv):
    """idx | x | y_q | y_v back to back in one byte buffer."""
    import torch
    o1, o2 = T * 4, T * 4 + T * d * 2
    o3 = o2 + T * d * 2
    return (buf[:o1].view(torch.int32), buf[o1:o2].view(torch.bfloat16).view(T, d),
            [buf[o2:o3].view(torch.bfloat16).view(T, d), buf[o3:o3 + T * dv * 2].view(torch.bfloat16).view(T, dv)])


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("device_sets", [1, 2])
def test_host_buffer_path_matches_oracle(device_sets, packed):
    """lora_apply_multi_host, several calls queued back to back: copies in on
    the upload stream ordered per device buffer, apply and copies back on the
    compute stream. With one device buffer set the calls serialise, with two
    they overlap; with packed buffers (idx | x | y_q | y_v back to back on both
    sides) the copies each way are merged into one. Every call's result equals
    the oracle's."""
    import torch
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300.harness import to_torch
    from rank_adapter_apply_gb300.slots import LoraSlots
    rng = np.random.default_rng(21)
    S, R, T, d, dv = 4, 16, 96, 512, 384
    layers = [wl.Layer("q", d, d, "x"), wl.Layer("v", d, dv, "x")]
    ranks = np.array([16, 8, 16, 12], np.int32)
    ads = [wl._adapter(rng, layers, int(r), wl.DTYPE_BF16) for r in ranks]
    sl = LoraSlots([(d, d), (d, dv)], S, R, T, dtype=torch.bfloat16, device="cuda:0")
    try:
        for s in range(S):
            sl.load_slot(s, [to_torch(ads[s][l.name][0], wl.DTYPE_BF16).pin_memory() for l in layers],
                         [to_torch(ads[s][l.name][1], wl.DTYPE_BF16).pin_memory() for l in layers],
                         int(ranks[s]), 2.0 * float(ranks[s]))
        sl.sync_uploads()
        batches = []
        for k in range(6):
            x = wl._mat(rng, (T, d), "normal", 1.0, wl.DTYPE_BF16)
            ys = {"q": wl._mat(rng, (T, d), "normal", 1.0, wl.DTYPE_BF16),
                  "v": wl._mat(rng, (T, dv), "normal", 1.0, wl.DTYPE_BF16)}
            idx = rng.integers(-1, S, size=T).astype(np.int32)
            if packed:
                hidx, hx, hy = _packed_views(torch.empty(_packed_bytes(T, d, dv), dtype=torch.uint8).pin_memory(),
                                             T, d, dv)
                hidx.copy_(torch.from_numpy(idx))
                hx.copy_(to_torch(x, wl.DTYPE_BF16))
                for t, n in zip(hy, ("q", "v")):
                    t.copy_(to_torch(ys[n], wl.DTYPE_BF16))
            else:
                hx = to_torch(x, wl.DTYPE_BF16).pin_memory()
                hy = [to_torch(ys[n], wl.DTYPE_BF16).clone().pin_memory() for n in ("q", "v")]
                hidx = torch.from_numpy(idx).pin_memory()
            batches.append((x, ys, idx, hx, hy, hidx))
        if packed:
            dev_sets = []
            for _ in range(device_sets):
                di, dx, dy = _packed_views(torch.empty(_packed_bytes(T, d, dv), dtype=torch.uint8, device="cuda:0"),
                                           T, d, dv)
                dev_sets.append((dx, dy, di))
        else:
            dev_sets = [(torch.empty((T, d), dtype=torch.bfloat16, device="cuda:0"),
                         [torch.empty((T, d), dtype=torch.bfloat16, device="cuda:0"),
                          torch.empty((T, dv), dtype=torch.bfloat16, device="cuda:0")],
                         torch.empty(T, dtype=torch.int32, device="cuda:0")) for _ in range(device_sets)]
        for k, (_, _, _, hx, hy, hidx) in enumerate(batches):
            xd, yd, idd = dev_sets[k % device_sets]
            B.lora_apply_multi_host(sl.ctx, [0, 1], [hx.data_ptr()] * 2, [t.data_ptr() for t in hy],
                                    hidx.data_ptr(), T, [xd.data_ptr()] * 2, [t.data_ptr() for t in yd],
                                    idd.data_ptr())
        B.lora_sync_host(sl.ctx)
        for x, ys, idx, hx, hy, hidx in batches:
            w = wl.Workload("custom", wl.DTYPE_BF16, S, R, layers, idx, {"x": x}, ys, ads, ranks,
                            2.0 * ranks.astype(np.float64))
            for name, t in zip(("q", "v"), hy):
                check_layer(w, name, t.view(torch.int16).numpy().view(np.uint16))
    finally:
        sl.close()


@pytest.mark.parametrize("T,prefill_min", [(40000, None), (40000, 0), (18000, None), (18000, 0), (8193, None)])
def test_grouping_across_blocks(T, prefill_min):
    """The grouping kernel splits a batch into G = ceil(T / 4096) blocks of one
    CTA each (block c from token T*c/G), exchanging per-block figures through a
    cluster's shared memory for G <= 8 (8,193 and 18,000 tokens) and through
    the workspace at grid barriers beyond (40,000 tokens). Long runs that cross
    the block edges (tensor-core prefill tiles, or decode tiles when the
    prefill path is off), short decode runs, base-only tokens and out-of-range
    indices next to the edges; sampled tokens (every edge among them) against
    the oracle, base-only and invalid rows bit for bit, the invalid count
    exact."""
    rng = np.random.default_rng(40)
    G = (T + 4095) // 4096
    edges = [T * c // G for c in range(1, G)]
    parts, n = [], 0
    while n < T:
        kind = rng.random()
        if kind < 0.3:
            ln, s = int(rng.integers(100, 3000)), int(rng.integers(0, 12))
        elif kind < 0.9:
            ln, s = int(rng.integers(1, 40)), int(rng.integers(-1, 12))
        else:
            ln, s = int(rng.integers(1, 5)), int(rng.choice([12, 99, -7]))
        parts.append(np.full(ln, s))
        n += ln
    idx = np.concatenate(parts)[:T].astype(np.int32)
    # one run straight across each edge, with an invalid index and a base-only
    # token right after the first edge
    for e in edges:
        idx[e - 700:e + 900] = 5
    idx[edges[0] + 901] = 99
    idx[edges[0] + 902] = -1
    w = _custom(T, 256, 192, 12, 16, [16, 8, 16, 12, 16, 16, 8, 16, 16, 4, 16, 16], idx, seed=41)
    out, st = _run(w, prefill_min_tokens=prefill_min)
    near = np.concatenate([np.arange(e - 3, e + 4) for e in edges] + [[0, T - 1, edges[0] + 901, edges[0] + 902]])
    tok = np.unique(np.concatenate([_sample(w, 600, seed=3), near]))
    check_layer(w, "l0", out["l0"], tokens=tok)
    assert st["invalid_token_index"] == int(((idx < -1) | (idx >= 12)).sum())
    assert st["device_wait_timeouts"] == 0
