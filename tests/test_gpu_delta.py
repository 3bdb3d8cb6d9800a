"""Delta-only parity: every path of the CUDA library run with base outputs
y_in = 0, so each output element is the rounded LoRA delta itself, compared
with the fp64 oracle's delta element by element (sampled tokens at the full
prefill and mixed-rank sizes). The bound, 2**-8 |o| + 2**-12 rms_t(o) per
element, is derived in tests/parity_util.py. Each test prints its error
statistics (max abs, max rel over elements not cancelled to ~0, max abs over
the token's rms, worst ratio to the bound)."""
import numpy as np
import pytest

from rank_adapter_apply_gb300 import workloads as wl
from tests.parity_util import check_delta, zero_base

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from rank_adapter_apply_gb300 import build
    build.build()


def _run(w, **kw):
    from rank_adapter_apply_gb300.harness import DeviceWorkload
    dw = DeviceWorkload(w, **kw)
    try:
        out = dw.run(None, multi=True)
        st = dw.slots.stats()
    finally:
        dw.close()
    assert st["device_wait_timeouts"] == 0
    return out, st


def _sample(w, n, seed=0):
    rng = np.random.default_rng(seed)
    tok = rng.choice(w.n_tokens, size=min(n, w.n_tokens), replace=False)
    return np.unique(np.concatenate([tok, [0, w.n_tokens - 1]]))


def _report(path, stats):
    worst = max(stats, key=lambda s: s["worst_ratio"])
    print(f"delta[{path}] max_abs={max(s['max_abs'] for s in stats):.3e} "
          f"max_rel={max(s['max_rel'] for s in stats):.3e} "
          f"max_abs/rms={max(s['max_abs_over_rms'] for s in stats):.3e} "
          f"worst_ratio={worst['worst_ratio']:.3f} ({worst['layer']})")


def test_delta_decode_cluster():
    """The single-launch cluster decode kernel (256 tokens, q_proj + v_proj)."""
    w = zero_base(wl.decode_qv_4096(0))
    out, st = _run(w)
    assert (st["cluster_applies"], st["grouped_applies"]) == (1, 0)
    _report("decode_cluster", [check_delta(w, ly.name, out[ly.name]) for ly in w.layers])


def test_delta_decode_grouped():
    """The grouping + decode shrink / expand kernels on the same batch."""
    w = zero_base(wl.decode_qv_4096(0))
    out, st = _run(w, small_batch_tokens=0, prefill_min_tokens=0)
    assert (st["cluster_applies"], st["grouped_applies"]) == (0, 1)
    _report("decode_grouped", [check_delta(w, ly.name, out[ly.name]) for ly in w.layers])


def test_delta_prefill_rank32_full_size():
    """The tcgen05 prefill shrink / expand at rank 32: the whole prefill
    workload (18,167 tokens, q/k/v/o), sampled tokens."""
    w = zero_base(wl.prefill_5120(0))
    out, _ = _run(w)
    tok = _sample(w, 400)
    _report("prefill_r32", [check_delta(w, ly.name, out[ly.name], tokens=tok) for ly in w.layers])


def test_delta_prefill_rank16():
    """The tcgen05 prefill path at rank 16: runs of 64..700 tokens over 8
    slots, q_proj / v_proj shapes (4096 -> 4096), some decode tokens."""
    rng = np.random.default_rng(16)
    lens = rng.integers(64, 700, size=8)
    slots = rng.integers(0, 8, size=8)
    idx = np.concatenate([np.repeat(slots, lens), rng.integers(-1, 8, size=40)]).astype(np.int32)
    layers = [wl.Layer("q_proj", 4096, 4096, "x"), wl.Layer("v_proj", 4096, 4096, "x")]
    adapters = [wl._adapter(rng, layers, 16, wl.DTYPE_BF16) for _ in range(8)]
    T = idx.shape[0]
    x = wl._mat(rng, (T, 4096), "normal", 1.0, wl.DTYPE_BF16)
    ys = {ly.name: np.zeros((T, 4096), np.uint16) for ly in layers}
    w = wl.Workload("prefill_r16", wl.DTYPE_BF16, 8, 16, layers, idx, {"x": x}, ys, adapters,
                    np.full(8, 16, np.int32), np.full(8, 32.0))
    out, _ = _run(w, small_batch_tokens=0)
    tok = _sample(w, 400)
    _report("prefill_r16", [check_delta(w, ly.name, out[ly.name], tokens=tok) for ly in w.layers])


def test_delta_mixed_ranks_rank64_full_size():
    """max_lora_rank 64 with true ranks 8..64: the tcgen05 prefill path for the
    six 640-token segments and the grouped decode kernels for the 256 decode
    tokens, every Llama-8B layer, sampled tokens of both kinds."""
    w = zero_base(wl.mixed_ranks_8b(0))
    out, _ = _run(w)
    tok = np.unique(np.concatenate([_sample(w, 300), np.arange(w.n_tokens - 256, w.n_tokens, 4)]))
    _report("mixed_r64", [check_delta(w, ly.name, out[ly.name], tokens=tok) for ly in w.layers])
