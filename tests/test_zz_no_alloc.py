"""lora_apply_static_scratch: the delta of one layer for callers that cannot
allocate device memory (the scratch is a fixed array inside the library).
Its output must match lora_apply on the same inputs, on two calls in a row
(the second call finds the previous call's leftovers in the shared array)."""
import numpy as np
import pytest

from rank_adapter_apply_gb300 import workloads as wl
from tests.parity_util import TOL, decode

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
