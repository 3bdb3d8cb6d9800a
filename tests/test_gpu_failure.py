"""Failure detection on the GPU without a fault: every wait of the kernels is
bounded; when one gives up, the kernel records it in the device error word and
returns, the host reads it through lora_stats, and the context keeps working.
The self-test kernel waits on a barrier that nothing completes."""
import pytest

from rank_adapter_apply_gb300 import workloads as wl
from tests.parity_util import check_layer

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_context_stays_usable():
    from rank_adapter_apply_gb300 import binding as B
    from rank_adapter_apply_gb300 import build
    from rank_adapter_apply_gb300.harness import DeviceWorkload
    build.build()
    w = wl.decode_qv_4096(6, n_tokens=64)
    dw = DeviceWorkload(w)
    try:
        assert dw.slots.stats()["device_wait_timeouts"] == 0
        assert B.lora_selftest_wait_timeout(dw.slots.ctx) == 1
        assert dw.slots.stats()["device_wait_timeouts"] == 1
        out = dw.run()
        for ly in w.layers:
            check_layer(w, ly.name, out[ly.name])
    finally:
        dw.close()
