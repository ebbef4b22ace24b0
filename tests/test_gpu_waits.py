"""Every on-chip wait of the library is bounded.  Here each kind of wait is
made to run out on purpose (an mbarrier phase nobody completes, a counter
nobody increments) with a short limit: the kernel must give up near that
limit, report LORA_DEV_TIMEOUT, return normally, and leave the context
usable for the next call.  No fault is involved: the wait simply ends."""
import numpy as np
import pytest

import oracle
import workloads as W
from workloads import bf16_bits_to_f32
from workloads.device import DeviceWorkload, bf16_to_numpy_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

LORA_DEV_TIMEOUT = 16


@pytest.fixture(scope="module", autouse=True)
def built():
    from tenant_composite_lora_gb300 import build
    build.build()


@pytest.mark.parametrize("kind", [0, 1], ids=["mbarrier", "counter"])
def test_bounded_wait_expires_and_reports(kind):
    import tenant_composite_lora_gb300 as tcl
    limit_ns = 2_000_000  # 2 ms
    words = torch.zeros(4, dtype=torch.int32, device="cuda")
    tcl.lora_diag_wait_expiry(kind, limit_ns, words)
    torch.cuda.synchronize()  # the kernel returned
    w = words.cpu().numpy()
    assert w[0] & LORA_DEV_TIMEOUT, w
    assert w[2] == 0, "the wait cannot have been satisfied"
    assert limit_ns / 1000 <= w[3] < 50 * limit_ns / 1000, f"waited {w[3]} us for a {limit_ns / 1000} us limit"
    # the context is still usable: a real delta afterwards is right
    wl = W.tiny(y_zero=True)
    dw = DeviceWorkload(wl)
    try:
        y = bf16_to_numpy_bits(dw.apply())
        assert dw.mapping.status() == 0
    finally:
        dw.close()
    _, acc, _ = oracle.apply_workload(wl)
    yf = bf16_bits_to_f32(y).astype(np.float64)
    rms = float(np.sqrt(np.mean(acc ** 2)))
    assert np.all(np.abs(yf - acc) <= 2.0 ** -7 * np.abs(acc) + 1e-3 * rms)


def test_bounded_wait_limits_are_checked():
    import tenant_composite_lora_gb300 as tcl
    words = torch.zeros(4, dtype=torch.int32, device="cuda")
    for kind, lim in ((2, 10_000), (0, 10), (1, 10 ** 9)):
        with pytest.raises(tcl.LoraError):
            tcl.lora_diag_wait_expiry(kind, lim, words)
