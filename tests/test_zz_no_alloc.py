"""lora_delta_apply_noalloc: the whole batch with its scratch in the library's
fixed static device buffer.  Checked against the allocating entry points
(lora_build_mapping + lora_delta_apply_path on the same split path) and the
oracle, on two calls in a row, with no change in free device memory across
the calls after the first.  Collected last, so it runs alone or after every
other GPU test."""
import numpy as np
import pytest

import oracle
import workloads as W
from workloads import bf16_bits_to_f32
from workloads.device import DeviceWorkload, bf16_to_numpy_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PATH_SPLIT = 1


def _close(a_bits, b_bits):
    a = bf16_bits_to_f32(a_bits).astype(np.float64)
    b = bf16_bits_to_f32(b_bits).astype(np.float64)
    bad = np.abs(a - b) > 1e-2 + 1e-2 * np.abs(b)
    assert not bad.any(), f"{bad.sum()} elements differ beyond the stated tolerance"


@pytest.mark.parametrize("name", ["zipf", "sweep64"])
def test_noalloc_matches_allocating_entry_points(name):
    import tenant_composite_lora_gb300 as tcl
    from tenant_composite_lora_gb300 import build
    build.build()
    wl = W.make(name)
    dw = DeviceWorkload(wl)
    try:
        ref = bf16_to_numpy_bits(dw.apply(path=PATH_SPLIT))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        outs, free = [], []
        for _ in range(3):
            y = dw.y0.clone()
            torch.cuda.synchronize()
            free.append(torch.cuda.mem_get_info()[0])
            tcl.lora_delta_apply_noalloc(dw.x, y, dw.pool.handle, None, dw.offsets, dw.ids, dw.alpha,
                                         wl.T, wl.P, status=status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            outs.append(bf16_to_numpy_bits(y))
    finally:
        dw.close()
    for o in outs:
        _close(o, ref)
    np.testing.assert_array_equal(outs[1], outs[2])
    assert free[1] == free[2], "device memory changed across a call"
    yref, _, _ = oracle.apply_workload(wl, threads=0)
    _close(outs[2], yref)


def test_noalloc_rejects_oversize_batch():
    import tenant_composite_lora_gb300 as tcl
    wl = W.tiny()
    dw = DeviceWorkload(wl)
    try:
        big_p = 1 << 20  # scratch for this many pairs exceeds the fixed buffer
        with pytest.raises(tcl.LoraError) as e:
            tcl.lora_delta_apply_noalloc(dw.x, dw.y0.clone(), dw.pool.handle, None, dw.offsets, dw.ids,
                                         dw.alpha, wl.T, big_p)
        assert e.value.status == tcl.native.LORA_ERR_NOT_SUPPORTED
    finally:
        dw.close()
