"""lora_delta_apply_noalloc: one whole batch with its scratch in the library's
fixed static device buffer, for callers that cannot allocate device memory.

Each case starts from y = 0, so the result is the delta alone and the
delta-only bound (one bf16 rounding plus fp32 summation noise) applies: a
wrong or missing term fails it, which the stated gate at y ~ N(0, 1) would
not notice.  Two calls in a row are checked against the allocating entry
points (lora_build_mapping + lora_delta_apply_path on the same split path)
and against the fp64 oracle; free device memory must not change across the
calls.  The file is collected last, so a run that stops at its first failure
has run every other test before it."""
import numpy as np
import pytest

import oracle
import workloads as W
from workloads import bf16_bits_to_f32
from workloads.device import DeviceWorkload, bf16_to_numpy_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PATH_SPLIT = 1


def _delta_gate(y_bits, acc):
    """|y - ref| <= 2^-7 |ref| + 1e-3 rms(ref) per element (ref: fp64)."""
    y = bf16_bits_to_f32(y_bits).astype(np.float64)
    rms = float(np.sqrt(np.mean(acc ** 2)))
    lim = 2.0 ** -7 * np.abs(acc) + 1e-3 * rms
    bad = np.abs(y - acc) > lim
    assert rms > 0
    assert not bad.any(), f"{bad.sum()} / {acc.size} elements outside the delta bound"


def _near_limit_batch():
    """4096 tokens x 3 pairs at r_max = 64: about 88 % of the fixed scratch
    (small widths keep the oracle quick)."""
    rng = np.random.default_rng(17)
    cap, T = 64, 4096
    lists = [list(rng.permutation(cap)[:3]) for _ in range(T)]
    alphas = [list(rng.random(3).astype(np.float32)) for _ in range(T)]
    ranks = rng.integers(0, 65, size=cap).astype(np.int32)
    return W.make_custom(rng, d_in=256, d_out=256, r_max=64, capacity=cap, id_lists=lists,
                         alpha_lists=alphas, ranks=ranks, y_sigma=0.0, name="noalloc_near_limit")


@pytest.mark.parametrize("name", ["zipf", "sweep64", "near_limit"])
def test_noalloc_matches_allocating_entry_points_and_oracle(name):
    import tenant_composite_lora_gb300 as tcl
    from tenant_composite_lora_gb300 import build
    build.build()
    wl = _near_limit_batch() if name == "near_limit" else W.make(name, y_zero=True)
    dw = DeviceWorkload(wl)
    try:
        ref = bf16_to_numpy_bits(dw.apply(path=PATH_SPLIT))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        outs, free = [], []
        for _ in range(3):
            y = torch.zeros_like(dw.y0)
            torch.cuda.synchronize()
            free.append(torch.cuda.mem_get_info()[0])
            tcl.lora_delta_apply_noalloc(dw.x, y, dw.pool, None, dw.offsets, dw.ids, dw.alpha,
                                         wl.T, wl.P, status=status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            outs.append(bf16_to_numpy_bits(y))
    finally:
        dw.close()
    _, acc, ost = oracle.apply_workload(wl, threads=0)
    assert ost == 0
    ref_f = bf16_bits_to_f32(ref).astype(np.float64)
    for o in outs:
        _delta_gate(o, acc)      # against the oracle
        _delta_gate(o, ref_f)    # against the allocating entry points
    np.testing.assert_array_equal(outs[1], outs[2])
    assert free[1] == free[2], "device memory changed across a call"


def test_noalloc_rejects_oversize_batch():
    import tenant_composite_lora_gb300 as tcl
    wl = W.tiny()
    dw = DeviceWorkload(wl)
    try:
        big_p = 1 << 20  # scratch for this many pairs exceeds the fixed buffer
        # raw addresses: the binding's length checks would refuse this P before the library
        with pytest.raises(tcl.LoraError) as e:
            tcl.lora_delta_apply_noalloc(dw.x, dw.y0.clone(), dw.pool.handle, None, dw.offsets.data_ptr(),
                                         dw.ids.data_ptr(), dw.alpha.data_ptr(), wl.T, big_p)
        assert e.value.status == tcl.native.LORA_ERR_NOT_SUPPORTED
    finally:
        dw.close()
