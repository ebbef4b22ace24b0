"""The pages' kernel ablation (naive per-adapter loop, Copy + SGMV, explicit
pre-merge): each variant must compute the same delta as the fused path, so
each is checked against the fp64 oracle from y = 0 (delta-only bound)."""
import numpy as np
import pytest

import oracle
import workloads as W
from workloads import bf16_bits_to_f32
from workloads.device import DeviceWorkload, bf16_to_numpy_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

VARIANTS = {"naive": 1, "copy_sgmv": 2, "premerge": 3}


@pytest.fixture(scope="module", autouse=True)
def built():
    from tenant_composite_lora_gb300 import build
    build.build()


def delta_gate(y_bits, acc):
    y = bf16_bits_to_f32(y_bits).astype(np.float64)
    rms = float(np.sqrt(np.mean(acc ** 2)))
    lim = 2.0 ** -7 * np.abs(acc) + 1e-3 * rms
    assert rms > 0
    bad = np.abs(y - acc) > lim
    assert not bad.any(), f"{bad.sum()} / {acc.size} elements outside the delta bound"


def run_ablation(wl, variant):
    import tenant_composite_lora_gb300 as tcl
    dw = DeviceWorkload(wl)
    try:
        nb = tcl.lora_ablation_workspace_bytes(variant, wl.T, wl.P, wl.d_in, wl.d_out, wl.r_max)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
        y = dw.y0.clone()
        tcl.lora_delta_apply_ablation(dw.x, y, dw.pool.handle, None, dw.mapping.handle, variant, ws, nb)
        torch.cuda.synchronize()
        return bf16_to_numpy_bits(y)
    finally:
        dw.close()


def _duplicates():
    rng = np.random.default_rng(12)
    lists = [[1, 1, 3], [2], [], [0, 3, 1, 2]] * 5
    return W.make_custom(rng, d_in=128, d_out=192, r_max=16, capacity=4, id_lists=lists,
                         alpha_lists=[list(rng.random(len(l)).astype(np.float32)) for l in lists],
                         ranks=np.array([16, 5, 0, 9], np.int32), y_sigma=0.0)


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("name", ["tiny", "distinct", "zipf", "sweep8", "duplicates"])
def test_ablation_variant_matches_oracle(name, variant):
    wl = _duplicates() if name == "duplicates" else W.make(name, y_zero=True)
    y = run_ablation(wl, VARIANTS[variant])
    _, acc, _ = oracle.apply_workload(wl, threads=0)
    delta_gate(y, acc)


def test_ablation_rejects_short_workspace_and_unknown_variant():
    import tenant_composite_lora_gb300 as tcl
    wl = W.tiny()
    dw = DeviceWorkload(wl)
    try:
        nb = tcl.lora_ablation_workspace_bytes(2, wl.T, wl.P, wl.d_in, wl.d_out, wl.r_max)
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        with pytest.raises(tcl.LoraError) as e:
            tcl.lora_delta_apply_ablation(dw.x, dw.y0.clone(), dw.pool.handle, None, dw.mapping.handle, 2, ws, nb - 1)
        assert e.value.status == tcl.native.LORA_ERR_INVALID_ARG
        with pytest.raises(tcl.LoraError) as e:
            tcl.lora_delta_apply_ablation(dw.x, dw.y0.clone(), dw.pool.handle, None, dw.mapping.handle, 7, ws, nb)
        assert e.value.status == tcl.native.LORA_ERR_NOT_SUPPORTED
    finally:
        dw.close()
