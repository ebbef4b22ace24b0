"""lora_delta_apply_multi: several projections (each its own pool and shape)
over one shared mapping, in one launch pair for decode batches.

Each projection's result is checked against the fp64 oracle (delta-only
bound, from y = 0) and must equal, bit for bit, what a separate
lora_delta_apply of that projection on the decode path gives wherever that
call uses the same expand kernel (the wide-rank expand, taken by a single
call for r_max > 16 with few (token, column) items, sums in another order).
Long batches fall back to one apply per projection and must equal the
separate applies bit for bit."""
import numpy as np
import pytest

import oracle
import workloads as W
from workloads import bf16_bits_to_f32
from workloads.device import bf16_tensor, bf16_to_numpy_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PATH_DECODE = 4


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


def _projections(base, shapes, seed):
    """One workload per projection: the batch's pair lists, with each
    projection's own widths, ranks and factors (and its own x)."""
    rng = np.random.default_rng(seed)
    lists, alphas = [], []
    for t in range(base.T):
        a, b = int(base.offsets[t]), int(base.offsets[t + 1])
        lists.append([int(v) for v in base.ids[a:b]])
        alphas.append([np.float32(v) for v in base.alpha[a:b]])
    out = []
    for d_in, d_out, r_max, ranks in shapes:
        rk = None if ranks is None else ranks(rng, base.capacity, r_max)
        out.append(W.make_custom(rng, d_in=d_in, d_out=d_out, r_max=r_max, capacity=base.capacity,
                                 id_lists=lists, alpha_lists=alphas, ranks=rk, y_sigma=0.0))
    return out


def _run(wls, multi: bool):
    import tenant_composite_lora_gb300 as tcl
    base = wls[0]
    pools, xs, ys = [], [], []
    s = torch.cuda.Stream()
    m = tcl.LoraMapping(base.T, base.P, base.capacity)
    try:
        for wl in wls:
            p = tcl.LoraPool(wl.d_in, wl.d_out, wl.r_max, wl.capacity)
            for a in range(wl.capacity):
                p.register(a, bf16_tensor(wl.A[a]), bf16_tensor(wl.B[a]), int(wl.ranks[a]), s)
            pools.append(p)
            xs.append(bf16_tensor(wl.x))
            ys.append(bf16_tensor(wl.y))
        with torch.cuda.stream(s):
            m.build(torch.from_numpy(base.offsets).cuda(), torch.from_numpy(base.ids).cuda(),
                    torch.from_numpy(base.alpha).cuda(), s)
            if multi:
                tcl.lora_delta_apply_multi([(x, y, p.handle, None) for x, y, p in zip(xs, ys, pools)],
                                           m.handle, s)
            else:
                for x, y, p in zip(xs, ys, pools):
                    tcl.delta_apply(x, y, p, m, path=PATH_DECODE if base.T <= 256 else 0, stream=s)
        s.synchronize()
        assert m.status(s) == 0
        return [bf16_to_numpy_bits(y) for y in ys]
    finally:
        for p in pools:
            p.close()
        m.close()


def _rank_uniform(rng, cap, r_max):
    return rng.integers(1, r_max + 1, size=cap).astype(np.int32)


# q, k, v, o projections of a Llama-3-8B layer (GQA: k/v 4096 -> 1024), the
# last two at larger and heterogeneous retained ranks
LAYER = [(4096, 4096, 8, None), (4096, 1024, 8, None), (4096, 1024, 16, None), (4096, 4096, 64, _rank_uniform)]


@pytest.mark.parametrize("name", ["distinct", "zipf", "sweep8"])
def test_multi_matches_oracle_and_separate_applies(name):
    wls = _projections(W.make(name), LAYER, seed=7)
    got = _run(wls, multi=True)
    sep = _run(wls, multi=False)
    for wl, g, s_ in zip(wls, got, sep):
        wide = wl.r_max > 16 and wl.T * ((wl.d_out + 255) // 256) <= 2 * torch.cuda.get_device_properties(0).multi_processor_count
        if not wide:
            np.testing.assert_array_equal(g, s_)
        _, acc, _ = oracle.apply_workload(wl, threads=0)
        delta_gate(g, acc)
        delta_gate(s_, acc)


def test_multi_long_batch_falls_back_to_separate_applies():
    base = W.sparse_prefill(n_requests=3)
    wls = _projections(base, [(256, 512, 16, None), (512, 256, 8, None)], seed=3)
    got = _run(wls, multi=True)
    sep = _run(wls, multi=False)
    for wl, g, s_ in zip(wls, got, sep):
        np.testing.assert_array_equal(g, s_)
        _, acc, _ = oracle.apply_workload(wl, threads=0)
        delta_gate(g, acc)


def test_multi_rejects_aliased_outputs_and_mismatched_pools():
    import tenant_composite_lora_gb300 as tcl
    wl = W.tiny()
    m = tcl.LoraMapping(wl.T, wl.P, wl.capacity)
    p = tcl.LoraPool(wl.d_in, wl.d_out, wl.r_max, wl.capacity)
    q = tcl.LoraPool(wl.d_in, wl.d_out, wl.r_max, wl.capacity + 1)
    try:
        m.build(torch.from_numpy(wl.offsets).cuda(), torch.from_numpy(wl.ids).cuda(),
                torch.from_numpy(wl.alpha).cuda())
        x, y, y2 = bf16_tensor(wl.x), bf16_tensor(wl.y), bf16_tensor(wl.y)
        for projs in ([(x, y, p.handle, None), (x, y, p.handle, None)],   # one y twice
                      [(x, y, p.handle, None), (y, y2, p.handle, None)],  # an output read as an input
                      [(x, y, q.handle, None)]):                          # capacity differs from the mapping's
            with pytest.raises(tcl.LoraError) as e:
                tcl.lora_delta_apply_multi(projs, m.handle)
            assert e.value.status == tcl.native.LORA_ERR_INVALID_ARG
        with pytest.raises(tcl.LoraError) as e:
            tcl.lora_delta_apply_multi([(x, y2, p.handle, None)] * 9, m.handle)
        assert e.value.status == tcl.native.LORA_ERR_NOT_SUPPORTED
    finally:
        p.close()
        q.close()
        m.close()
