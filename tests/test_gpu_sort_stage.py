"""The mapping's two stages: lora_build_mapping enqueues only the CSR copy
of the batch; the adapter-sorted tuples come from a second kernel that the
paths reading them (split, tensor-core, fused, export) enqueue first and that
does nothing when the mapping's current build is sorted already (a build
counter on the device decides).

Each case checks that a path needing the sorted tuples sees those of the
latest build -- after a decode apply that never sorted, inside a CUDA graph
replayed across builds, and when the sort is skipped -- against the fp64
oracle (delta-only bound, y starts at zero) and the oracle's mapping (bit for
bit)."""
import dataclasses

import numpy as np
import pytest

import oracle
import workloads as W
from workloads import bf16_bits_to_f32
from workloads.device import DeviceWorkload, bf16_to_numpy_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PATH_SPLIT, PATH_FUSED, PATH_MMA, PATH_DECODE = 1, 2, 3, 4


@pytest.fixture(scope="module", autouse=True)
def built():
    from tenant_composite_lora_gb300 import build
    build.build()


def make_case(name):
    """A workload by name; "long" is a batch of 2500 tokens with two pairs
    each over a pool of 32 (5000 pairs): the sort of long batches, in two
    kernels, instead of the one-CTA sort."""
    if name != "long":
        return W.make(name, y_zero=True)
    rng = np.random.default_rng(77)
    T, cap = 2500, 32
    lists = [[int(v) for v in rng.choice(cap, size=2, replace=False)] for _ in range(T)]
    alphas = [list(rng.random(2).astype(np.float32)) for _ in range(T)]
    return W.make_custom(rng, d_in=256, d_out=256, r_max=16, capacity=cap, id_lists=lists, alpha_lists=alphas,
                         y_sigma=0.0, name="long_batch")


def delta_gate(y_bits, acc):
    y = bf16_bits_to_f32(y_bits).astype(np.float64)
    rms = float(np.sqrt(np.mean(acc ** 2)))
    lim = 2.0 ** -7 * np.abs(acc) + 1e-3 * rms
    assert rms > 0
    bad = np.abs(y - acc) > lim
    assert not bad.any(), f"{bad.sum()} / {acc.size} elements outside the delta bound"


def mapping_matches(got, wl):
    ref = oracle.build_mapping(wl.offsets, wl.ids, wl.alpha, capacity=wl.capacity)
    assert got["U"] == ref["U"] and got["P_valid"] == ref["P_valid"]
    for k in ("tok", "adapter", "src", "pos", "seg_adapter", "seg_start"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    assert got["alpha"].tobytes() == ref["alpha"].tobytes()


def other_batch(wl, seed):
    """Same pool and tokens, new pair lists (same count per token)."""
    rng = np.random.default_rng(seed)
    counts = np.diff(wl.offsets)
    ids = np.concatenate([rng.choice(wl.capacity, size=int(c), replace=False) for c in counts]).astype(np.int32)
    return dataclasses.replace(wl, ids=ids, alpha=rng.random(ids.size).astype(np.float32))


def device_lists(b):
    return (torch.from_numpy(b.offsets).cuda(), torch.from_numpy(b.ids).cuda(), torch.from_numpy(b.alpha).cuda())


@pytest.mark.parametrize("path", [PATH_SPLIT, PATH_MMA, PATH_FUSED])
@pytest.mark.parametrize("name", ["zipf", "sweep8", "long"])
def test_decode_apply_then_sorted_path_each_build(name, path):
    """build, decode apply (CSR only), then an apply on a sorted path, batch
    after batch on one stream without a break: the sorted path must sort the
    current build, not reuse the previous one."""
    import tenant_composite_lora_gb300 as tcl
    wl = make_case(name)
    batches = [wl] + [other_batch(wl, 200 + i) for i in range(3)]
    dw = DeviceWorkload(wl, build=False)
    s = torch.cuda.Stream()
    try:
        lists = [device_lists(b) for b in batches]
        y_dec = [dw.y0.clone() for _ in batches]
        y_srt = [dw.y0.clone() for _ in batches]
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            for (off, ids, al), yd, ys in zip(lists, y_dec, y_srt):
                dw.mapping.build(off, ids, al, s)
                tcl.delta_apply(dw.x, yd, dw.pool, dw.mapping, path=PATH_DECODE, stream=s)
                tcl.delta_apply(dw.x, ys, dw.pool, dw.mapping, path=path, stream=s)
        s.synchronize()
        assert dw.mapping.status(s) == 0
        mapping_matches(dw.mapping.export(s), batches[-1])
        got = [(bf16_to_numpy_bits(a), bf16_to_numpy_bits(b)) for a, b in zip(y_dec, y_srt)]
    finally:
        dw.close()
    for b, (yd, ys) in zip(batches, got):
        _, acc, _ = oracle.apply_workload(b, threads=0)
        delta_gate(yd, acc)
        delta_gate(ys, acc)


def test_export_after_decode_only_use():
    """A mapping only ever used by the decode path has not been sorted; the
    export sorts it first."""
    import tenant_composite_lora_gb300 as tcl
    wl = W.make("zipf", y_zero=True)
    b2 = other_batch(wl, 7)
    dw = DeviceWorkload(wl)
    try:
        y = dw.y0.clone()
        tcl.delta_apply(dw.x, y, dw.pool, dw.mapping, path=PATH_DECODE)
        dw.mapping.build(*device_lists(b2))
        tcl.delta_apply(dw.x, y, dw.pool, dw.mapping, path=PATH_DECODE)
        mapping_matches(dw.mapping.export(), b2)
    finally:
        dw.close()


@pytest.mark.parametrize("name", ["zipf", "long"])
@pytest.mark.parametrize("path", [PATH_SPLIT, PATH_MMA])
def test_graph_of_apply_sorts_each_new_build(path, name):
    """A CUDA graph holding only the apply (sort stage included), replayed
    after eager builds of different batches: every replay applies the batch
    built last."""
    from tenant_composite_lora_gb300 import native
    wl = make_case(name)
    batches = [wl, other_batch(wl, 31), other_batch(wl, 32)]
    dw = DeviceWorkload(wl)
    s = torch.cuda.Stream()
    try:
        y = dw.y0.clone()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            # one eager call first: the launch set-up runs outside the capture
            native.lora_delta_apply_path(dw.x, y, dw.pool.handle, None, dw.mapping.handle, path, s)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                native.lora_delta_apply_path(dw.x, y, dw.pool.handle, None, dw.mapping.handle, path, s)
            got = []
            for b in batches:
                off, ids, al = device_lists(b)
                s.synchronize()
                y.zero_()
                dw.mapping.build(off, ids, al, s)
                g.replay()
                s.synchronize()
                got.append(bf16_to_numpy_bits(y))
                mapping_matches(dw.mapping.export(s), b)
    finally:
        dw.close()
    for b, yb in zip(batches, got):
        _, acc, _ = oracle.apply_workload(b, threads=0)
        delta_gate(yb, acc)


@pytest.mark.parametrize("name", ["sweep64", "long"])
@pytest.mark.parametrize("path", [PATH_SPLIT, PATH_MMA])
def test_second_apply_skips_the_sort_and_agrees(path, name):
    """Two applies of one build from the same y: the second finds the tuples
    sorted (its sort stage returns at once) and gives the same bits."""
    import tenant_composite_lora_gb300 as tcl
    wl = make_case(name)
    dw = DeviceWorkload(wl)
    try:
        y1, y2 = dw.y0.clone(), dw.y0.clone()
        tcl.delta_apply(dw.x, y1, dw.pool, dw.mapping, path=path)
        tcl.delta_apply(dw.x, y2, dw.pool, dw.mapping, path=path)
        torch.cuda.synchronize()
        a, b = bf16_to_numpy_bits(y1), bf16_to_numpy_bits(y2)
        mapping_matches(dw.mapping.export(), wl)
    finally:
        dw.close()
    np.testing.assert_array_equal(a, b)
    _, acc, _ = oracle.apply_workload(wl, threads=0)
    delta_gate(a, acc)


@pytest.mark.parametrize("name", ["zipf", "long"])
def test_sorted_path_across_streams_and_builds(name):
    """The host leaves out the sort launch only after an eager sort of the
    same build on the same stream: applies alternating between two streams
    (ordered by events) over two builds each give the oracle's delta."""
    import tenant_composite_lora_gb300 as tcl
    wl = make_case(name)
    b2 = other_batch(wl, 91)
    dw = DeviceWorkload(wl)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    try:
        ys = [dw.y0.clone() for _ in range(4)]
        torch.cuda.synchronize()
        ev = torch.cuda.Event()
        with torch.cuda.stream(sa):
            tcl.delta_apply(dw.x, ys[0], dw.pool, dw.mapping, path=PATH_MMA, stream=sa)
            tcl.delta_apply(dw.x, ys[1], dw.pool, dw.mapping, path=PATH_SPLIT, stream=sa)
            ev.record(sa)
        sb.wait_event(ev)
        with torch.cuda.stream(sb):
            dw.mapping.build(*device_lists(b2), sb)
            tcl.delta_apply(dw.x, ys[2], dw.pool, dw.mapping, path=PATH_MMA, stream=sb)
            ev.record(sb)
        sa.wait_event(ev)
        with torch.cuda.stream(sa):
            tcl.delta_apply(dw.x, ys[3], dw.pool, dw.mapping, path=PATH_SPLIT, stream=sa)
        torch.cuda.synchronize()
        got = [bf16_to_numpy_bits(y) for y in ys]
        mapping_matches(dw.mapping.export(), b2)
    finally:
        dw.close()
    _, acc1, _ = oracle.apply_workload(wl, threads=0)
    _, acc2, _ = oracle.apply_workload(b2, threads=0)
    for g, acc in zip(got, (acc1, acc1, acc2, acc2)):
        delta_gate(g, acc)


@pytest.mark.parametrize("name", ["zipf", "long"])
def test_eager_sorted_apply_after_replayed_graph_build(name):
    """A build captured into a caller's graph and replayed rebuilds the
    mapping without the host seeing it: an eager sorted-path apply on the
    same stream afterwards must still sort the replayed build."""
    import tenant_composite_lora_gb300 as tcl
    wl = make_case(name)
    b2 = other_batch(wl, 57)
    dw = DeviceWorkload(wl, build=False)
    s = torch.cuda.Stream()
    try:
        l1, l2 = device_lists(wl), device_lists(b2)
        ys = [dw.y0.clone() for _ in range(3)]
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            dw.mapping.build(*l1, s)
            tcl.delta_apply(dw.x, ys[0], dw.pool, dw.mapping, path=PATH_SPLIT, stream=s)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                dw.mapping.build(*l2, s)
            # the capture ran nothing: the mapping still holds the first batch
            tcl.delta_apply(dw.x, ys[1], dw.pool, dw.mapping, path=PATH_SPLIT, stream=s)
            g.replay()
            tcl.delta_apply(dw.x, ys[2], dw.pool, dw.mapping, path=PATH_SPLIT, stream=s)
        s.synchronize()
        got = [bf16_to_numpy_bits(y) for y in ys]
        mapping_matches(dw.mapping.export(s), b2)
    finally:
        dw.close()
    _, acc1, _ = oracle.apply_workload(wl, threads=0)
    _, acc2, _ = oracle.apply_workload(b2, threads=0)
    for gy, acc in zip(got, (acc1, acc1, acc2)):
        delta_gate(gy, acc)
