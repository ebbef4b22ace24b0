"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Mapping: bit-exact (tuples, alpha bits, inverse permutation, segments).
Delta: |y - y_ref| <= 1e-2 + 1e-2 |y_ref| per element (the stated gate), and
on runs with y_in = 0 the delta-only bound |y - ref| <= 2^-7 |ref| +
1e-3 rms(ref), which one bf16 rounding plus fp32 summation noise satisfy and a
wrong or missing term does not (|delta| is far below the bf16 spacing of y_in).
"""
import dataclasses

import numpy as np
import pytest

import oracle
import workloads as W
from workloads import bf16_bits_to_f32
from workloads.device import DeviceWorkload, bf16_tensor, bf16_to_numpy_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built_and_stream():
    from tenant_composite_lora_gb300 import build
    build.build()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        yield s
    torch.cuda.synchronize()


def stated_gate(y_bits, yref_bits):
    y = bf16_bits_to_f32(y_bits).astype(np.float64)
    r = bf16_bits_to_f32(yref_bits).astype(np.float64)
    bad = np.abs(y - r) > 1e-2 + 1e-2 * np.abs(r)
    assert not bad.any(), f"{bad.sum()} elements outside the stated tolerance"


def delta_gate(y_bits, acc):
    y = bf16_bits_to_f32(y_bits).astype(np.float64)
    rms = float(np.sqrt(np.mean(acc ** 2))) if acc.size else 0.0
    err = np.abs(y - acc)
    lim = 2.0 ** -7 * np.abs(acc) + 1e-3 * rms
    bad = err > lim
    assert not bad.any(), (f"{bad.sum()} / {acc.size} elements outside the delta bound; "
                           f"worst {float((err - lim).max()):.3g}, rms {rms:.3g}")
    assert rms > 0


def run_gpu(wl, ranks=None, path=0, y_in=None):
    dw = DeviceWorkload(wl)
    try:
        y = dw.y0.clone() if y_in is None else bf16_tensor(y_in)
        r = None if ranks is None else torch.from_numpy(np.asarray(ranks, np.int32)).cuda()
        dw.apply(y=y, ranks=r, path=path)
        torch.cuda.synchronize()
        st = dw.mapping.status()
        return bf16_to_numpy_bits(y), st
    finally:
        dw.close()


# ---------------------------------------------------------------- mapping
def compare_mapping(got, ref):
    assert got["U"] == ref["U"] and got["P_valid"] == ref["P_valid"]
    for k in ("tok", "adapter", "src", "pos", "seg_adapter", "seg_start"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    assert got["alpha"].tobytes() == ref["alpha"].tobytes()
    assert got["status"] == ref["status"]


MAP_CASES = ["tiny", "distinct", "zipf", "prefill", "sweep1", "sweep8", "sweep64", "sweep256"]


@pytest.mark.parametrize("name", MAP_CASES)
def test_mapping_bit_exact(name):
    wl = W.make(name)
    dw = DeviceWorkload(wl)
    try:
        got = dw.mapping.export()
    finally:
        dw.close()
    compare_mapping(got, oracle.build_mapping(wl.offsets, wl.ids, wl.alpha, capacity=wl.capacity))


def _map_raw(offsets, ids, alpha, cap):
    import tenant_composite_lora_gb300 as tcl
    m = tcl.LoraMapping(max(len(offsets) - 1, 1), max(len(ids), 1), cap)
    try:
        m.build(torch.from_numpy(np.asarray(offsets, np.int32)).cuda(),
                torch.from_numpy(np.asarray(ids, np.int32)).cuda(),
                torch.from_numpy(np.asarray(alpha, np.float32)).cuda())
        return m.export()
    finally:
        m.close()


@pytest.mark.parametrize("n_tok", [300, 2000])
def test_mapping_invalid_ids_and_empty_tokens(n_tok):
    """Out-of-range ids among valid ones; 2000 tokens (about 4000 pairs) takes
    the long-batch variant that stages the sorted arrays in shared memory."""
    rng = np.random.default_rng(11)
    cap = 37
    counts = rng.integers(0, 5, size=n_tok)
    offsets = np.zeros(n_tok + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    ids = rng.integers(-3, cap + 3, size=int(counts.sum())).astype(np.int32)
    alpha = rng.standard_normal(ids.size).astype(np.float32)
    compare_mapping(_map_raw(offsets, ids, alpha, cap), oracle.build_mapping(offsets, ids, alpha, capacity=cap))


def test_mapping_bad_offsets_and_degenerate():
    for offsets, ids in (([0, 2, 1, 3], [0, 1, 2]), ([1, 2, 3], [0, 1, 2]), ([0, 1, 2], [0, 1, 2])):
        ref = oracle.build_mapping(np.array(offsets, np.int32), np.array(ids, np.int32),
                                   np.ones(len(ids), np.float32), capacity=4)
        got = _map_raw(offsets, ids, np.ones(len(ids)), 4)
        compare_mapping(got, ref)
        assert got["status"] & 2
    # no pairs at all, and one token with every adapter of a large pool
    compare_mapping(_map_raw([0, 0, 0], [], [], 5), oracle.build_mapping(
        np.zeros(3, np.int32), np.zeros(0, np.int32), np.zeros(0, np.float32), capacity=5))
    # no token: offsets {0} and no pair; offsets {2} with two pairs is malformed
    compare_mapping(_map_raw([0], [], [], 5), oracle.build_mapping(
        np.zeros(1, np.int32), np.zeros(0, np.int32), np.zeros(0, np.float32), capacity=5))
    got = _map_raw([2], [0, 1], np.ones(2), 5)
    compare_mapping(got, oracle.build_mapping(np.array([2], np.int32), np.array([0, 1], np.int32),
                                              np.ones(2, np.float32), capacity=5))
    assert got["status"] & 2
    cap = 3000
    ids = np.random.default_rng(3).permutation(cap).astype(np.int32)
    offsets = np.array([0, cap], np.int32)
    compare_mapping(_map_raw(offsets, ids, np.ones(cap), cap),
                    oracle.build_mapping(offsets, ids, np.ones(cap, np.float32), capacity=cap))


@pytest.mark.parametrize("form", ["step_down", "first", "last", "beyond_p", "valid"])
def test_mapping_long_batch_offsets(form):
    """3000 tokens: the CSR stage runs over several CTAs, each checking its own
    tokens' offsets; malformed offsets anywhere (inside one CTA's range, at
    either end, beyond P) leave every pair out, as the oracle does, and some
    ids outside the pool are among them."""
    rng = np.random.default_rng(23)
    n_tok, cap = 3000, 50
    counts = rng.integers(0, 4, size=n_tok)
    offsets = np.zeros(n_tok + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    P = int(offsets[-1])
    ids = rng.integers(-2, cap + 2, size=P).astype(np.int32)
    alpha = rng.standard_normal(P).astype(np.float32)
    if form == "step_down":
        offsets[1700] = offsets[1701] + 1
    elif form == "first":
        offsets[0] = 1
    elif form == "last":
        offsets[-1] = P - 1
    elif form == "beyond_p":
        offsets[900] = P + 5
    got = _map_raw(offsets, ids, alpha, cap)
    compare_mapping(got, oracle.build_mapping(offsets, ids, alpha, capacity=cap))
    assert bool(got["status"] & 2) == (form != "valid")


@pytest.mark.parametrize("cap", [20000, 49152])
def test_mapping_large_pools(cap):
    """Pools too large for the shared-memory histograms (up to the library's
    capacity limit) take the global-memory histograms: still bit-exact,
    out-of-range ids included."""
    rng = np.random.default_rng(cap)
    n_tok = 1500
    counts = rng.integers(0, 6, size=n_tok)
    offsets = np.zeros(n_tok + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    ids = rng.integers(-2, cap + 2, size=int(counts.sum())).astype(np.int32)
    ids[::7] = cap - 1 - (np.arange(ids[::7].size) % 5)  # repeated keys at the top of the range
    alpha = rng.standard_normal(ids.size).astype(np.float32)
    compare_mapping(_map_raw(offsets, ids, alpha, cap), oracle.build_mapping(offsets, ids, alpha, capacity=cap))


def test_apply_large_pool():
    """A pool of 20000 slots (global-memory histograms in the mapping, rank
    lookups outside the staged table) through every path."""
    rng = np.random.default_rng(8)
    cap = 20000
    lists = [list(rng.choice(cap, size=int(rng.integers(1, 4)), replace=False)) for _ in range(40)]
    lists += [[cap - 1, 0, 12345]]
    ranks = rng.integers(0, 3, size=cap).astype(np.int32)
    wl = W.make_custom(rng, d_in=64, d_out=128, r_max=2, capacity=cap, id_lists=lists,
                       alpha_lists=[list(rng.random(len(l)).astype(np.float32)) for l in lists],
                       ranks=ranks, y_sigma=0.0)
    _, acc, _ = oracle.apply_workload(wl)
    for path in ALL_PATHS:
        y, st = run_gpu(wl, path=path)
        assert st == 0
        delta_gate(y, acc)


# ---------------------------------------------------------------- delta, element-wise
APPLY_CASES = ["tiny", "distinct", "zipf", "sweep1", "sweep8", "sweep64", "sweep256"]
PATH_AUTO, PATH_SPLIT, PATH_FUSED, PATH_MMA, PATH_DECODE = 0, 1, 2, 3, 4
DECODE_PATHS = [PATH_AUTO, PATH_SPLIT, PATH_FUSED, PATH_DECODE]
ALL_PATHS = [PATH_AUTO, PATH_SPLIT, PATH_FUSED, PATH_MMA, PATH_DECODE]


@pytest.mark.parametrize("name", APPLY_CASES)
def test_apply_matches_oracle(name):
    wl = W.make(name)
    y, st = run_gpu(wl)
    yref, _, ost = oracle.apply_workload(wl, threads=0)
    assert st == ost == 0
    stated_gate(y, yref)


@pytest.mark.parametrize("path", ALL_PATHS)
@pytest.mark.parametrize("name", APPLY_CASES)
def test_apply_delta_only(name, path):
    wl = W.make(name, y_zero=True)
    y, st = run_gpu(wl, path=path)
    _, acc, ost = oracle.apply_workload(wl, threads=0)
    assert st == ost == 0
    delta_gate(y, acc)


@pytest.mark.parametrize("path", [PATH_AUTO, PATH_SPLIT, PATH_MMA])
def test_prefill_small_delta_only(path):
    wl = W.sparse_prefill(n_requests=3, y_zero=True)
    y, st = run_gpu(wl, path=path)
    _, acc, ost = oracle.apply_workload(wl, threads=0)
    assert st == ost == 0
    delta_gate(y, acc)


def test_paths_agree_bitwise_where_order_matches():
    """Split and fused paths sum in the same order only per window; both must
    pass the delta bound, and repeated fused launches (barrier counters
    carried across launches) must give identical bits."""
    wl = W.zipf_decode(y_zero=True)
    dw = DeviceWorkload(wl)
    try:
        runs = [bf16_to_numpy_bits(dw.apply(path=PATH_FUSED)) for _ in range(4)]
    finally:
        dw.close()
    for r in runs[1:]:
        np.testing.assert_array_equal(r, runs[0])


_PREFILL_REF = {}


def _prefill_reference(y_zero: bool):
    """The full sparse-prefill batch and the oracle's result on every token
    (computed once per module; OpenMP over tokens)."""
    if y_zero not in _PREFILL_REF:
        wl = W.sparse_prefill(y_zero=y_zero)
        yref, acc, ost = oracle.apply_workload(wl, threads=0)
        assert ost == 0
        _PREFILL_REF[y_zero] = (wl, yref, acc)
    return _PREFILL_REF[y_zero]


@pytest.mark.parametrize("path", [PATH_AUTO, PATH_MMA, PATH_SPLIT, PATH_DECODE])
def test_prefill_full_size_every_token(path):
    """The whole sparse-prefill batch (3250 tokens, 6500 pairs) in the
    benchmark's launch configuration (the dispatch table sends it to the
    tensor-core path), every element of every token against the oracle's
    delta: a tile-boundary or scheduling slip anywhere in the batch fails.
    Forced onto the decode path the batch takes the long-batch instances
    (two row groups per shrink CTA, the one-wave expand)."""
    wl, _, acc = _prefill_reference(True)
    y, st = run_gpu(wl, path=path)
    assert st == 0
    delta_gate(y, acc)


@pytest.mark.parametrize("path", [PATH_AUTO, PATH_MMA])
def test_prefill_full_size_stated_gate(path):
    """The same batch from y ~ N(0, 1), every element against the stated
    tolerance."""
    wl, yref, _ = _prefill_reference(False)
    y, st = run_gpu(wl, path=path)
    assert st == 0
    stated_gate(y, yref)


# ---------------------------------------------------------------- stream ordering
def _other_batch(wl, seed):
    """The same pool and tokens with new pair lists: per token the same number
    of pairs, distinct ids drawn afresh, new alpha."""
    rng = np.random.default_rng(seed)
    counts = np.diff(wl.offsets)
    ids = np.concatenate([rng.choice(wl.capacity, size=int(c), replace=False) for c in counts]).astype(np.int32)
    alpha = rng.random(ids.size).astype(np.float32)
    return dataclasses.replace(wl, ids=ids, alpha=alpha)


@pytest.mark.parametrize("path", [PATH_DECODE, PATH_FUSED])
@pytest.mark.parametrize("name", ["zipf", "sweep8", "distinct"])
def test_new_mapping_then_apply_without_a_break(name, path):
    """Batch after batch on one stream, each apply straight after its mapping
    (no other kernel, no synchronisation in between), as a decode loop runs:
    every apply must see its own batch's mapping, not the previous one."""
    import tenant_composite_lora_gb300 as tcl
    wl = W.make(name, y_zero=True)
    batches = [wl] + [_other_batch(wl, 100 + i) for i in range(3)]
    dw = DeviceWorkload(wl, build=False)
    s = torch.cuda.Stream()
    try:
        dev = [(torch.from_numpy(b.offsets).cuda(), torch.from_numpy(b.ids).cuda(),
                torch.from_numpy(b.alpha).cuda()) for b in batches]
        ys = [dw.y0.clone() for _ in batches]
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            for (off, ids, al), y in zip(dev, ys):
                dw.mapping.build(off, ids, al, s)
                tcl.delta_apply(dw.x, y, dw.pool, dw.mapping, path=path, stream=s)
        s.synchronize()
        got = [bf16_to_numpy_bits(y) for y in ys]
    finally:
        dw.close()
    for b, y in zip(batches, got):
        _, acc, _ = oracle.apply_workload(b, threads=0)
        delta_gate(y, acc)


@pytest.mark.parametrize("path", [PATH_DECODE, PATH_FUSED])
@pytest.mark.parametrize("name", ["zipf", "sweep8"])
def test_two_applies_into_one_y_without_a_break(name, path):
    """Two applies of one mapping into the same y back to back (y starts at
    zero): the second must read the first one's result, so y ends at twice
    the delta."""
    import tenant_composite_lora_gb300 as tcl
    wl = W.make(name, y_zero=True)
    dw = DeviceWorkload(wl)
    s = torch.cuda.Stream()
    try:
        y = dw.y0.clone()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            for _ in range(2):
                tcl.delta_apply(dw.x, y, dw.pool, dw.mapping, path=path, stream=s)
        s.synchronize()
        got = bf16_to_numpy_bits(y)
    finally:
        dw.close()
    _, acc, _ = oracle.apply_workload(wl, threads=0)
    delta_gate(got, 2.0 * acc)


# ---------------------------------------------------------------- contracts
@pytest.mark.parametrize("path", ALL_PATHS)
def test_garbage_padding_is_inert(path):
    zero = W.rank_sweep(64)
    garb = W.rank_sweep(64, garbage_padding=True)
    y0, _ = run_gpu(zero, path=path)
    y1, _ = run_gpu(garb, path=path)
    np.testing.assert_array_equal(y0, y1)


@pytest.mark.parametrize("path", [PATH_AUTO, PATH_MMA, PATH_SPLIT])
def test_rank_override_and_bad_rank(path):
    wl = W.rank_sweep(64, y_zero=True)
    rng = np.random.default_rng(5)
    ranks = np.minimum(wl.ranks, rng.integers(0, 65, size=wl.capacity)).astype(np.int32)
    y, st = run_gpu(wl, ranks=ranks, path=path)
    _, acc, _ = oracle.apply_workload(wl, ranks=ranks)
    assert st == 0
    delta_gate(y, acc)
    bad = ranks.copy()
    victim = int(wl.ids[0])
    bad[victim] = wl.r_max + 5
    y, st = run_gpu(wl, ranks=bad, path=path)
    assert st & 8
    ok = bad.copy()
    ok[victim] = 0
    _, acc, _ = oracle.apply_workload(wl, ranks=ok)
    delta_gate(y, acc)


@pytest.mark.parametrize("path", [PATH_AUTO, PATH_MMA, PATH_SPLIT])
def test_unregistered_slot(path):
    wl = W.zipf_decode(y_zero=True)
    victim = int(wl.ids[1])
    reg = wl.ranks.copy()
    reg[victim] = -1
    dw = DeviceWorkload(wl, register_ranks=reg)
    try:
        y = dw.apply(y=torch.zeros_like(dw.y0), path=path)
        st = dw.mapping.status()
    finally:
        dw.close()
    assert st & 4
    _, acc, ost = oracle.apply_workload(wl, ranks=reg)
    assert ost & 4
    delta_gate(bf16_to_numpy_bits(y), acc)


@pytest.mark.parametrize("path", ALL_PATHS)
def test_deterministic(path):
    wl = W.rank_sweep(256)
    dw = DeviceWorkload(wl)
    try:
        a = bf16_to_numpy_bits(dw.apply(path=path))
        b = bf16_to_numpy_bits(dw.apply(path=path))
    finally:
        dw.close()
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("path", [PATH_AUTO, PATH_MMA, PATH_SPLIT])
def test_noops(path):
    wl = W.tiny()
    wl.alpha[:] = 0
    y, _ = run_gpu(wl, path=path)
    np.testing.assert_array_equal(bf16_bits_to_f32(y), bf16_bits_to_f32(wl.y))
    wl = W.tiny()
    y, _ = run_gpu(wl, ranks=np.zeros(wl.capacity, np.int32), path=path)
    np.testing.assert_array_equal(bf16_bits_to_f32(y), bf16_bits_to_f32(wl.y))


def test_order_invariance():
    wl = W.zipf_decode(y_zero=True)
    y0, _ = run_gpu(wl)
    rng = np.random.default_rng(9)
    for t in range(wl.T):
        a, b = wl.offsets[t], wl.offsets[t + 1]
        perm = rng.permutation(b - a) + a
        wl.ids[a:b] = wl.ids[perm]
        wl.alpha[a:b] = wl.alpha[perm]
    y1, _ = run_gpu(wl)
    _, acc, _ = oracle.apply_workload(wl)
    delta_gate(y0, acc)
    delta_gate(y1, acc)


@pytest.mark.parametrize("name", ["zipf", "sweep400"])
def test_host_entry_point_matches_device_path(name):
    """The host entry point from pinned buffers gives the device path's bits:
    a decode batch (x brought over once by a copy kernel, the pair lists and
    y read and written in host memory by the step's kernels) and a 400-token
    rank-64 batch (tensor-core path, copy kernels around it)."""
    import tenant_composite_lora_gb300 as tcl
    from tenant_composite_lora_gb300 import native
    wl = W.zipf_decode() if name == "zipf" else W.rank_sweep(400)
    want = native.LORA_PATH_DECODE if name == "zipf" else native.LORA_PATH_MMA
    assert native.lora_dispatch_choose(wl.T, wl.P, wl.r_max, wl.d_in, wl.d_out) == want
    dw = DeviceWorkload(wl)
    try:
        ref = bf16_to_numpy_bits(dw.apply())
        y_host = torch.from_numpy(wl.y.view(np.int16).copy()).pin_memory()
        x_host = torch.from_numpy(wl.x.view(np.int16).copy()).pin_memory()
        off = torch.from_numpy(wl.offsets).pin_memory()
        ids = torch.from_numpy(wl.ids).pin_memory()
        al = torch.from_numpy(wl.alpha).pin_memory()
        tcl.lora_delta_apply_host(x_host, y_host, off, ids, al, wl.T, wl.P, dw.pool.handle, None,
                                  dw.mapping.handle)
        torch.cuda.current_stream().synchronize()
        got = y_host.numpy().view(np.uint16)
    finally:
        dw.close()
    np.testing.assert_array_equal(got, ref)


def test_host_entry_point_chained_steps():
    """Each step's x is the previous step's y (a square pool, d_in = d_out),
    host steps enqueued back to back on one stream: the step that brings x
    over the host link must not read it before the step ahead has written
    it.  The chain's bits equal the same chain on device buffers."""
    import tenant_composite_lora_gb300 as tcl
    from tenant_composite_lora_gb300 import native
    wl = W.make("distinct")
    assert wl.d_in == wl.d_out
    assert native.lora_dispatch_choose(wl.T, wl.P, wl.r_max, wl.d_in, wl.d_out) == native.LORA_PATH_DECODE
    n = 5
    rng = np.random.default_rng(12)
    starts = [W.f32_to_bf16_bits(rng.standard_normal(wl.x.shape).astype(np.float32)) for _ in range(n + 1)]
    dw = DeviceWorkload(wl)
    s = torch.cuda.Stream()
    try:
        dev = [torch.from_numpy(v.view(np.int16).copy()).cuda() for v in starts]
        hst = [torch.from_numpy(v.view(np.int16).copy()).pin_memory() for v in starts]
        off = torch.from_numpy(wl.offsets).pin_memory()
        ids = torch.from_numpy(wl.ids).pin_memory()
        al = torch.from_numpy(wl.alpha).pin_memory()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            for i in range(n):
                native.lora_delta_apply(dev[i], dev[i + 1], dw.pool.handle, None, dw.mapping.handle, s)
            for i in range(n):
                tcl.lora_delta_apply_host(hst[i], hst[i + 1], off, ids, al, wl.T, wl.P, dw.pool.handle, None,
                                          dw.mapping.handle, s)
        s.synchronize()
        assert dw.mapping.status(s) == 0
        want = [t.cpu().numpy().view(np.uint16) for t in dev]
        got = [t.numpy().view(np.uint16) for t in hst]
    finally:
        dw.close()
    for i in range(1, n + 1):
        np.testing.assert_array_equal(got[i], want[i], err_msg=f"step {i}")
    assert not np.array_equal(want[n], starts[n])


def _host_calls(wl, dw, x_host, y_host, off, ids, al, n_calls, before_call=None):
    """n_calls host-entry steps on one stream with new alpha and y values each
    time, every result checked against the oracle."""
    import tenant_composite_lora_gb300 as tcl
    s = torch.cuda.Stream()
    rng = np.random.default_rng(4)
    for it in range(n_calls):
        if before_call is not None:
            before_call(it)
        y_in = W.f32_to_bf16_bits(rng.standard_normal(wl.y.shape).astype(np.float32))
        al.copy_(torch.from_numpy((wl.alpha * (1 + it)).astype(np.float32)))
        y_host.copy_(torch.from_numpy(y_in.view(np.int16)))
        tcl.lora_delta_apply_host(x_host, y_host, off, ids, al, wl.T, wl.P, dw.pool.handle, None,
                                  dw.mapping.handle, s)
        s.synchronize()
        got = y_host.numpy().view(np.uint16).copy()
        wl_it = dataclasses.replace(wl, alpha=(wl.alpha * (1 + it)).astype(np.float32), y=y_in)
        yref, _, _ = oracle.apply_workload(wl_it, threads=0)
        stated_gate(got, yref)


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_entry_point_graph_replay(pinned):
    """Repeated identical host calls: eager, then captured, then replayed;
    new input values between calls must be picked up by the replay.  Pinned
    buffers take the copy kernels, pageable ones the copy calls (whose
    capture may be refused, leaving every call eager)."""
    wl = W.distinct_decode()
    dw = DeviceWorkload(wl)
    host = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    try:
        _host_calls(wl, dw, host(torch.from_numpy(wl.x.view(np.int16).copy())),
                    host(torch.empty(wl.y.shape, dtype=torch.int16)), host(torch.from_numpy(wl.offsets)),
                    host(torch.from_numpy(wl.ids)), host(torch.from_numpy(wl.alpha)), 5)
    finally:
        dw.close()


def test_host_entry_point_new_pool_at_old_address():
    """A step graph captured against a pool must not replay after that pool is
    destroyed and another is created, even when the new pool's host object
    lands at the old address (the usual outcome of free + calloc of the same
    size): the new pool's factors must be used."""
    import tenant_composite_lora_gb300 as tcl
    wl1 = W.tiny(seed=0, y_zero=True)
    wl2 = dataclasses.replace(W.tiny(seed=1, y_zero=True), offsets=wl1.offsets, ids=wl1.ids, alpha=wl1.alpha,
                              x=wl1.x, y=wl1.y)
    s = torch.cuda.Stream()
    host = [torch.from_numpy(a).pin_memory() for a in
            (wl1.x.view(np.int16).copy(), wl1.offsets, wl1.ids, wl1.alpha)]
    y_host = torch.empty(wl1.y.shape, dtype=torch.int16).pin_memory()
    m = tcl.LoraMapping(wl1.T, wl1.P, wl1.capacity)

    def pool_of(wl):
        p = tcl.LoraPool(wl.d_in, wl.d_out, wl.r_max, wl.capacity)
        for a in range(wl.capacity):
            p.register(a, bf16_tensor(wl.A[a]), bf16_tensor(wl.B[a]), int(wl.ranks[a]), s)
        s.synchronize()
        return p

    def step(pool):
        y_host.copy_(torch.from_numpy(wl1.y.view(np.int16)))
        tcl.lora_delta_apply_host(host[0], y_host, host[1], host[2], host[3], wl1.T, wl1.P, pool.handle, None,
                                  m.handle, s)
        s.synchronize()
        return y_host.numpy().view(np.uint16).copy()

    try:
        p1 = pool_of(wl1)
        for _ in range(3):  # eager, captured, replayed
            got1 = step(p1)
        p1.close()
        p2 = pool_of(wl2)
        got2 = step(p2)
        p2.close()
    finally:
        m.close()
    # from y = 0 the results are the deltas, which differ between the pools:
    # a replay against the old pool fails the second check
    delta_gate(got1, oracle.apply_workload(wl1, threads=0)[1])
    delta_gate(got2, oracle.apply_workload(wl2, threads=0)[1])


def test_host_entry_point_buffer_unpinned_between_calls():
    """x is page-locked in place for the first calls (eager, captured with the
    copy kernels, replayed), then unlocked at the same address: the next call
    must see that the GPU no longer addresses it and run with copy calls."""
    cudart = torch.cuda.cudart()
    wl = W.distinct_decode()
    dw = DeviceWorkload(wl)
    x_host = torch.from_numpy(wl.x.view(np.int16).copy())
    nbytes = x_host.numel() * x_host.element_size()
    assert int(cudart.cudaHostRegister(x_host.data_ptr(), nbytes, 0)) == 0
    state = {"registered": True}

    def unpin_at_fourth(it):
        if it == 3:
            assert int(cudart.cudaHostUnregister(x_host.data_ptr())) == 0
            state["registered"] = False

    try:
        _host_calls(wl, dw, x_host, torch.empty(wl.y.shape, dtype=torch.int16).pin_memory(),
                    torch.from_numpy(wl.offsets).pin_memory(), torch.from_numpy(wl.ids).pin_memory(),
                    torch.from_numpy(wl.alpha).pin_memory(), 6, before_call=unpin_at_fourth)
    finally:
        if state["registered"]:
            cudart.cudaHostUnregister(x_host.data_ptr())
        dw.close()


# ---------------------------------------------------------------- edge shapes
def _custom(rng, d_in, d_out, r, cap, lists, ranks=None):
    alpha_lists = [list(rng.random(len(l)).astype(np.float32)) for l in lists]
    return W.make_custom(rng, d_in=d_in, d_out=d_out, r_max=r, capacity=cap, id_lists=lists,
                         alpha_lists=alpha_lists, ranks=ranks, y_sigma=0.0)


@pytest.mark.parametrize("path", [PATH_AUTO, PATH_MMA, PATH_SPLIT])
@pytest.mark.parametrize("ntok", [300, 200])
def test_big_segments_and_many_pairs_per_token(ntok, path):
    """Segments far longer than a shrink tile or an expand job, one token with
    40 pairs, an empty token; 200 tokens also runs the fused path."""
    rng = np.random.default_rng(21)
    lists = [[0, 1, 2] for _ in range(ntok)] + [list(rng.permutation(64)[:40])] + [[]] + [[5]]
    wl = _custom(rng, 128, 192, 16, 64, lists)
    y, st = run_gpu(wl, path=path)
    _, acc, _ = oracle.apply_workload(wl)
    assert st == 0
    delta_gate(y, acc)


@pytest.mark.parametrize("path", ALL_PATHS)
@pytest.mark.parametrize("d_in,d_out,r,k", [(64, 128, 1, 1), (6208, 64, 5, 3), (14336, 4096, 8, 8),
                                            (256, 256, 64, 64), (192, 320, 13, 7)])
def test_shapes(d_in, d_out, r, k, path):
    rng = np.random.default_rng(d_in + d_out)
    cap = 6
    lists = [list(rng.permutation(cap)[:rng.integers(1, 4)]) for _ in range(9)]
    ranks = np.full(cap, k, np.int32)
    ranks[0] = 0
    wl = _custom(rng, d_in, d_out, r, cap, lists, ranks)
    y, st = run_gpu(wl, path=path)
    _, acc, _ = oracle.apply_workload(wl)
    delta_gate(y, acc)


@pytest.mark.parametrize("path", [PATH_AUTO, PATH_DECODE, PATH_FUSED])
def test_decode_many_tokens_rank64_wide(path):
    """256 tokens x 3 adapters of 1000 at rank 64 and a wide output (the
    largest decode batch: more (token, column) items than a wave of warps,
    the wide-rank expand, every row of every adapter)."""
    rng = np.random.default_rng(44)
    lists = [list(rng.choice(1000, size=3, replace=False)) for _ in range(256)]
    wl = W.make_custom(rng, d_in=256, d_out=4096, r_max=64, capacity=1000, id_lists=lists,
                       alpha_lists=[list(rng.random(3).astype(np.float32)) for _ in lists], y_sigma=0.0)
    y, st = run_gpu(wl, path=path)
    _, acc, _ = oracle.apply_workload(wl, threads=0)
    assert st == 0
    delta_gate(y, acc)


def test_mma_many_adapters_and_pairs_per_tile():
    """Tensor-core path: a 128-token tile whose pairs name more adapters than
    one listing window holds (8 distinct of 2048 per token) and more pairs
    than the tile's pair cache; duplicates of one adapter within a token;
    token tiles with no pair; a ragged last tile."""
    rng = np.random.default_rng(33)
    cap = 2048
    lists = [list(rng.permutation(cap)[:8]) for _ in range(130)]
    lists += [[] for _ in range(140)]
    lists += [[7, 7, 9] for _ in range(3)]
    wl = _custom(rng, 64, 128, 4, cap, lists)
    for path in (PATH_MMA, PATH_SPLIT):
        y, st = run_gpu(wl, path=path)
        _, acc, _ = oracle.apply_workload(wl)
        assert st == 0
        delta_gate(y, acc)


def test_no_pairs_leaves_y():
    rng = np.random.default_rng(2)
    wl = W.make_custom(rng, d_in=64, d_out=64, r_max=4, capacity=2, id_lists=[[], []],
                       alpha_lists=[[], []])
    y, st = run_gpu(wl)
    np.testing.assert_array_equal(y, wl.y)


def _large_batch():
    """12000 tokens with 1-4 pairs each (about 30000 pairs), ranks 1..16 over
    a pool of 64: more than the mapping stages stage in shared memory, so the
    CSR stage and the sort run their global-memory forms."""
    rng = np.random.default_rng(41)
    T, cap = 12000, 64
    counts = rng.integers(1, 5, size=T)
    lists = [[int(v) for v in rng.choice(cap, size=int(c), replace=False)] for c in counts]
    alphas = [list(rng.random(len(l)).astype(np.float32)) for l in lists]
    ranks = rng.integers(1, 17, size=cap).astype(np.int32)
    return W.make_custom(rng, d_in=256, d_out=256, r_max=16, capacity=cap, id_lists=lists, alpha_lists=alphas,
                         ranks=ranks, y_sigma=0.0, name="large_batch")


def test_large_batch_mapping_bit_exact():
    wl = _large_batch()
    assert (wl.offsets.size - 1) + 1 + 2 * wl.ids.size > 51200  # beyond the staged CSR form
    dw = DeviceWorkload(wl)
    try:
        got = dw.mapping.export()
    finally:
        dw.close()
    compare_mapping(got, oracle.build_mapping(wl.offsets, wl.ids, wl.alpha, capacity=wl.capacity))


@pytest.mark.parametrize("path", [PATH_AUTO, PATH_MMA, PATH_SPLIT, PATH_DECODE])
def test_large_batch_every_token(path):
    """Every token of the large batch against the fp64 oracle (y = 0, so the
    delta-only bound applies)."""
    wl = _large_batch()
    y, st = run_gpu(wl, path=path)
    assert st == 0
    _, acc, _ = oracle.apply_workload(wl, threads=0)
    delta_gate(y, acc)
