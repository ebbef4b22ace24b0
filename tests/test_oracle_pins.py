"""Pins for the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself:
  - the worked example the ELORA page prints (Sec. 1.4, table 1.4.2);
  - the post-merge = pre-merge identity (DyMerge-LoRA page, "Core idea",
    paper Sec. 3.1 M1 and Sec. 5.4): y' = y + x (sum_i alpha_i A_i B_i), formed
    explicitly with numpy;
  - exact rational arithmetic (Fractions) and an exact round-to-nearest-even on
    tiny dyadic inputs, exhaustive over a small alpha grid;
  - linearity in alpha, invariance to pair order, alpha = 0 and k = 0 no-ops;
  - the rank bound rank(sum alpha A B) <= sum k (DyMerge-LoRA page, "Core
    idea", paper Figure 4) on the linear map the oracle applies;
  - the retained-rank prefix contract (LoRAForge page, "Approach" (1)):
    garbage beyond k_i changes nothing;
  - the mapping against Python's sort and numpy's stable argsort.
"""
import itertools
import json
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as W
from workloads import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def exact_rne_bf16(v: Fraction) -> int:
    """Exact nearest-even bf16 bits of a rational (written independently of
    the oracle's C rounding)."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** (e - 1) > a:
        e -= 1
    while a >= Fraction(2) ** e:
        e += 1
    q = max(e - 8, -133)
    scaled = a / Fraction(2) ** q
    r = scaled.numerator // scaled.denominator
    rem = scaled - r
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and r % 2 == 1):
        r += 1
    val = r * Fraction(2) ** q
    if val >= Fraction(2) ** 128:
        return sign | 0x7F80
    bits = struct.unpack("<I", struct.pack("<f", float(val)))[0]
    return sign | ((bits >> 16) & 0x7FFF)


def bits_of(vals):
    return f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def run(offsets, ids, alpha, x, A, B, ranks, y, **kw):
    cap, d_in, r = A.shape
    d_out = B.shape[2]
    return oracle.delta_apply(offsets, ids, alpha, x, A, B, ranks, y, d_in=d_in, d_out=d_out,
                              r_max=r, capacity=cap, **kw)


def premerge_reference(wl, tokens, ranks=None):
    """y_in + x_t (sum_p alpha_p A_a[:, :k] B_a[:k, :]) with the update matrix
    formed explicitly in fp64; also returns the absolute-value scale."""
    ranks = wl.ranks if ranks is None else ranks
    x = bf16_bits_to_f32(wl.x).astype(np.float64)
    y = bf16_bits_to_f32(wl.y).astype(np.float64)
    out, scale = [], []
    for t in tokens:
        dW = np.zeros((wl.d_in, wl.d_out))
        absW = np.zeros((wl.d_in, wl.d_out))
        for p in range(wl.offsets[t], wl.offsets[t + 1]):
            a = int(wl.ids[p])
            k = int(ranks[a])
            Aa = bf16_bits_to_f32(wl.A[a][:, :k]).astype(np.float64)
            Ba = bf16_bits_to_f32(wl.B[a][:k, :]).astype(np.float64)
            dW += float(wl.alpha[p]) * (Aa @ Ba)
            absW += abs(float(wl.alpha[p])) * (np.abs(Aa) @ np.abs(Ba))
        out.append(y[t] + x[t] @ dW)
        scale.append(np.abs(y[t]) + np.abs(x[t]) @ absW)
    return np.array(out), np.array(scale)


# ---------------------------------------------------------------- worked example
def test_elora_worked_example():
    """K = (W_K + A B) h for the two LoRAs of the ELORA page, through the row
    form y = x + (x A') B' with A' = B^T, B' = A^T (W_K = I, so y_in = h)."""
    g = json.load(open(os.path.join(GOLDEN, "elora_kv_example.json")))
    h = np.array(g["h"], dtype=np.float32)
    assert np.array_equal(np.array(g["W_K"]), np.eye(2))
    loras = [c for c in g["cases"] if c["A"] is not None]
    cap, d, r = len(loras), 2, 1
    A = np.zeros((cap, d, r), np.uint16)
    B = np.zeros((cap, r, d), np.uint16)
    for i, c in enumerate(loras):
        A[i] = bits_of(np.array(c["B"], dtype=np.float32).T)   # A' = B^T (d x r)
        B[i] = bits_of(np.array(c["A"], dtype=np.float32).T)   # B' = A^T (r x d)
    base = [c for c in g["cases"] if c["A"] is None][0]
    # tokens: base only, LoRA-1, LoRA-2, and the derived composite 1/2 + 1/2
    offsets = np.array([0, 0, 1, 2, 4], np.int32)
    ids = np.array([0, 1, 0, 1], np.int32)
    alpha = np.array([1.0, 1.0, 0.5, 0.5], np.float32)
    x = np.tile(bits_of(h), (4, 1))
    y_in = x.copy()
    ranks = np.array([1, 1], np.int32)
    y, acc, st = run(offsets, ids, alpha, x, A, B, ranks, y_in)
    assert st == 0
    got = bf16_bits_to_f32(y)
    np.testing.assert_array_equal(got[0], base["K"])
    np.testing.assert_array_equal(got[1], loras[0]["K"])
    np.testing.assert_array_equal(got[2], loras[1]["K"])
    # derived: K = h + (K1 - h)/2 + (K2 - h)/2 = [2, 2.5], exact in bf16
    np.testing.assert_array_equal(got[3], [2.0, 2.5])


# ---------------------------------------------------------------- rounding
@pytest.mark.parametrize("v", [
    1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1 + 2 ** -8 + 2 ** -40, 3.0, -0.0078125,
    2 ** -126, 2 ** -133, 2 ** -134, 3 * 2 ** -134, 1.5 * 2 ** -133, 2 ** -140,
    255 * 2 ** 120, 255.5 * 2 ** 120, 255.25 * 2 ** 120, 1e-3, -123.456, 2.0 ** 127 * 1.99,
])
def test_round_bf16_exact(v):
    assert oracle.round_bf16(v) == exact_rne_bf16(Fraction(v))


def test_round_bf16_random():
    rng = np.random.default_rng(7)
    for v in np.concatenate([rng.standard_normal(300), rng.standard_normal(100) * 1e-38,
                             rng.standard_normal(100) * 1e30]):
        assert oracle.round_bf16(float(v)) == exact_rne_bf16(Fraction(float(v)))


# ---------------------------------------------------------------- brute force
def _dyadic_case(rng, T, cap, d_in, d_out, r, ranks, lists):
    def grid(shape):  # multiples of 1/8 in [-2, 2]: exact in bf16 and in fp64 sums
        return (rng.integers(-16, 17, size=shape) / 8.0).astype(np.float32)
    x = bits_of(grid((T, d_in)))
    A = bits_of(grid((cap, d_in, r)))
    B = bits_of(grid((cap, r, d_out)))
    y = bits_of(grid((T, d_out)) * 64)
    offsets = np.zeros(T + 1, np.int32)
    offsets[1:] = np.cumsum([len(l) for l in lists])
    ids = np.array([i for l in lists for i in l], np.int32)
    return x, A, B, y, offsets, ids


def _exact(x, A, B, y, offsets, ids, alpha, ranks):
    T, d_in = x.shape
    d_out = y.shape[1]
    xf, Af, Bf, yf = (bf16_bits_to_f32(v) for v in (x, A, B, y))
    out = []
    for t in range(T):
        acc = [Fraction(float(v)) for v in yf[t]]
        for p in range(offsets[t], offsets[t + 1]):
            a, k, al = int(ids[p]), int(ranks[ids[p]]), Fraction(float(alpha[p]))
            z = [sum(Fraction(float(xf[t, d])) * Fraction(float(Af[a, d, j])) for d in range(d_in))
                 for j in range(k)]
            for c in range(d_out):
                acc[c] += al * sum(z[j] * Fraction(float(Bf[a, j, c])) for j in range(k))
        out.append(acc)
    return out


def test_bruteforce_exhaustive_alpha_grid():
    """All-pairs loops in exact rationals on d <= 16, pool 4, T = 2, every k
    in 0..r over the pool, and every alpha from a small dyadic grid on each
    of the four pairs: the oracle must equal the exact nearest-even result."""
    rng = np.random.default_rng(1)
    T, cap, d_in, d_out, r = 2, 4, 12, 16, 3
    lists = [[2, 0], [1, 3]]
    ranks = np.array([0, 1, 2, 3], np.int32)
    x, A, B, y, offsets, ids = _dyadic_case(rng, T, cap, d_in, d_out, r, ranks, lists)
    grid = [0.0, 0.5, -1.0, 0.75]
    for combo in itertools.product(grid, repeat=4):
        alpha = np.array(combo, np.float32)
        yo, acc, st = run(offsets, ids, alpha, x, A, B, ranks, y)
        assert st == 0
        ex = _exact(x, A, B, y, offsets, ids, alpha, ranks)
        for t in range(T):
            for c in range(d_out):
                assert acc[t, c] == float(ex[t][c])           # exact: dyadic inputs
                assert yo[t, c] == exact_rne_bf16(ex[t][c])


def test_bruteforce_random_alpha():
    rng = np.random.default_rng(2)
    T, cap, d_in, d_out, r = 4, 4, 16, 8, 4
    lists = [[0], [1, 2, 3], [3, 1], []]
    ranks = np.array([4, 2, 3, 1], np.int32)
    x, A, B, y, offsets, ids = _dyadic_case(rng, T, cap, d_in, d_out, r, ranks, lists)
    alpha = rng.random(len(ids)).astype(np.float32)
    yo, acc, st = run(offsets, ids, alpha, x, A, B, ranks, y)
    ex = _exact(x, A, B, y, offsets, ids, alpha, ranks)
    for t in range(T):
        for c in range(d_out):
            e = ex[t][c]
            assert abs(Fraction(acc[t, c]) - e) <= Fraction(1, 2 ** 40) * (1 + abs(e))
            if yo[t, c] != exact_rne_bf16(e):  # only possible right at a tie
                lo = exact_rne_bf16(e)
                assert abs(int(yo[t, c]) - lo) == 1


# ---------------------------------------------------------------- pre-merge identity
@pytest.mark.parametrize("name,tokens", [
    ("tiny", None), ("distinct", [0, 7, 31]), ("zipf", [0, 13, 63]), ("sweep8", None),
])
def test_premerge_identity(name, tokens):
    wl = W.make(name)
    tokens = list(range(wl.T)) if tokens is None else tokens
    y, acc, st = oracle.apply_tokens(wl, tokens)
    assert st == 0
    ref, scale = premerge_reference(wl, tokens)
    assert np.all(np.abs(acc - ref) <= 1e-12 * scale + 1e-300)
    # and the delta is not vacuous
    assert np.max(np.abs(ref - bf16_bits_to_f32(wl.y[tokens]))) > 1e-4


def test_premerge_identity_prefill_sampled():
    wl = W.sparse_prefill(n_requests=3)
    tokens = [0, 5, wl.T // 2, wl.T - 1]
    y, acc, st = oracle.apply_tokens(wl, tokens)
    ref, scale = premerge_reference(wl, tokens)
    assert st == 0 and np.all(np.abs(acc - ref) <= 1e-12 * scale)


def test_single_adapter_is_xAB():
    """One pair, alpha = 1, k = r: the delta is the textbook product x A B.
    Small-integer inputs make every value exact."""
    rng = np.random.default_rng(3)
    d_in, d_out, r = 24, 40, 5
    xi = rng.integers(-3, 4, size=(1, d_in)).astype(np.float32)
    Ai = rng.integers(-3, 4, size=(d_in, r)).astype(np.float32)
    Bi = rng.integers(-3, 4, size=(r, d_out)).astype(np.float32)
    y0 = np.zeros((1, d_out), np.float32)
    yo, acc, st = run(np.array([0, 1], np.int32), np.array([0], np.int32),
                      np.array([1.0], np.float32), bits_of(xi), bits_of(Ai)[None],
                      bits_of(Bi)[None], np.array([r], np.int32), bits_of(y0))
    np.testing.assert_array_equal(acc, (xi.astype(np.int64) @ Ai.astype(np.int64)
                                        @ Bi.astype(np.int64)).astype(np.float64))


# ---------------------------------------------------------------- linearity / order / no-ops
def test_linearity_in_alpha():
    wl = W.tiny(y_zero=True)
    _, a1, _ = oracle.apply_workload(wl)
    wl2 = W.tiny(y_zero=True)
    wl2.alpha = (wl.alpha * np.float32(2.0)).astype(np.float32)
    _, a2, _ = oracle.apply_workload(wl2)
    np.testing.assert_array_equal(a2, 2.0 * a1)  # power-of-two scaling is exact
    rng = np.random.default_rng(4)
    al1 = rng.random(wl.P).astype(np.float32)
    al2 = rng.random(wl.P).astype(np.float32)
    wl3 = W.tiny(y_zero=True)
    wl3.alpha = al1
    _, b1, _ = oracle.apply_workload(wl3)
    wl3.alpha = al2
    _, b2, _ = oracle.apply_workload(wl3)
    s = (al1.astype(np.float64) + al2.astype(np.float64))
    wl3.alpha = s.astype(np.float32)
    exact_sum = np.all(s.astype(np.float32).astype(np.float64) == s)
    _, b12, _ = oracle.apply_workload(wl3)
    tol = 1e-12 * (np.abs(b1) + np.abs(b2)).max()
    if exact_sum:
        assert np.max(np.abs(b12 - (b1 + b2))) <= tol
    else:  # fp32 alpha rounding: within one fp32 ulp of alpha
        assert np.max(np.abs(b12 - (b1 + b2))) <= 1e-6 * (np.abs(b1) + np.abs(b2)).max()


def test_order_invariance():
    wl = W.zipf_decode()
    tokens = list(range(0, wl.T, 5))
    y, acc, _ = oracle.apply_tokens(wl, tokens)
    rng = np.random.default_rng(5)
    for t in range(wl.T):
        a, b = wl.offsets[t], wl.offsets[t + 1]
        perm = rng.permutation(b - a) + a
        wl.ids[a:b] = wl.ids[perm]
        wl.alpha[a:b] = wl.alpha[perm]
    y2, acc2, _ = oracle.apply_tokens(wl, tokens)
    ref, scale = premerge_reference(wl, tokens)
    assert np.all(np.abs(acc2 - acc) <= 1e-12 * scale)


def test_noops_alpha_zero_and_rank_zero():
    wl = W.tiny()
    wl.alpha[:] = 0.0
    y, acc, st = oracle.apply_workload(wl)
    assert st == 0
    np.testing.assert_array_equal(bf16_bits_to_f32(y), bf16_bits_to_f32(wl.y))
    wl = W.tiny()
    y, acc, st = oracle.apply_workload(wl, ranks=np.zeros(wl.capacity, np.int32))
    assert st == 0
    np.testing.assert_array_equal(bf16_bits_to_f32(y), bf16_bits_to_f32(wl.y))


def test_rank_bound_on_applied_map():
    """The oracle's map x -> y - y_in for a fixed pair list, probed on the
    basis vectors, is a d_in x d_out matrix of rank <= sum of k."""
    rng = np.random.default_rng(6)
    d, cap, r = 24, 4, 4
    ranks = np.array([1, 2, 3, 4], np.int32)
    A = f32_to_bf16_bits(rng.standard_normal((cap, d, r)).astype(np.float32))
    B = f32_to_bf16_bits(rng.standard_normal((cap, r, d)).astype(np.float32))
    for lst in ([0, 1], [1, 2], [0, 3], [0, 1, 2]):
        offsets = np.arange(d + 1, dtype=np.int32) * len(lst)
        ids = np.tile(np.array(lst, np.int32), d)
        alpha = np.tile(rng.random(len(lst)).astype(np.float32), d)
        x = bits_of(np.eye(d, dtype=np.float32))
        _, acc, _ = run(offsets, ids, alpha, x, A, B, ranks, np.zeros((d, d), np.uint16))
        sv = np.linalg.svd(acc, compute_uv=False)
        rank = int(np.sum(sv > sv[0] * 1e-10))
        assert rank == int(ranks[lst].sum())  # generic factors reach the bound


def test_prefix_contract_garbage_padding():
    zero = W.rank_sweep(8)
    garb = W.rank_sweep(8, garbage_padding=True)
    assert np.any(garb.A != zero.A)
    y0, a0, _ = oracle.apply_workload(zero)
    y1, a1, _ = oracle.apply_workload(garb)
    np.testing.assert_array_equal(a0, a1)
    np.testing.assert_array_equal(y0, y1)


def test_error_semantics():
    wl = W.tiny()
    base_y, base_acc, _ = oracle.apply_workload(wl)
    ranks = wl.ranks.copy()
    victim = int(wl.ids[0])
    ranks[victim] = -1                       # unregistered slot
    y, acc, st = oracle.apply_workload(wl, ranks=ranks)
    assert st & oracle.UNREGISTERED
    zero_k = wl.ranks.copy()
    zero_k[victim] = 0
    y0, acc0, _ = oracle.apply_workload(wl, ranks=zero_k)
    np.testing.assert_array_equal(acc, acc0)  # the pair contributes nothing
    ranks[victim] = wl.r_max + 1
    y, acc, st = oracle.apply_workload(wl, ranks=ranks)
    assert st & oracle.BAD_RANK
    np.testing.assert_array_equal(acc, acc0)
    ids = wl.ids.copy()
    ids[0] = wl.capacity
    y, acc, st = oracle.delta_apply(wl.offsets, ids, wl.alpha, wl.x, wl.A, wl.B, wl.ranks, wl.y,
                                    d_in=wl.d_in, d_out=wl.d_out, r_max=wl.r_max,
                                    capacity=wl.capacity)
    assert st & oracle.BAD_ID
    bad = wl.offsets.copy()
    bad[3] = bad[2] - 1
    y, acc, st = oracle.delta_apply(bad, wl.ids, wl.alpha, wl.x, wl.A, wl.B, wl.ranks, wl.y,
                                    d_in=wl.d_in, d_out=wl.d_out, r_max=wl.r_max,
                                    capacity=wl.capacity)
    assert st & oracle.BAD_OFFSETS
    np.testing.assert_array_equal(y, wl.y)


# ---------------------------------------------------------------- mapping
def _mapping_by_sorted(offsets, ids, alpha, cap):
    tok = np.repeat(np.arange(len(offsets) - 1), np.diff(offsets))
    valid = [p for p in range(len(ids)) if 0 <= ids[p] < cap]
    order = sorted(valid, key=lambda p: (int(ids[p]), p))
    return tok, order


def test_mapping_bruteforce_tiny():
    wl = W.tiny()
    ids = wl.ids.copy()
    ids[3] = -2
    ids[10] = wl.capacity  # out of range: left out
    m = oracle.build_mapping(wl.offsets, ids, wl.alpha, capacity=wl.capacity)
    tok, order = _mapping_by_sorted(wl.offsets, ids, wl.alpha, wl.capacity)
    assert m["status"] == oracle.BAD_ID
    assert list(m["src"]) == order
    assert list(m["tok"]) == [int(tok[p]) for p in order]
    assert list(m["adapter"]) == [int(ids[p]) for p in order]
    assert m["alpha"].tobytes() == wl.alpha[order].tobytes()
    for q, p in enumerate(order):
        assert m["pos"][p] == q
    assert m["pos"][3] == -1 and m["pos"][10] == -1
    seg = sorted(set(int(ids[p]) for p in order))
    assert list(m["seg_adapter"]) == seg
    counts = [sum(1 for p in order if ids[p] == a) for a in seg]
    assert list(np.diff(m["seg_start"])) == counts


@pytest.mark.parametrize("name", ["distinct", "zipf", "prefill", "sweep256"])
def test_mapping_stable_argsort(name):
    wl = W.make(name) if name not in ("sweep256",) else W.rank_sweep(256, capacity=1000)
    m = oracle.build_mapping(wl.offsets, wl.ids, wl.alpha, capacity=wl.capacity)
    order = np.argsort(wl.ids, kind="stable")
    tok = np.repeat(np.arange(wl.T), np.diff(wl.offsets))
    np.testing.assert_array_equal(m["src"], order)
    np.testing.assert_array_equal(m["tok"], tok[order])
    np.testing.assert_array_equal(m["adapter"], wl.ids[order])
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    np.testing.assert_array_equal(m["pos"], inv)
    u, c = np.unique(wl.ids, return_counts=True)
    np.testing.assert_array_equal(m["seg_adapter"], u)
    np.testing.assert_array_equal(np.diff(m["seg_start"]), c)


def test_mapping_bad_offsets_and_empty():
    m = oracle.build_mapping(np.array([0, 2, 1, 3], np.int32), np.array([0, 1, 2], np.int32),
                             np.ones(3, np.float32), capacity=4)
    assert m["status"] == oracle.BAD_OFFSETS and m["U"] == 0 and np.all(m["pos"] == -1)
    m = oracle.build_mapping(np.zeros(5, np.int32), np.zeros(0, np.int32),
                             np.zeros(0, np.float32), capacity=4)
    assert m["status"] == 0 and m["U"] == 0 and m["P_valid"] == 0


# ---------------------------------------------------------------- MoE-LoRA gating
def test_gate_topk_worked_examples():
    """Hand-worked cases (tests/golden/gate_examples.json): ties to the lower
    candidate, renormalisation over the kept pairs, masking of padding,
    tokens short of candidates."""
    import json
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "gate_examples.json")))
    for case in g["cases"]:
        off, ids, al, _ = oracle.gate_topk(np.array(case["logits"], np.float32), np.array(case["cand"], np.int32),
                                           case["top_k"])
        assert off.tolist() == [0, case["top_k"]], case["name"]
        assert ids.tolist() == case["ids"], case["name"]
        np.testing.assert_allclose(al, case["alpha"], rtol=1e-6, atol=1e-7, err_msg=case["name"])


def test_gate_topk_against_full_softmax_and_stable_sort():
    """Random padded candidate lists: the kept ids are those of a stable sort
    on the negated logits (numpy), and alpha equals the explicit softmax over
    all valid candidates divided by the kept mass (not the cancelled form the
    oracle uses)."""
    rng = np.random.default_rng(21)
    T, E, k = 400, 8, 3
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[::7, 2] = logits[::7, 5]  # exact ties
    cand = rng.integers(0, 50, size=(T, E)).astype(np.int32)
    cand[rng.random((T, E)) < 0.2] = -1
    off, ids, al, empty = oracle.gate_topk(logits, cand, k)
    assert off.tolist() == [t * k for t in range(T + 1)]
    n_empty = 0
    for t in range(T):
        valid = np.nonzero(cand[t] >= 0)[0]
        if valid.size == 0:
            n_empty += 1
            assert ids[t * k:(t + 1) * k].tolist() == [-1] * k
            continue
        order = valid[np.argsort(-logits[t, valid].astype(np.float64), kind="stable")]
        kept = order[:k]
        p = np.exp(logits[t, valid].astype(np.float64))
        p /= p.sum()
        pk = np.exp(logits[t, kept].astype(np.float64)) / np.exp(logits[t, valid].astype(np.float64)).sum()
        want_ids = list(cand[t, kept]) + [cand[t, kept[0]]] * (k - kept.size)
        want_al = list(pk / pk.sum()) + [0.0] * (k - kept.size)
        assert ids[t * k:(t + 1) * k].tolist() == want_ids
        np.testing.assert_allclose(al[t * k:(t + 1) * k], want_al, rtol=2e-7, atol=1e-8)
    assert empty == n_empty


def test_gate_logits_against_einsum():
    """The batched gate logits (a router per request) against numpy's einsum
    on the same bf16 values."""
    rng = np.random.default_rng(4)
    T, E, d, R = 37, 8, 96, 3
    x = W.f32_to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    Wg = W.f32_to_bf16_bits(rng.standard_normal((R, E, d)).astype(np.float32) * 0.1)
    req = rng.integers(0, R, size=T).astype(np.int32)
    got = oracle.gate_logits(x, Wg, req)
    xf = W.bf16_bits_to_f32(x).astype(np.float64)
    wf = W.bf16_bits_to_f32(Wg).astype(np.float64)
    want = np.einsum("td,ted->te", xf, wf[req])
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
