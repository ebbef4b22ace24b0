"""Seeded synthetic inputs for the composite multi-LoRA delta.

This module only draws numbers.  It holds none of the delta's arithmetic: it
produces per-token pair lists (CSR offsets, adapter ids, weights alpha), the
activations x, the adapter factors A and B, the retained ranks k and the
incoming y.  The same arrays feed the fp64 oracle and the CUDA path.

Workload shapes follow the pages' serving experiments (DyMerge-LoRA, "What
they did": Single / Distinct / Skewed(Zipf) / Sparse adapter assignment, bf16,
rank-8 LoRA on every dense projection of Llama-3; LoRAForge, "Approach": a
retained effective rank k_m per module).  The pages measure on ShareGPT
lengths with randomly initialised LoRA weights; these seeded draws stand in
for both.

Draw order per workload (one ``numpy.random.default_rng(seed)`` stream):
  1. structure: retained ranks (rank sweep only), per-token pair counts,
     adapter ids, alpha;
  2. x;
  3. A then B, for each adapter in id order;
  4. y.
Normals are drawn in fp32 with the stated standard deviation and rounded to
bf16 with round-to-nearest-even.

Layouts (all C-contiguous numpy arrays):
  offsets int32 [T+1]       CSR row pointer of each token's pair list
  ids     int32 [P]         adapter id of each pair, CSR order
  alpha   float32 [P]       weight of each pair
  x       uint16 [T, d_in]  bf16 bit patterns
  A       uint16 [cap, d_in, r_max]   A_i in R^{d_in x r}
  B       uint16 [cap, r_max, d_out]  B_i in R^{r x d_out}
  ranks   int32 [cap]       retained rank k_i (0..r_max)
  y       uint16 [T, d_out] incoming y, bf16 bit patterns
"""
from __future__ import annotations

import dataclasses
import numpy as np

SIGMA = 0.02


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits.

    Input generation only: finite values are assumed (normal draws)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Workload:
    name: str
    d_in: int
    d_out: int
    r_max: int
    capacity: int
    offsets: np.ndarray
    ids: np.ndarray
    alpha: np.ndarray
    x: np.ndarray
    A: np.ndarray
    B: np.ndarray
    ranks: np.ndarray
    y: np.ndarray
    note: str = ""

    @property
    def T(self) -> int:
        return int(self.offsets.shape[0] - 1)

    @property
    def P(self) -> int:
        return int(self.ids.shape[0])


def _normal_bf16(rng, shape, sigma):
    v = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        v = v * np.float32(sigma)
    return f32_to_bf16_bits(v)


def _zipf_probs(n: int, s: float) -> np.ndarray:
    # P(rank k) proportional to k^-s over k = 1..n; id = k - 1.
    k = np.arange(1, n + 1, dtype=np.float64)
    w = k ** (-s)
    return w / w.sum()


def _draw_distinct(rng, probs: np.ndarray, m: int) -> list[int]:
    """Sequential draws from ``probs``, rejecting ids already drawn."""
    out: list[int] = []
    while len(out) < m:
        v = int(rng.choice(probs.shape[0], p=probs))
        if v not in out:
            out.append(v)
    return out


def _factors(rng, cap, d_in, d_out, r_max, ranks, zero_padding: bool):
    A = np.empty((cap, d_in, r_max), dtype=np.uint16)
    B = np.empty((cap, r_max, d_out), dtype=np.uint16)
    for a in range(cap):
        A[a] = _normal_bf16(rng, (d_in, r_max), SIGMA)
        B[a] = _normal_bf16(rng, (r_max, d_out), SIGMA)
        if zero_padding:
            k = int(ranks[a])
            A[a, :, k:] = 0
            B[a, k:, :] = 0
    return A, B


def _csr(lists):
    counts = np.array([len(l) for l in lists], dtype=np.int64)
    offsets = np.zeros(len(lists) + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return offsets


def make_custom(rng, *, d_in, d_out, r_max, capacity, id_lists, alpha_lists,
                ranks=None, y_sigma=1.0, zero_padding=True, name="custom"):
    """Build a workload from explicit pair lists (draws x, A, B, y)."""
    if ranks is None:
        ranks = np.full(capacity, r_max, dtype=np.int32)
    ranks = np.asarray(ranks, dtype=np.int32)
    offsets = _csr(id_lists)
    ids = np.array([i for l in id_lists for i in l], dtype=np.int32)
    alpha = np.array([w for l in alpha_lists for w in l], dtype=np.float32)
    T = len(id_lists)
    x = _normal_bf16(rng, (T, d_in), SIGMA)
    A, B = _factors(rng, capacity, d_in, d_out, r_max, ranks, zero_padding)
    y = _normal_bf16(rng, (T, d_out), y_sigma) if y_sigma > 0 else np.zeros((T, d_out), np.uint16)
    return Workload(name, d_in, d_out, r_max, capacity, offsets, ids, alpha, x, A, B, ranks, y)


def tiny(seed: int = 0, y_zero: bool = False) -> Workload:
    """d_in = d_out = 256, r = k = 8, pool 16, 32 tokens, 1-3 distinct
    uniform adapters per token, alpha ~ U(0,1) normalised to sum 1."""
    rng = np.random.default_rng(seed)
    T, cap, d, r = 32, 16, 256, 8
    counts = rng.integers(1, 4, size=T)
    id_lists = [[int(v) for v in rng.choice(cap, size=int(m), replace=False)] for m in counts]
    raw = rng.random(int(counts.sum()))
    alpha_lists, p = [], 0
    for m in counts:
        w = raw[p:p + m]
        alpha_lists.append(list((w / w.sum()).astype(np.float32)))
        p += m
    wl = make_custom(rng, d_in=d, d_out=d, r_max=r, capacity=cap, id_lists=id_lists,
                     alpha_lists=alpha_lists, y_sigma=0.0 if y_zero else 1.0, name="tiny")
    return wl


def distinct_decode(seed: int = 0, capacity: int = 96, y_zero: bool = False) -> Workload:
    """Distinct decode, Llama-3-8B q_proj shape (4096 x 4096), r = k = 8,
    32 tokens, 3 adapters per token shared with no other token, alpha = 1/3.

    Three unshared adapters for each of 32 tokens need 96 slots, so the pool
    holds 96 adapters.  ``capacity=64`` gives the sensitivity variant in
    which tokens 21..31 reuse ids (not a config of its own)."""
    rng = np.random.default_rng(seed)
    T, d, r = 32, 4096, 8
    perm = rng.permutation(max(capacity, 96))
    if capacity < 96:
        perm = perm % capacity
    id_lists = [[int(v) for v in perm[3 * t:3 * t + 3]] for t in range(T)]
    alpha_lists = [[np.float32(1.0 / 3.0)] * 3 for _ in range(T)]
    wl = make_custom(rng, d_in=d, d_out=d, r_max=r, capacity=capacity, id_lists=id_lists,
                     alpha_lists=alpha_lists, y_sigma=0.0 if y_zero else 1.0,
                     name="distinct_decode_q_proj")
    return wl


def zipf_decode(seed: int = 0, y_zero: bool = False) -> Workload:
    """Zipf-skewed decode, gate_proj shape (4096 -> 14336), r = k = 8, pool
    128, 64 tokens, 2-4 distinct ids per token drawn from Zipf(1.5) with
    repeats rejected, alpha ~ Dirichlet(1) (normalised Exp(1))."""
    rng = np.random.default_rng(seed)
    T, cap, r = 64, 128, 8
    probs = _zipf_probs(cap, 1.5)
    counts = rng.integers(2, 5, size=T)
    id_lists = [_draw_distinct(rng, probs, int(m)) for m in counts]
    alpha_lists = []
    for m in counts:
        e = rng.exponential(1.0, size=int(m))
        alpha_lists.append(list((e / e.sum()).astype(np.float32)))
    return make_custom(rng, d_in=4096, d_out=14336, r_max=r, capacity=cap, id_lists=id_lists,
                       alpha_lists=alpha_lists, y_sigma=0.0 if y_zero else 1.0,
                       name="zipf_decode_gate_proj")


def sparse_prefill(seed: int = 0, y_zero: bool = False, n_requests: int = 16,
                   d: int = 4096) -> Workload:
    """Sparse MoE-LoRA prefill, 4096 x 4096, r = k = 16, pool 64.  16
    requests of length clip(round(lognormal(5.3, 0.8)), 16, 1024), laid out
    request-contiguous; each request references 8 distinct uniform ids; each
    token keeps the top-2 of softmax(N(0,1)^8) gate logits (ties to the lower
    list index), alpha renormalised over the two."""
    rng = np.random.default_rng(seed)
    cap, r = 64, 16
    lens = np.clip(np.round(rng.lognormal(5.3, 0.8, size=n_requests)), 16, 1024).astype(int)
    req_ids = [rng.choice(cap, size=8, replace=False) for _ in range(n_requests)]
    id_lists, alpha_lists = [], []
    for q in range(n_requests):
        logits = rng.standard_normal(size=(int(lens[q]), 8))
        for row in logits:
            e = np.exp(row - row.max())
            prob = e / e.sum()
            order = np.argsort(-prob, kind="stable")[:2]
            p1, p2 = prob[order[0]], prob[order[1]]
            id_lists.append([int(req_ids[q][order[0]]), int(req_ids[q][order[1]])])
            alpha_lists.append([np.float32(p1 / (p1 + p2)), np.float32(p2 / (p1 + p2))])
    wl = make_custom(rng, d_in=d, d_out=d, r_max=r, capacity=cap, id_lists=id_lists,
                     alpha_lists=alpha_lists, y_sigma=0.0 if y_zero else 1.0,
                     name="sparse_moe_prefill")
    wl.note = f"{n_requests} requests, lengths {lens.tolist()}"
    return wl


def rank_sweep(T: int, seed: int = 0, y_zero: bool = False, garbage_padding: bool = False,
               capacity: int = 1000) -> Workload:
    """Heterogeneous retained rank, k/v_proj GQA shape (4096 -> 1024), pool
    1000 padded to r_max = 64, k_i ~ U{1..64} with factor entries beyond k_i
    zero (``garbage_padding`` keeps them random instead), T decode tokens,
    1-3 distinct ids per token from Zipf(1.2), alpha ~ U(0,1) unnormalised."""
    rng = np.random.default_rng(seed)
    r = 64
    ranks = rng.integers(1, r + 1, size=capacity).astype(np.int32)
    probs = _zipf_probs(capacity, 1.2)
    counts = rng.integers(1, 4, size=T)
    id_lists = [_draw_distinct(rng, probs, int(m)) for m in counts]
    alpha_lists = [list(rng.random(int(m)).astype(np.float32)) for m in counts]
    wl = make_custom(rng, d_in=4096, d_out=1024, r_max=r, capacity=capacity, id_lists=id_lists,
                     alpha_lists=alpha_lists, ranks=ranks, y_sigma=0.0 if y_zero else 1.0,
                     zero_padding=not garbage_padding, name=f"rank_sweep_T{T}")
    return wl


CONFIGS = {
    "tiny": lambda **kw: tiny(**kw),
    "distinct": lambda **kw: distinct_decode(**kw),
    "zipf": lambda **kw: zipf_decode(**kw),
    "prefill": lambda **kw: sparse_prefill(**kw),
    "sweep1": lambda **kw: rank_sweep(1, **kw),
    "sweep8": lambda **kw: rank_sweep(8, **kw),
    "sweep64": lambda **kw: rank_sweep(64, **kw),
    "sweep256": lambda **kw: rank_sweep(256, **kw),
}


def make(name: str, **kw) -> Workload:
    return CONFIGS[name](**kw)


def algorithmic_bytes(wl: Workload, ranks=None) -> dict:
    """Bytes the delta must move once: x read, y read + written, each distinct
    adapter's retained A and B rows once, and the pair lists (12 B/pair +
    4 B/token).  bf16 = 2 bytes."""
    ranks = wl.ranks if ranks is None else ranks
    used = np.unique(wl.ids[(wl.ids >= 0) & (wl.ids < wl.capacity)])
    sum_k = int(np.clip(ranks[used], 0, wl.r_max).sum()) if used.size else 0
    b = {
        "x": wl.T * wl.d_in * 2,
        "y": 2 * wl.T * wl.d_out * 2,
        "adapters": sum_k * (wl.d_in + wl.d_out) * 2,
        "mapping": wl.P * 12 + (wl.T + 1) * 4,
        "U": int(used.size),
        "sum_k": sum_k,
    }
    b["total"] = b["x"] + b["y"] + b["adapters"] + b["mapping"]
    return b
