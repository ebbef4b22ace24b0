"""fp64 oracle for batched LoRA recompression (FlashTSQR factor construction)
and retained-rank allocation.

TEST INFRASTRUCTURE ONLY (tests, smoke check, the benchmark's CPU leg);
nothing in the product imports it.

LoRAForge summary page, "Key contributions" and "Approach" (2)-(3):
  * factor construction: a thin QR of the tall-skinny factor gives R; with
    H = R B the spectrum of the module's update comes from the
    eigen-decomposition of H H^T, and balanced factors F, T whose first k
    directions reproduce the exact rank-k truncated SVD are formed;
  * FlashTSQR: each of the M factors is split into P row tiles, the M P leaf
    QRs run independently and their triangular factors are merged level by
    level (the Q factors are never formed);
  * rank allocation: LoRAForge-U keeps u_m = max(1, floor(r_m / d)) per
    module, which fixes the parameter budget; LoRAForge-S spends the same
    budget greedily by energy per parameter, eta = sigma^2 / (d_in + d_out),
    above a rank floor.

Row form as in the delta: dW = A B, A in R^{d_in x r}, B in R^{r x d_out};
the balanced factors are F (d_in x r) and T (r x d_out) with dW = F T.
numpy's QR and symmetric eigen-decomposition serve as steps (library
primitives); everything around them is written out.
"""
from __future__ import annotations

import numpy as np


def _r_positive(r: np.ndarray) -> np.ndarray:
    """R with a non-negative diagonal (flip the sign of each negative row)."""
    s = np.where(np.diag(r) < 0, -1.0, 1.0)
    return r * s[:, None]


def tsqr_r(a: np.ndarray, tiles: int) -> np.ndarray:
    """R of the thin QR of a (n x r, n >= r) by the tall-skinny tree: `tiles`
    row tiles (each at least r rows), a QR per tile, then pairwise merges of
    the stacked triangular factors, level by level (a power-of-two count)."""
    a = np.asarray(a, np.float64)
    n, r = a.shape
    assert tiles >= 1 and tiles & (tiles - 1) == 0 and n % tiles == 0 and n // tiles >= r
    h = n // tiles
    rs = [np.linalg.qr(a[p * h:(p + 1) * h], mode="r") for p in range(tiles)]
    while len(rs) > 1:
        rs = [np.linalg.qr(np.vstack([rs[i], rs[i + 1]]), mode="r") for i in range(0, len(rs), 2)]
    return _r_positive(rs[0])


def balanced_factors(a: np.ndarray, b: np.ndarray, rel_floor: float = 1e-6):
    """(sigma [r] descending, F [d_in x r], T [r x d_out]) with F T = A B,
    F^T F = diag(sigma) = T T^T, and F[:, :k] T[:k] the rank-k truncated
    SVD.  Directions with sigma <= rel_floor * sigma_0 are dead (zero)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    q, r = np.linalg.qr(a, mode="reduced")
    s = np.where(np.diag(r) < 0, -1.0, 1.0)
    q, r = q * s[None, :], r * s[:, None]
    h = r @ b
    lam, u = np.linalg.eigh(h @ h.T)
    order = np.argsort(-lam, kind="stable")
    lam, u = lam[order], u[:, order]
    sigma = np.sqrt(np.clip(lam, 0.0, None))
    live = sigma > rel_floor * (sigma[0] if sigma.size else 0.0)
    f = np.zeros((a.shape[0], r.shape[1]))
    t = np.zeros((r.shape[1], b.shape[1]))
    for j in range(sigma.size):
        if live[j]:
            f[:, j] = (q @ u[:, j]) * np.sqrt(sigma[j])
            t[j, :] = (u[:, j] @ h) / np.sqrt(sigma[j])
    sigma = np.where(live, sigma, 0.0)
    return sigma, f, t


def rank_allocate(sigma, cost, rank, policy: str, d: int, floor: int = 1):
    """Retained ranks k_m for modules with singular values sigma[m] (sorted
    descending; zeros are dead directions), per-direction parameter cost
    cost[m] = d_in + d_out and original rank rank[m].

    'U': k_m = min(max(1, floor(r_m / d)), live directions).
    'S': the budget of 'U' (sum of k_m * cost_m) spent greedily: every module
         first keeps min(floor, live) directions; the remaining directions
         (m, j) are visited by eta = sigma^2 / cost descending (ties: lower m,
         then lower j) and taken when j is the module's next direction and its
         cost still fits the budget."""
    sigma = [np.asarray(s, np.float64) for s in sigma]
    M = len(sigma)
    live = [int(np.count_nonzero(s > 0)) for s in sigma]
    uni = [min(max(1, int(rank[m]) // d), live[m]) for m in range(M)]
    if policy == "U":
        return uni
    budget = sum(uni[m] * int(cost[m]) for m in range(M))
    k = [min(floor, live[m]) for m in range(M)]
    spent = sum(k[m] * int(cost[m]) for m in range(M))
    cand = [(-(sigma[m][j] ** 2) / cost[m], m, j) for m in range(M) for j in range(k[m], live[m])]
    cand.sort()
    for _, m, j in cand:
        if j == k[m] and spent + cost[m] <= budget:
            k[m] += 1
            spent += cost[m]
    return k
