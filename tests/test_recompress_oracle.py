"""Pins of the recompression oracle (oracle/recompress.py) to what the
mathematics fixes: the tall-skinny tree's R against a library QR, the
balanced factors against the SVD (Eckart-Young truncation, balance, exact
reconstruction, dead directions of a padded factor), and the rank policies
against a hand-worked example and a brute-force optimum."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import recompress as RC

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("n,r,tiles", [(64, 8, 1), (256, 16, 4), (4096, 64, 16), (512, 64, 8)])
def test_tsqr_tree_matches_library_qr(n, r, tiles):
    rng = np.random.default_rng(n + r)
    a = rng.standard_normal((n, r))
    want = np.linalg.qr(a, mode="r")
    want = want * np.where(np.diag(want) < 0, -1.0, 1.0)[:, None]
    got = RC.tsqr_r(a, tiles)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-10 * np.abs(want).max())
    np.testing.assert_allclose(got.T @ got, a.T @ a, rtol=1e-10, atol=1e-9)


@pytest.mark.parametrize("d_in,d_out,r", [(256, 128, 8), (512, 1024, 16), (1024, 256, 64)])
def test_balanced_factors_are_the_truncated_svd(d_in, d_out, r):
    rng = np.random.default_rng(r)
    a = rng.standard_normal((d_in, r)) * 0.02
    b = rng.standard_normal((r, d_out)) * 0.02
    sigma, f, t = RC.balanced_factors(a, b)
    dw = a @ b
    u, s, vt = np.linalg.svd(dw, full_matrices=False)
    np.testing.assert_allclose(sigma, s[:r], rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(f @ t, dw, atol=1e-12 * np.abs(dw).max() * r)
    for k in (1, r // 2, r):
        trunc = (u[:, :k] * s[:k]) @ vt[:k]
        np.testing.assert_allclose(f[:, :k] @ t[:k], trunc, atol=1e-9 * np.abs(dw).max())
        # Eckart-Young: the residual is the energy of the dropped directions
        assert np.isclose(np.linalg.norm(dw - f[:, :k] @ t[:k]), np.sqrt(np.sum(s[k:] ** 2)), rtol=1e-6, atol=1e-12)
    np.testing.assert_allclose(f.T @ f, np.diag(sigma), atol=1e-10 * sigma[0])
    np.testing.assert_allclose(t @ t.T, np.diag(sigma), atol=1e-10 * sigma[0])


def test_padded_factor_has_dead_directions():
    """A factor pair padded beyond its retained rank k (columns of A and rows
    of B zero) has exactly k live directions."""
    rng = np.random.default_rng(3)
    a = rng.standard_normal((512, 16))
    b = rng.standard_normal((16, 256))
    a[:, 5:] = 0
    b[5:] = 0
    sigma, f, t = RC.balanced_factors(a, b)
    assert np.count_nonzero(sigma) == 5
    np.testing.assert_allclose(f @ t, a @ b, atol=1e-10 * np.abs(a @ b).max())


def test_rank_policies_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "rank_allocation_example.json")))
    args = (g["sigma"], g["cost"], g["rank"])
    assert RC.rank_allocate(*args, "U", g["d"], g["floor"]) == g["U"]
    assert RC.rank_allocate(*args, "S", g["d"], g["floor"]) == g["S"]


def test_spectral_policy_is_optimal_at_equal_costs():
    """With equal per-direction costs the greedy by energy keeps the largest
    singular values of the fleet, which no other prefix choice within the
    budget beats (brute force over every prefix choice)."""
    rng = np.random.default_rng(8)
    for trial in range(30):
        M, r, d = 3, 4, 2
        sigma = [np.sort(rng.random(r))[::-1] for _ in range(M)]
        cost = [6] * M
        k = RC.rank_allocate(sigma, cost, [r] * M, "S", d, floor=0)
        budget = sum(max(1, r // d) * cost[m] for m in range(M))
        best = max(sum(np.sum(sigma[m][:c[m]] ** 2) for m in range(M))
                   for c in itertools.product(range(r + 1), repeat=M)
                   if sum(c[m] * cost[m] for m in range(M)) <= budget)
        got = sum(np.sum(sigma[m][:k[m]] ** 2) for m in range(M))
        assert np.isclose(got, best), trial
        assert sum(k[m] * cost[m] for m in range(M)) <= budget


def test_spectral_policy_respects_floor_and_budget():
    rng = np.random.default_rng(9)
    M = 12
    sigma = [np.sort(rng.random(16) ** 3)[::-1] for _ in range(M)]
    cost = list(rng.integers(100, 1000, size=M))
    k_u = RC.rank_allocate(sigma, cost, [16] * M, "U", 4)
    k_s = RC.rank_allocate(sigma, cost, [16] * M, "S", 4, floor=2)
    assert k_u == [4] * M
    assert all(v >= 2 for v in k_s)
    assert sum(k * c for k, c in zip(k_s, cost)) <= sum(k * c for k, c in zip(k_u, cost))
