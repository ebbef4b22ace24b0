"""Batched recompression on the device (FlashTSQR factor construction)
against the fp64 oracle: singular values, the rank-k truncations F_k T_k of
the balanced factors (equal to the truncated SVD), their balance, dead
directions of padded factors; then recompressed factors with spectral
retained ranks serve the delta."""
import numpy as np
import pytest

import oracle
import workloads as W
from oracle import recompress as RC
from workloads import bf16_bits_to_f32
from workloads.device import bf16_tensor, bf16_to_numpy_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    from tenant_composite_lora_gb300 import build
    build.build()


def _fleet(rng, M, d_in, d_out, r, decay=0.9, pad=None):
    """Factor pairs whose product has a decaying spectrum, mixed so that the
    factors are not already orthogonal; optionally zero-padded beyond a
    retained rank."""
    A = np.empty((M, d_in, r), np.uint16)
    B = np.empty((M, r, d_out), np.uint16)
    for m in range(M):
        u, _ = np.linalg.qr(rng.standard_normal((d_in, r)))
        v, _ = np.linalg.qr(rng.standard_normal((d_out, r)))
        s = 0.02 * decay ** np.arange(r)
        mix = rng.standard_normal((r, r)) * 0.3 + np.eye(r)
        a = (u * np.sqrt(s)) @ mix
        b = np.linalg.solve(mix, (v * np.sqrt(s)).T)
        if pad is not None:
            a[:, pad[m]:] = 0
            b[pad[m]:] = 0
        A[m] = W.f32_to_bf16_bits(a.astype(np.float32))
        B[m] = W.f32_to_bf16_bits(b.astype(np.float32))
    return A, B


def _run(A, B):
    import tenant_composite_lora_gb300 as tcl
    M, d_in, r = A.shape
    d_out = B.shape[2]
    F = torch.empty(M, d_in, r, dtype=torch.float32, device="cuda")
    Tt = torch.empty(M, r, d_out, dtype=torch.float32, device="cuda")
    sig = torch.empty(M, r, dtype=torch.float32, device="cuda")
    nb = tcl.lora_recompress_workspace_bytes(M, d_in, r)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    tcl.lora_recompress(bf16_tensor(A), bf16_tensor(B), M, d_in, d_out, r, F, Tt, sig, ws, nb)
    torch.cuda.synchronize()
    return sig.cpu().numpy(), F.cpu().numpy().astype(np.float64), Tt.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,d_in,d_out,r", [(5, 256, 512, 8), (7, 4096, 4096, 16), (3, 4096, 1024, 64),
                                           (2, 192, 320, 13)])
def test_recompress_matches_oracle(M, d_in, d_out, r):
    rng = np.random.default_rng(d_in + r)
    A, B = _fleet(rng, M, d_in, d_out, r)
    sig, F, Tt = _run(A, B)
    for m in range(M):
        a = bf16_bits_to_f32(A[m]).astype(np.float64)
        b = bf16_bits_to_f32(B[m]).astype(np.float64)
        s_ref, f_ref, t_ref = RC.balanced_factors(a, b)
        # singular values: fp32 Gram of H, relative to the largest
        np.testing.assert_allclose(sig[m], s_ref, rtol=1e-3, atol=2e-4 * s_ref[0])
        dw = a @ b
        nrm = np.linalg.norm(dw)
        for k in sorted({1, max(1, r // 4), max(1, r // 2), r}):
            got = F[m][:, :k] @ Tt[m][:k]
            want = f_ref[:, :k] @ t_ref[:k]
            assert np.linalg.norm(got - want) <= 2e-3 * nrm, (m, k)
        np.testing.assert_allclose(F[m].T @ F[m], np.diag(sig[m]), atol=2e-3 * s_ref[0])
        np.testing.assert_allclose(Tt[m] @ Tt[m].T, np.diag(sig[m]), atol=2e-3 * s_ref[0])


def test_recompress_padded_factors_keep_their_rank():
    rng = np.random.default_rng(31)
    M, d_in, d_out, r = 6, 1024, 512, 16
    pad = [16, 11, 5, 1, 8, 3]
    A, B = _fleet(rng, M, d_in, d_out, r, decay=0.8, pad=pad)
    sig, F, Tt = _run(A, B)
    for m in range(M):
        assert np.count_nonzero(sig[m]) == pad[m], (m, sig[m])
        a = bf16_bits_to_f32(A[m]).astype(np.float64)
        b = bf16_bits_to_f32(B[m]).astype(np.float64)
        assert np.linalg.norm(F[m] @ Tt[m] - a @ b) <= 2e-3 * np.linalg.norm(a @ b)


def test_recompressed_fleet_serves_the_delta():
    """Recompress a pool's adapters, keep spectral retained ranks, register
    the bf16 factor prefixes: the delta with those ranks matches the oracle's
    delta on the same factors and ranks, and the retained directions carry
    most of each update's energy."""
    import tenant_composite_lora_gb300 as tcl
    rng = np.random.default_rng(5)
    base = W.make("distinct", y_zero=True)
    M, d_in, d_out, r = base.capacity, base.d_in, base.d_out, 16
    A, B = _fleet(rng, M, d_in, d_out, r, decay=0.75)
    sig, F, Tt = _run(A, B)
    k = tcl.lora_rank_allocate(sig, np.full(M, r), np.full(M, d_in + d_out), tcl.native.LORA_RANK_SPECTRAL, 4, 1)
    Fb = W.f32_to_bf16_bits(F.astype(np.float32))
    Tb = W.f32_to_bf16_bits(Tt.astype(np.float32))
    wl = W.Workload("recompressed", d_in, d_out, r, M, base.offsets, base.ids, base.alpha, base.x, Fb, Tb,
                    k.astype(np.int32), np.zeros((base.T, d_out), np.uint16))
    pool = tcl.LoraPool(d_in, d_out, r, M)
    m = tcl.LoraMapping(wl.T, wl.P, M)
    try:
        for a in range(M):
            pool.register(a, bf16_tensor(Fb[a]), bf16_tensor(Tb[a]), int(k[a]))
        m.build(torch.from_numpy(wl.offsets).cuda(), torch.from_numpy(wl.ids).cuda(),
                torch.from_numpy(wl.alpha).cuda())
        y = torch.zeros(wl.T, d_out, dtype=torch.bfloat16, device="cuda")
        tcl.delta_apply(bf16_tensor(wl.x), y, pool, m)
        torch.cuda.synchronize()
        got = bf16_to_numpy_bits(y)
    finally:
        pool.close()
        m.close()
    _, acc, st = oracle.apply_workload(wl, threads=0)
    assert st == 0
    yf = bf16_bits_to_f32(got).astype(np.float64)
    rms = float(np.sqrt(np.mean(acc ** 2)))
    assert np.all(np.abs(yf - acc) <= 2.0 ** -7 * np.abs(acc) + 1e-3 * rms)
    kept = np.mean([np.sum(sig[a][:k[a]] ** 2) / np.sum(sig[a] ** 2) for a in range(M)])
    assert kept > 0.6 and k.sum() <= M * (r // 4)
