"""On-device MoE-LoRA gating: gate logits (fp32 accumulation) against the
fp64 oracle within one fp32 summation's rounding; the top-k selection taken
on the device's own fp32 logits on both sides, so the kept ids are compared
bit for bit and alpha within fp32 rounding; then the pair lists feed the
mapping and the delta directly, checked against the oracle."""
import numpy as np
import pytest

import oracle
import workloads as W
from workloads import bf16_bits_to_f32
from workloads.device import bf16_tensor, bf16_to_numpy_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    from tenant_composite_lora_gb300 import build
    build.build()


def _moe_batch(rng, n_req, E, d_in, cap, lens):
    """Request-contiguous tokens, E candidate adapters per request (some slots
    padded with -1), a router per request."""
    req = np.concatenate([np.full(L, r, np.int32) for r, L in enumerate(lens)])
    T = req.size
    cands = np.stack([rng.choice(cap, size=E, replace=False) for _ in range(n_req)]).astype(np.int32)
    cands[rng.random((n_req, E)) < 0.15] = -1
    x = W.f32_to_bf16_bits(rng.standard_normal((T, d_in)).astype(np.float32) * 0.02)
    wg = W.f32_to_bf16_bits(rng.standard_normal((n_req, E, d_in)).astype(np.float32))
    return req, cands[req], x, wg


@pytest.mark.parametrize("top_k", [1, 2, 3])
def test_gating_matches_oracle(top_k):
    import tenant_composite_lora_gb300 as tcl
    rng = np.random.default_rng(top_k)
    n_req, E, d_in, cap = 16, 8, 4096, 64
    lens = np.clip(np.round(rng.lognormal(4.0, 0.8, size=n_req)), 4, 300).astype(int)
    req, cand, x, wg = _moe_batch(rng, n_req, E, d_in, cap, lens)
    cand[5] = -1  # a token with no valid candidate
    T = req.size
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    offs = torch.empty(T + 1, dtype=torch.int32, device="cuda")
    ids = torch.empty(T * top_k, dtype=torch.int32, device="cuda")
    al = torch.empty(T * top_k, dtype=torch.float32, device="cuda")
    tcl.lora_gate_logits(bf16_tensor(x), bf16_tensor(wg), dev(req), T, E, d_in, logits)
    tcl.lora_gate_topk(logits, dev(cand), T, E, top_k, offs, ids, al)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    ref = oracle.gate_logits(x, wg, req)
    # fp32 accumulation over d_in terms: |error| <= d_in * 2^-24 * sum |x w|
    bound = d_in * 2.0 ** -24 * np.einsum("td,ted->te", np.abs(bf16_bits_to_f32(x).astype(np.float64)),
                                          np.abs(bf16_bits_to_f32(wg).astype(np.float64))[req])
    assert np.all(np.abs(lg - ref) <= bound)
    r_off, r_ids, r_al, empty = oracle.gate_topk(lg, cand, top_k)
    assert empty == 1
    np.testing.assert_array_equal(offs.cpu().numpy(), r_off)
    np.testing.assert_array_equal(ids.cpu().numpy(), r_ids)
    np.testing.assert_allclose(al.cpu().numpy(), r_al, rtol=4e-7, atol=1e-7)


def test_gated_pairs_feed_the_delta():
    """Gating -> mapping -> delta on the device, with no host step between:
    the result matches the oracle's delta on the same pair lists."""
    import tenant_composite_lora_gb300 as tcl
    rng = np.random.default_rng(9)
    n_req, E, d_in, d_out, cap, top_k = 6, 8, 1024, 512, 48, 2
    lens = np.array([40, 7, 120, 33, 64, 9])
    req, cand, x, wg = _moe_batch(rng, n_req, E, d_in, cap, lens)
    T = req.size
    base = W.make_custom(rng, d_in=d_in, d_out=d_out, r_max=16, capacity=cap, id_lists=[[0]] * T,
                         alpha_lists=[[np.float32(1)]] * T, y_sigma=0.0)
    base.x[:] = x
    pool = tcl.LoraPool(d_in, d_out, 16, cap)
    m = tcl.LoraMapping(T, T * top_k, cap)
    try:
        for a in range(cap):
            pool.register(a, bf16_tensor(base.A[a]), bf16_tensor(base.B[a]), int(base.ranks[a]))
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        xd, y = bf16_tensor(x), torch.zeros(T, d_out, dtype=torch.bfloat16, device="cuda")
        logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
        offs = torch.empty(T + 1, dtype=torch.int32, device="cuda")
        ids = torch.empty(T * top_k, dtype=torch.int32, device="cuda")
        al = torch.empty(T * top_k, dtype=torch.float32, device="cuda")
        tcl.lora_gate_logits(xd, bf16_tensor(wg), dev(req), T, E, d_in, logits)
        tcl.lora_gate_topk(logits, dev(cand), T, E, top_k, offs, ids, al)
        tcl.lora_build_mapping(m.handle, offs, ids, al, T, T * top_k)
        m.T, m.P = T, T * top_k
        tcl.delta_apply(xd, y, pool, m)
        torch.cuda.synchronize()
        assert m.status() == 0
        got = bf16_to_numpy_bits(y)
        wl = W.Workload("gated", d_in, d_out, 16, cap, offs.cpu().numpy(), ids.cpu().numpy(), al.cpu().numpy(),
                        x, base.A, base.B, base.ranks, np.zeros((T, d_out), np.uint16))
    finally:
        pool.close()
        m.close()
    _, acc, st = oracle.apply_workload(wl, threads=0)
    assert st == 0
    yf = bf16_bits_to_f32(got).astype(np.float64)
    rms = float(np.sqrt(np.mean(acc ** 2)))
    assert rms > 0
    assert np.all(np.abs(yf - acc) <= 2.0 ** -7 * np.abs(acc) + 1e-3 * rms)


def test_gating_argument_limits():
    import tenant_composite_lora_gb300 as tcl
    t = torch.zeros(16, dtype=torch.float32, device="cuda")
    i = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(tcl.LoraError) as e:
        tcl.lora_gate_topk(t, i, 2, 8, 9, i, i, t)  # top_k above 8
    assert e.value.status == tcl.native.LORA_ERR_NOT_SUPPORTED
    with pytest.raises(tcl.LoraError) as e:
        tcl.lora_gate_topk(t, i, 2, 65, 2, i, i, t)  # E above 64
    assert e.value.status == tcl.native.LORA_ERR_NOT_SUPPORTED
