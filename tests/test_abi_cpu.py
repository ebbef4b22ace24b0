"""Host-side checks of the C-ABI library that need no GPU: it builds, loads,
exports every entry point that include/lora.h declares, answers host-only
calls, rejects bad arguments before touching the device, and the product
package never reaches the oracle."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lora.h")


@pytest.fixture(scope="module")
def lib():
    from tenant_composite_lora_gb300 import build, native
    build.build()
    return native.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("lora_pool_create", "lora_pool_register", "lora_build_mapping", "lora_delta_apply",
                 "lora_mapping_status", "lora_pool_destroy", "lora_mapping_destroy"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from tenant_composite_lora_gb300 import native
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(native.EXPORTS) == names


def test_host_only_calls(lib):
    from tenant_composite_lora_gb300 import native
    assert native.status_string(0) == "ok"
    assert "not supported" in native.status_string(5)
    assert "sm_103a" in native.lora_version()
    # the dispatch table: decode batches, long prefill batches, the rank
    # classes' crossovers, and shapes only the split path takes
    assert native.lora_dispatch_choose(32, 96, 8, 4096, 4096) == native.LORA_PATH_DECODE
    assert native.lora_dispatch_choose(256, 512, 64, 4096, 1024) == native.LORA_PATH_DECODE
    assert native.lora_dispatch_choose(3250, 6500, 16, 4096, 4096) == native.LORA_PATH_MMA
    assert native.lora_dispatch_choose(300, 900, 16, 4096, 4096) == native.LORA_PATH_DECODE
    assert native.lora_dispatch_choose(383, 766, 64, 4096, 4096) == native.LORA_PATH_DECODE
    assert native.lora_dispatch_choose(384, 768, 64, 4096, 4096) == native.LORA_PATH_MMA
    assert native.lora_dispatch_choose(3071, 6142, 16, 4096, 4096) == native.LORA_PATH_DECODE
    assert native.lora_dispatch_choose(8191, 16382, 8, 4096, 4096) == native.LORA_PATH_DECODE
    assert native.lora_dispatch_choose(8192, 16384, 8, 4096, 4096) == native.LORA_PATH_MMA
    assert native.lora_dispatch_choose(4096, 8192, 16, 4104, 4096) == native.LORA_PATH_DECODE  # no tensor maps
    assert native.lora_dispatch_choose(32, 96, 8, 110592, 4096) == native.LORA_PATH_SPLIT    # x row > smem
    assert native.lora_dispatch_choose(32, 96, 8, 110600, 4096) == native.LORA_PATH_SPLIT


def test_bad_arguments_rejected_before_device(lib):
    out = ctypes.c_void_p()
    assert lib.lora_pool_create(0, 64, 8, 4, ctypes.byref(out)) == 1
    assert lib.lora_pool_create(64, 64, 8, 4, None) == 1
    assert lib.lora_pool_create(100, 64, 8, 4, ctypes.byref(out)) == 5   # not a multiple of 64
    assert lib.lora_pool_create(64, 64, 65, 4, ctypes.byref(out)) == 5   # rank above the limit
    assert lib.lora_pool_create(64, 64, 8, 49153, ctypes.byref(out)) == 5
    assert lib.lora_mapping_create(-1, 4, 4, ctypes.byref(out)) == 1
    assert lib.lora_mapping_create(4, 4, 0, ctypes.byref(out)) == 1
    assert lib.lora_build_mapping(None, None, None, None, 1, 1, None) == 1
    assert lib.lora_delta_apply(None, None, None, None, None, None) == 1
    assert lib.lora_pool_register(None, 0, None, None, 1, None) == 1
    assert lib.lora_pool_destroy(None) == 0
    assert lib.lora_mapping_destroy(None) == 0
    assert lib.lora_delta_apply_multi(None, 1, None, None) == 1
    assert lib.lora_delta_apply_ablation(None, None, None, None, None, 1, None, 0, None) == 1


def test_ablation_workspace_sizes(lib):
    """The ablation's scratch, host-computed: z rows and an fp32 y (naive
    loop), gathered x rows, z rows and per-pair fp32 rows (Copy + SGMV), one
    fp32 d_in x d_out weight per token (pre-merge); 256-byte pieces."""
    from tenant_composite_lora_gb300 import native
    r = lambda b: (b + 255) // 256 * 256
    T, P, d_in, d_out, r_max = 32, 96, 4096, 4096, 8
    assert native.lora_ablation_workspace_bytes(1, T, P, d_in, d_out, r_max) == r(P * 8 * 4) + r(T * d_out * 4)
    assert native.lora_ablation_workspace_bytes(2, T, P, d_in, d_out, r_max) == \
        r(P * d_in * 2) + r(P * 8 * 4) + r(P * d_out * 4)
    assert native.lora_ablation_workspace_bytes(3, T, P, d_in, d_out, r_max) == r(T * d_in * d_out * 4)
    assert native.lora_ablation_workspace_bytes(9, T, P, d_in, d_out, r_max) == 0


def test_missing_library_fails_loudly(tmp_path):
    from tenant_composite_lora_gb300 import native
    saved = native._lib
    native._lib = None
    try:
        with pytest.raises(RuntimeError, match="no CPU or Python fallback"):
            native.load(str(tmp_path / "nope.so"))
    finally:
        native._lib = saved


def test_product_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "tenant_composite_lora_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.lower(), f
                assert "lora_oracle" not in src
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            src = open(os.path.join(ROOT, "oracle", f)).read()
            assert "tenant_composite_lora_gb300" not in src


def test_binding_refuses_wrong_memory_and_layouts():
    """The binding hands kernels only what they can read: host memory, a
    non-contiguous view or a wrong element type is refused before the
    library is called (no GPU involved: the checks come first)."""
    import numpy as np
    import torch
    from tenant_composite_lora_gb300 import native

    fake = 1  # never dereferenced: every call below raises before the library
    off = torch.zeros(5, dtype=torch.int32)
    ids = torch.zeros(4, dtype=torch.int32)
    alpha = torch.zeros(4, dtype=torch.float32)
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    # device entry points: host tensors and numpy arrays are refused
    with pytest.raises(ValueError, match="offsets: a CUDA tensor is expected"):
        native.lora_build_mapping(fake, off, ids, alpha, 4, 4, 0)
    with pytest.raises(ValueError, match="x: a device array is expected"):
        native.lora_delta_apply(np.zeros((4, 64), np.int16), 0, fake, None, fake, 0)
    with pytest.raises(ValueError, match="A: a CUDA tensor is expected"):
        native.lora_pool_register(fake, 0, x, x, 1, 0)
    with pytest.raises(ValueError, match="x: a CUDA tensor is expected"):
        native.lora_delta_apply_noalloc(x, 0, fake, None, 0, 0, 0, 4, 4, stream=0)
    # host entry point: layouts and element types
    y = torch.zeros(4, 64, dtype=torch.int16)
    with pytest.raises(ValueError, match="x_host: the tensor must be contiguous"):
        native.lora_delta_apply_host(torch.zeros(64, 4, dtype=torch.int16).t(), y, off, ids, alpha, 4, 4,
                                     fake, None, fake, 0)
    with pytest.raises(ValueError, match="ids_host: int32 elements expected"):
        native.lora_delta_apply_host(x, y, off, ids.long(), alpha, 4, 4, fake, None, fake, 0)
    with pytest.raises(ValueError, match="alpha_host: float32 elements expected"):
        native.lora_delta_apply_host(x, y, off, ids, alpha.double(), 4, 4, fake, None, fake, 0)
    with pytest.raises(ValueError, match="y_host: bf16 elements expected"):
        native.lora_delta_apply_host(x, y.float(), off, ids, alpha, 4, 4, fake, None, fake, 0)
    with pytest.raises(ValueError, match="offsets_host: the array must be C-contiguous"):
        native.lora_delta_apply_host(x, y, np.zeros((5, 2), np.int32)[:, 0], ids, alpha, 4, 4, fake, None,
                                     fake, 0)


def test_binding_accepts_what_the_library_takes():
    """The argument kinds the tests, the benchmark and the smoke run pass
    (bf16 or int16 x / y, int32 offsets / ids / ranks / status, float32
    alpha, contiguous) go through as their data pointers."""
    import numpy as np
    import torch
    from tenant_composite_lora_gb300 import native

    class OnDevice:  # a contiguous tensor as a CUDA tensor would present itself
        def __init__(self, t):
            self.t = t
            self.is_cuda = True
            self.dtype = t.dtype
            self.device = "cuda:0"

        def is_contiguous(self):
            return self.t.is_contiguous()

        def element_size(self):
            return self.t.element_size()

        def data_ptr(self):
            return self.t.data_ptr()

    for t, kind in ((torch.zeros(4, 64, dtype=torch.bfloat16), "bf16"),
                    (torch.zeros(4, 64, dtype=torch.int16), "bf16"),
                    (torch.zeros(5, dtype=torch.int32), "int32"),
                    (torch.zeros(5, dtype=torch.float32), "float32")):
        assert native._dptr(OnDevice(t), "arg", kind) == t.data_ptr()
        assert native._hptr(t, "arg", kind) == t.data_ptr()
    a = np.zeros(5, np.int32)
    assert native._hptr(a, "arg", "int32") == a.ctypes.data
    assert native._dptr(None, "arg", "int32") is None and native._dptr(1234, "arg", "int32") == 1234
    with pytest.raises(ValueError, match="int32 elements expected"):
        native._dptr(OnDevice(torch.zeros(5, dtype=torch.int64)), "arg", "int32")


def test_wrappers_check_shapes_before_the_library():
    """delta_apply and LoraMapping.build refuse shapes the kernels would read
    past (x / y rows and widths, alpha's length), before any library call."""
    import torch
    import tenant_composite_lora_gb300 as tcl

    class Pool:
        d_in, d_out, capacity, handle = 64, 128, 8, 1

    class Mapping(tcl.LoraMapping):
        def __init__(self, T):  # no library object: the checks come first
            self.T, self.P, self.handle = T, 0, 1

        def close(self):  # nothing to destroy
            self.handle = None

    m = Mapping(4)
    bf = torch.bfloat16
    with pytest.raises(ValueError, match="x must be"):
        tcl.delta_apply(torch.zeros(3, 64, dtype=bf), torch.zeros(4, 128, dtype=bf), Pool, m)
    with pytest.raises(ValueError, match="x must be"):
        tcl.delta_apply(torch.zeros(4, 32, dtype=bf), torch.zeros(4, 128, dtype=bf), Pool, m)
    with pytest.raises(ValueError, match="y must be"):
        tcl.delta_apply(torch.zeros(4, 64, dtype=bf), torch.zeros(4, 64, dtype=bf), Pool, m)
    with pytest.raises(ValueError, match="ranks must hold 8"):
        tcl.delta_apply(torch.zeros(4, 64, dtype=bf), torch.zeros(4, 128, dtype=bf), Pool, m,
                        ranks=torch.zeros(7, dtype=torch.int32))
    off = torch.zeros(5, dtype=torch.int32)
    with pytest.raises(ValueError, match="alpha has 3 entries for 4 ids"):
        m.build(off, torch.zeros(4, dtype=torch.int32), torch.zeros(3))
    with pytest.raises(ValueError, match="1-D"):
        m.build(off.view(5, 1), torch.zeros(4, dtype=torch.int32), torch.zeros(4))


def test_noalloc_binding_checks_sizes_before_the_library():
    """lora_delta_apply_noalloc refuses pair arrays whose lengths disagree
    with T and P, x / y with fewer than T rows or the wrong width, and a rank
    table shorter than the pool, before any library call (CPU tensors: the
    size checks come before the memory checks)."""
    import torch
    from tenant_composite_lora_gb300 import native

    class Pool:
        d_in, d_out, capacity, handle = 64, 128, 8, 1

    T, P = 4, 6
    bf = torch.bfloat16
    x, y = torch.zeros(T, 64, dtype=bf), torch.zeros(T, 128, dtype=bf)
    off, ids, al = torch.zeros(T + 1, dtype=torch.int32), torch.zeros(P, dtype=torch.int32), torch.zeros(P)

    def call(**kw):
        a = dict(x=x, y=y, pool=Pool, ranks=None, offsets=off, ids=ids, alpha=al, T=T, P=P)
        a.update(kw)
        native.lora_delta_apply_noalloc(a["x"], a["y"], a["pool"], a["ranks"], a["offsets"], a["ids"],
                                        a["alpha"], a["T"], a["P"], stream=0)

    with pytest.raises(ValueError, match="ids holds 5 entries, 6 expected"):
        call(ids=torch.zeros(5, dtype=torch.int32))
    with pytest.raises(ValueError, match="ids holds 6 entries, 7 expected"):
        call(P=7, alpha=torch.zeros(7))
    with pytest.raises(ValueError, match="alpha holds 5 entries, 6 expected"):
        call(alpha=torch.zeros(5))
    with pytest.raises(ValueError, match="offsets holds 5 entries, 6 expected"):
        call(T=5)
    with pytest.raises(ValueError, match="x has 3 rows"):
        call(x=torch.zeros(3, 64, dtype=bf))
    with pytest.raises(ValueError, match="y has 3 rows"):
        call(y=torch.zeros(3, 128, dtype=bf))
    with pytest.raises(ValueError, match="x has 32 columns"):
        call(x=torch.zeros(T, 32, dtype=bf))
    with pytest.raises(ValueError, match="y has 64 columns"):
        call(y=torch.zeros(T, 64, dtype=bf))
    with pytest.raises(ValueError, match="ranks holds 7 entries"):
        call(ranks=torch.zeros(7, dtype=torch.int32))
    with pytest.raises(ValueError, match="must be >= 0"):
        call(T=-1)
    # everything consistent: the size checks pass and the memory check refuses the host tensors
    with pytest.raises(ValueError, match="x: a CUDA tensor is expected"):
        call(ranks=torch.zeros(8, dtype=torch.int32))


def test_rank_allocate_matches_the_oracle(lib):
    """lora_rank_allocate (host code of the library) against the oracle's
    policies: the worked example and random fleets with mixed shapes."""
    import json
    import numpy as np
    from oracle import recompress as RC
    from tenant_composite_lora_gb300 import native
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "rank_allocation_example.json")))
    sig = np.array(g["sigma"], np.float32)
    for pol, key in ((native.LORA_RANK_UNIFORM, "U"), (native.LORA_RANK_SPECTRAL, "S")):
        k = native.lora_rank_allocate(sig, g["rank"], g["cost"], pol, g["d"], g["floor"])
        assert k.tolist() == g[key]
    rng = np.random.default_rng(6)
    for trial in range(20):
        M, r = int(rng.integers(1, 30)), 16
        sig = np.sort(rng.random((M, r)).astype(np.float32) ** 3, axis=1)[:, ::-1].copy()
        sig[rng.random((M, r)) < 0.1] = 0
        sig = np.sort(sig, axis=1)[:, ::-1].copy()
        rank = rng.integers(1, r + 1, size=M).astype(np.int32)
        cost = rng.choice([5120, 8192, 18432], size=M).astype(np.int32)
        d, fl = int(rng.integers(1, 9)), int(rng.integers(0, 3))
        for pol, key in ((native.LORA_RANK_UNIFORM, "U"), (native.LORA_RANK_SPECTRAL, "S")):
            got = native.lora_rank_allocate(sig, rank, cost, pol, d, fl)
            want = RC.rank_allocate(list(sig.astype(np.float64)), cost, rank, key, d, fl)
            assert got.tolist() == want, (trial, key)


def test_binding_checks_array_sizes_before_the_library():
    """The other entry points taking arrays refuse one with fewer elements
    than their sizes imply (the kernels would read or write past it), before
    any library call (CPU tensors: the size checks come before the memory
    checks); calls whose parameters the library refuses itself reach it."""
    import numpy as np
    import torch
    from tenant_composite_lora_gb300 import native

    fake = 1  # never dereferenced: every call below raises before the library
    i32 = lambda n: torch.zeros(n, dtype=torch.int32)
    f32 = lambda *s: torch.zeros(*s, dtype=torch.float32)
    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)
    T, P = 4, 6
    with pytest.raises(ValueError, match="lora_build_mapping: offsets holds 4 entries, at least 5"):
        native.lora_build_mapping(fake, i32(4), i32(P), f32(P), T, P, 0)
    with pytest.raises(ValueError, match="lora_build_mapping: ids holds 5 entries, at least 6"):
        native.lora_build_mapping(fake, i32(T + 1), i32(5), f32(P), T, P, 0)
    with pytest.raises(ValueError, match="lora_build_mapping: alpha holds 5 entries, at least 6"):
        native.lora_build_mapping(fake, i32(T + 1), i32(P), f32(5), T, P, 0)
    # larger buffers than the batch are fine (the memory check is what fails here)
    with pytest.raises(ValueError, match="offsets: a CUDA tensor is expected"):
        native.lora_build_mapping(fake, i32(64), i32(64), f32(64), T, P, 0)

    x, y = bf(T, 64).view(torch.int16), bf(T, 64).view(torch.int16)
    with pytest.raises(ValueError, match="lora_delta_apply_host: offsets_host holds 4 entries"):
        native.lora_delta_apply_host(x, y, i32(4), i32(P), f32(P), T, P, fake, None, fake, 0)
    with pytest.raises(ValueError, match="lora_delta_apply_host: ids_host holds 5 entries"):
        native.lora_delta_apply_host(x, y, i32(T + 1), i32(5), f32(P), T, P, fake, None, fake, 0)
    with pytest.raises(ValueError, match="lora_delta_apply_host: alpha_host holds 5 entries"):
        native.lora_delta_apply_host(x, y, i32(T + 1), i32(P), f32(5), T, P, fake, None, fake, 0)
    with pytest.raises(ValueError, match="lora_delta_apply_host: x_host has 3 rows"):
        native.lora_delta_apply_host(x[:3], y, i32(T + 1), i32(P), f32(P), T, P, fake, None, fake, 0)
    with pytest.raises(ValueError, match="lora_delta_apply_host: y_host has 3 rows"):
        native.lora_delta_apply_host(x, y[:3], i32(T + 1), i32(P), f32(P), T, P, fake, None, fake, 0)

    E, d_in = 8, 64
    with pytest.raises(ValueError, match="lora_gate_logits: x holds"):
        native.lora_gate_logits(bf(T - 1, d_in), bf(E, d_in), i32(T), T, E, d_in, f32(T, E))
    with pytest.raises(ValueError, match="lora_gate_logits: wg holds"):
        native.lora_gate_logits(bf(T, d_in), bf(E - 1, d_in), i32(T), T, E, d_in, f32(T, E))
    with pytest.raises(ValueError, match="lora_gate_logits: req holds"):
        native.lora_gate_logits(bf(T, d_in), bf(E, d_in), i32(T - 1), T, E, d_in, f32(T, E))
    with pytest.raises(ValueError, match="lora_gate_logits: logits holds"):
        native.lora_gate_logits(bf(T, d_in), bf(E, d_in), i32(T), T, E, d_in, f32(T, E - 1))
    k = 2
    good = dict(logits=f32(T * E), cand=i32(T * E), offsets=i32(T + 1), ids=i32(T * k), alpha=f32(T * k))
    for name, short in (("logits", f32(T * E - 1)), ("cand", i32(T * E - 1)), ("offsets", i32(T)),
                        ("ids", i32(T * k - 1)), ("alpha", f32(T * k - 1))):
        a = dict(good, **{name: short})
        with pytest.raises(ValueError, match=f"lora_gate_topk: {name} holds"):
            native.lora_gate_topk(a["logits"], a["cand"], T, E, k, a["offsets"], a["ids"], a["alpha"])

    M, r, d_out = 2, 4, 32
    good = dict(A=bf(M, d_in, r), B=bf(M, r, d_out), F=f32(M, d_in, r), T=f32(M, r, d_out), sigma=f32(M, r))
    for name, short in (("A", bf(M, d_in, r - 1)), ("B", bf(M, r, d_out - 1)), ("F", f32(1, d_in, r)),
                        ("T", f32(M, r - 1, d_out)), ("sigma", f32(M, r - 1))):
        a = dict(good, **{name: short})
        with pytest.raises(ValueError, match=f"lora_recompress: {name} holds"):
            native.lora_recompress(a["A"], a["B"], M, d_in, d_out, r, a["F"], a["T"], a["sigma"], None, 0)

    with pytest.raises(ValueError, match="lora_rank_allocate: rank holds 2 entries, at least 3"):
        native.lora_rank_allocate(np.ones((3, 4), np.float32), [4, 4], [8, 8, 8], native.LORA_RANK_UNIFORM, 2)
    with pytest.raises(ValueError, match="lora_rank_allocate: cost holds 2 entries, at least 3"):
        native.lora_rank_allocate(np.ones((3, 4), np.float32), [4, 4, 4], [8, 8], native.LORA_RANK_UNIFORM, 2)
    with pytest.raises(ValueError, match="lora_diag_wait_expiry: words holds 3 entries, at least 4"):
        native.lora_diag_wait_expiry(0, 10_000, i32(3))
    # parameters the library refuses itself (top_k above 8, E above 64) skip
    # the size checks, so that the library's own status comes back
    with pytest.raises(ValueError, match="logits: a CUDA tensor is expected"):
        native.lora_gate_topk(f32(16), i32(16), 2, 8, 9, i32(16), i32(16), f32(16))
    with pytest.raises(ValueError, match="logits: a CUDA tensor is expected"):
        native.lora_gate_topk(f32(16), i32(16), 2, 65, 2, i32(16), i32(16), f32(16))
