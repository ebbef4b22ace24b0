"""ctypes binding of libtclora.so: the C-ABI entry points under the same names.

Argument marshalling only.  Device arrays are passed as contiguous torch CUDA
tensors (their data_ptr) or raw integer addresses, host arrays as contiguous
CPU tensors or numpy arrays; a tensor in the wrong memory, not contiguous or
of the wrong element type is refused before the library is called.  Streams
are torch.cuda.Stream, a raw cudaStream_t integer, or None for the current
torch stream.  Every step of the
delta runs inside the library's CUDA kernels; nothing here computes.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtclora.so")

LORA_OK = 0
LORA_ERR_INVALID_ARG = 1
LORA_ERR_OUT_OF_MEMORY = 2
LORA_ERR_CUDA = 3
LORA_ERR_BAD_ADAPTER = 4
LORA_ERR_NOT_SUPPORTED = 5

LORA_DEV_BAD_ID = 1
LORA_DEV_BAD_OFFSETS = 2
LORA_DEV_UNREGISTERED = 4
LORA_DEV_BAD_RANK = 8
LORA_DEV_TIMEOUT = 16

LORA_PATH_AUTO = 0
LORA_PATH_SPLIT = 1
LORA_PATH_FUSED = 2
LORA_PATH_MMA = 3
LORA_PATH_DECODE = 4

LORA_MAX_RANK = 64
LORA_MAX_CAPACITY = 49152

# every entry point of include/lora.h
EXPORTS = [
    "lora_pool_create", "lora_pool_register", "lora_pool_unregister", "lora_pool_destroy",
    "lora_mapping_create", "lora_build_mapping", "lora_delta_apply", "lora_delta_apply_path",
    "lora_dispatch_choose", "lora_delta_apply_host", "lora_mapping_status", "lora_mapping_export",
    "lora_mapping_destroy", "lora_status_string", "lora_version", "lora_delta_apply_noalloc",
    "lora_diag_wait_expiry", "lora_delta_apply_multi", "lora_ablation_workspace_bytes",
    "lora_delta_apply_ablation", "lora_gate_logits", "lora_gate_topk", "lora_recompress_workspace_bytes",
    "lora_recompress", "lora_rank_allocate",
]

LORA_RANK_UNIFORM = 0
LORA_RANK_SPECTRAL = 1

LORA_ABLATION_NAIVE = 1
LORA_ABLATION_COPY_SGMV = 2
LORA_ABLATION_PREMERGE = 3

LORA_MAX_PROJECTIONS = 8


class LoraProjection(ctypes.Structure):
    """lora_projection: one projection of lora_delta_apply_multi."""
    _fields_ = [("x_dev", ctypes.c_void_p), ("y_dev", ctypes.c_void_p), ("pool", ctypes.c_void_p),
                ("ranks_dev", ctypes.c_void_p)]

LORA_NOALLOC_SCRATCH_BYTES = 4 << 20


class LoraError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)} (status {status})")
        self.status = status


_lib = None


def load(path: str | None = None):
    """Loads libtclora.so; raises if it has not been built (there is no
    fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m tenant_composite_lora_gb300.build` "
            "(there is no CPU or Python fallback)")
    lib = ctypes.CDLL(path)
    V, I, PP = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "lora_pool_create": ([I, I, I, I, PP], I),
        "lora_pool_register": ([V, I, V, V, I, V], I),
        "lora_pool_unregister": ([V, I, V], I),
        "lora_pool_destroy": ([V], I),
        "lora_mapping_create": ([I, I, I, PP], I),
        "lora_build_mapping": ([V, V, V, V, I, I, V], I),
        "lora_delta_apply": ([V, V, V, V, V, V], I),
        "lora_delta_apply_path": ([V, V, V, V, V, I, V], I),
        "lora_dispatch_choose": ([I, I, I, I, I], I),
        "lora_delta_apply_host": ([V, V, V, V, V, I, I, V, V, V, V], I),
        "lora_delta_apply_noalloc": ([V, V, V, V, V, V, V, I, I, V, V], I),
        "lora_mapping_status": ([V, V, ctypes.POINTER(ctypes.c_int)], I),
        "lora_mapping_export": ([V, V, V, V, V, V, V, V, V, V], I),
        "lora_mapping_destroy": ([V], I),
        "lora_status_string": ([I], ctypes.c_char_p),
        "lora_version": ([], ctypes.c_char_p),
        "lora_diag_wait_expiry": ([I, ctypes.c_longlong, V, V], I),
        "lora_delta_apply_multi": ([ctypes.POINTER(LoraProjection), I, V, V], I),
        "lora_ablation_workspace_bytes": ([I, I, I, I, I, I], ctypes.c_size_t),
        "lora_delta_apply_ablation": ([V, V, V, V, V, I, V, ctypes.c_size_t, V], I),
        "lora_gate_logits": ([V, V, V, I, I, I, V, V], I),
        "lora_gate_topk": ([V, V, I, I, I, V, V, V, V], I),
        "lora_recompress_workspace_bytes": ([I, I, I], ctypes.c_size_t),
        "lora_recompress": ([V, V, I, I, I, I, V, V, V, V, ctypes.c_size_t, V], I),
        "lora_rank_allocate": ([V, I, I, V, V, I, I, I, V], I),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def status_string(s: int) -> str:
    try:
        return load().lora_status_string(int(s)).decode()
    except Exception:  # pragma: no cover
        return f"status {s}"


def _check(fn: str, s: int):
    if s != LORA_OK:
        raise LoraError(fn, s)


_BF16_LIKE = 2  # bytes per element of x, y, A, B (bf16, or its bits as int16)


def _dtype_ok(t, kind: str) -> bool:
    if kind == "bf16":
        return t.itemsize == _BF16_LIKE if isinstance(t, np.ndarray) else t.element_size() == _BF16_LIKE
    if isinstance(t, np.ndarray):
        return t.dtype == np.dtype(kind)
    import torch
    return t.dtype == {"int32": torch.int32, "float32": torch.float32}[kind]


def _dptr(t, name: str, kind: str) -> int | None:
    """Address of a device array: a contiguous CUDA tensor of the expected
    element type, or a raw integer address (the caller's responsibility).
    Host memory is refused here: a kernel must never be handed a host
    address."""
    if t is None or isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        raise ValueError(f"{name}: a device array is expected, not a numpy (host) array")
    if not t.is_cuda:
        raise ValueError(f"{name}: a CUDA tensor is expected, got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: the tensor must be contiguous")
    if not _dtype_ok(t, kind):
        raise ValueError(f"{name}: {kind} elements expected, got {t.dtype}")
    return t.data_ptr()


def _hptr(t, name: str, kind: str) -> int | None:
    """Address of a host array: a contiguous CPU tensor or C-ordered numpy
    array of the expected element type, or a raw integer address."""
    if t is None or isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        if not t.flags.c_contiguous:
            raise ValueError(f"{name}: the array must be C-contiguous")
        if not _dtype_ok(t, kind):
            raise ValueError(f"{name}: {kind} elements expected, got {t.dtype}")
        return t.ctypes.data
    if t.is_cuda:
        raise ValueError(f"{name}: a host tensor is expected, got a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: the tensor must be contiguous")
    if not _dtype_ok(t, kind):
        raise ValueError(f"{name}: {kind} elements expected, got {t.dtype}")
    return t.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ------------------------------------------------------------------ pools
def lora_pool_create(d_in: int, d_out: int, r_max: int, capacity: int) -> int:
    out = ctypes.c_void_p()
    _check("lora_pool_create", load().lora_pool_create(d_in, d_out, r_max, capacity, ctypes.byref(out)))
    return out.value


def lora_pool_register(pool: int, slot: int, A, B, k: int, stream=None):
    _check("lora_pool_register", load().lora_pool_register(pool, slot, _dptr(A, "A", "bf16"), _dptr(B, "B", "bf16"), k,
                                                     _stream(stream)))


def lora_pool_unregister(pool: int, slot: int, stream=None):
    _check("lora_pool_unregister", load().lora_pool_unregister(pool, slot, _stream(stream)))


def lora_pool_destroy(pool: int):
    _check("lora_pool_destroy", load().lora_pool_destroy(pool))


# ------------------------------------------------------------------ mappings
def lora_mapping_create(max_tokens: int, max_pairs: int, capacity: int) -> int:
    out = ctypes.c_void_p()
    _check("lora_mapping_create",
           load().lora_mapping_create(max_tokens, max_pairs, capacity, ctypes.byref(out)))
    return out.value


def lora_build_mapping(m: int, offsets, ids, alpha, T: int, P: int, stream=None):
    fn = "lora_build_mapping"
    _need(fn, "offsets", offsets, T + 1)
    _need(fn, "ids", ids, P)
    _need(fn, "alpha", alpha, P)
    _check("lora_build_mapping",
           load().lora_build_mapping(m, _dptr(offsets, "offsets", "int32"), _dptr(ids, "ids", "int32"),
                                     _dptr(alpha, "alpha", "float32"), T, P, _stream(stream)))


def lora_delta_apply(x, y, pool: int, ranks, m: int, stream=None):
    _check("lora_delta_apply",
           load().lora_delta_apply(_dptr(x, "x", "bf16"), _dptr(y, "y", "bf16"), pool,
                                   _dptr(ranks, "ranks", "int32"), m, _stream(stream)))


def lora_delta_apply_multi(projections, m: int, stream=None):
    """projections: a sequence of (x, y, pool handle, ranks or None), one per
    projection, all sharing the mapping m."""
    n = len(projections)
    arr = (LoraProjection * max(n, 1))()
    for i, (x, y, pool, ranks) in enumerate(projections):
        arr[i] = LoraProjection(_dptr(x, "x", "bf16"), _dptr(y, "y", "bf16"), pool, _dptr(ranks, "ranks", "int32"))
    _check("lora_delta_apply_multi", load().lora_delta_apply_multi(arr, n, m, _stream(stream)))


def lora_ablation_workspace_bytes(variant: int, T: int, P: int, d_in: int, d_out: int, r_max: int) -> int:
    return int(load().lora_ablation_workspace_bytes(variant, T, P, d_in, d_out, r_max))


def lora_delta_apply_ablation(x, y, pool: int, ranks, m: int, variant: int, workspace, workspace_bytes: int,
                              stream=None):
    """workspace: a device buffer (uint8 CUDA tensor or raw address) of at
    least lora_ablation_workspace_bytes(...) bytes."""
    ws = workspace if workspace is None or isinstance(workspace, int) else workspace.data_ptr()
    if workspace is not None and not isinstance(workspace, int) and not workspace.is_cuda:
        raise ValueError("workspace: a CUDA tensor is expected")
    _need_bytes("lora_delta_apply_ablation", workspace, workspace_bytes)
    _check("lora_delta_apply_ablation",
           load().lora_delta_apply_ablation(_dptr(x, "x", "bf16"), _dptr(y, "y", "bf16"), pool,
                                            _dptr(ranks, "ranks", "int32"), m, variant, ws, workspace_bytes,
                                            _stream(stream)))


def lora_gate_logits(x, wg, req, T: int, E: int, d_in: int, logits, stream=None):
    fn = "lora_gate_logits"
    if T > 0 and E > 0 and d_in > 0:
        _need(fn, "x", x, T * d_in)
        _need(fn, "wg", wg, E * d_in)
        _need(fn, "req", req, T)
        _need(fn, "logits", logits, T * E)
    _check("lora_gate_logits",
           load().lora_gate_logits(_dptr(x, "x", "bf16"), _dptr(wg, "wg", "bf16"), _dptr(req, "req", "int32"), T, E,
                                   d_in, _dptr(logits, "logits", "float32"), _stream(stream)))


def lora_gate_topk(logits, cand, T: int, E: int, top_k: int, offsets, ids, alpha, stream=None):
    fn = "lora_gate_topk"
    if T > 0 and 1 <= top_k <= min(E, 8) and E <= 64:  # (other values: the library refuses them)
        _need(fn, "logits", logits, T * E)
        _need(fn, "cand", cand, T * E)
        _need(fn, "offsets", offsets, T + 1)
        _need(fn, "ids", ids, T * top_k)
        _need(fn, "alpha", alpha, T * top_k)
    _check("lora_gate_topk",
           load().lora_gate_topk(_dptr(logits, "logits", "float32"), _dptr(cand, "cand", "int32"), T, E, top_k,
                                 _dptr(offsets, "offsets", "int32"), _dptr(ids, "ids", "int32"),
                                 _dptr(alpha, "alpha", "float32"), _stream(stream)))


def lora_recompress_workspace_bytes(M: int, d_in: int, r: int) -> int:
    return int(load().lora_recompress_workspace_bytes(M, d_in, r))


def lora_recompress(A, B, M: int, d_in: int, d_out: int, r: int, F, T, sigma, workspace, workspace_bytes: int,
                    stream=None):
    """A bf16 [M, d_in, r], B bf16 [M, r, d_out] (CUDA); F fp32 [M, d_in, r],
    T fp32 [M, r, d_out], sigma fp32 [M, r] written; workspace a CUDA byte
    buffer of lora_recompress_workspace_bytes(M, d_in, r)."""
    if workspace is not None and not isinstance(workspace, int) and not workspace.is_cuda:
        raise ValueError("workspace: a CUDA tensor is expected")
    fn = "lora_recompress"
    if M > 0 and d_in > 0 and d_out > 0 and r > 0:
        _need(fn, "A", A, M * d_in * r)
        _need(fn, "B", B, M * r * d_out)
        _need(fn, "F", F, M * d_in * r)
        _need(fn, "T", T, M * r * d_out)
        _need(fn, "sigma", sigma, M * r)
    _need_bytes(fn, workspace, workspace_bytes)
    ws = workspace if workspace is None or isinstance(workspace, int) else workspace.data_ptr()
    _check("lora_recompress",
           load().lora_recompress(_dptr(A, "A", "bf16"), _dptr(B, "B", "bf16"), M, d_in, d_out, r,
                                  _dptr(F, "F", "float32"), _dptr(T, "T", "float32"), _dptr(sigma, "sigma", "float32"),
                                  ws, workspace_bytes, _stream(stream)))


def lora_rank_allocate(sigma, rank, cost, policy: int, d: int, floor_k: int = 1) -> np.ndarray:
    """Host only: sigma float32 [M, r], rank and cost int32 [M] (numpy);
    returns the retained ranks k [M]."""
    sigma = np.ascontiguousarray(sigma, np.float32)
    rank = np.ascontiguousarray(rank, np.int32)
    cost = np.ascontiguousarray(cost, np.int32)
    M, r = sigma.shape
    _need("lora_rank_allocate", "rank", rank, M)
    _need("lora_rank_allocate", "cost", cost, M)
    k = np.zeros(M, np.int32)
    _check("lora_rank_allocate",
           load().lora_rank_allocate(sigma.ctypes.data, M, r, rank.ctypes.data, cost.ctypes.data, policy, d, floor_k,
                                     k.ctypes.data))
    return k


def lora_delta_apply_path(x, y, pool: int, ranks, m: int, path: int, stream=None):
    _check("lora_delta_apply_path",
           load().lora_delta_apply_path(_dptr(x, "x", "bf16"), _dptr(y, "y", "bf16"), pool,
                                        _dptr(ranks, "ranks", "int32"), m, path, _stream(stream)))


def lora_dispatch_choose(T: int, P: int, r_max: int, d_in: int, d_out: int) -> int:
    return int(load().lora_dispatch_choose(T, P, r_max, d_in, d_out))


def lora_delta_apply_host(x_host, y_host, offsets_host, ids_host, alpha_host, T: int, P: int,
                          pool: int, ranks, m: int, stream=None):
    fn = "lora_delta_apply_host"
    _need(fn, "offsets_host", offsets_host, T + 1)
    _need(fn, "ids_host", ids_host, P)
    _need(fn, "alpha_host", alpha_host, P)
    for name, t in (("x_host", x_host), ("y_host", y_host)):
        shape = getattr(t, "shape", None)
        if shape is not None and len(shape) == 2 and shape[0] < T:
            raise ValueError(f"{fn}: {name} has {shape[0]} rows, at least T = {T} needed")
    _check("lora_delta_apply_host",
           load().lora_delta_apply_host(_hptr(x_host, "x_host", "bf16"), _hptr(y_host, "y_host", "bf16"),
                                        _hptr(offsets_host, "offsets_host", "int32"),
                                        _hptr(ids_host, "ids_host", "int32"),
                                        _hptr(alpha_host, "alpha_host", "float32"), T, P, pool,
                                        _dptr(ranks, "ranks", "int32"), m, _stream(stream)))


def _numel(t) -> int | None:
    """Element count of a tensor or array (None for a raw address or None)."""
    if t is None or isinstance(t, int):
        return None
    return int(t.size) if isinstance(t, np.ndarray) else int(t.numel())


def _need(fn: str, name: str, t, want: int):
    """Refuse a tensor or array of fewer than `want` elements: the library
    would read or write past it (raw addresses and None are not checked)."""
    if want > 0 and t is not None and not isinstance(t, int):
        n = t.size if isinstance(t, np.ndarray) else t.numel()
        if n < want:
            raise ValueError(f"{fn}: {name} holds {n} entries, at least {want} needed")


def _need_bytes(fn: str, t, want: int):
    """The same for a workspace given as a tensor, in bytes."""
    if t is None or isinstance(t, int):
        return
    n = int(t.numel()) * int(t.element_size())
    if want > 0 and n < want:
        raise ValueError(f"{fn}: the workspace holds {n} bytes, {want} passed as its size")


def _rows_cols(t):
    """(rows, columns) of a 2-D tensor or array, else None."""
    if t is None or isinstance(t, int) or len(t.shape) != 2:
        return None
    return int(t.shape[0]), int(t.shape[1])


def _noalloc_checks(x, y, pool, ranks, offsets, ids, alpha, T: int, P: int):
    """Sizes the kernels would otherwise read past: the pair arrays against
    T and P, x and y against T rows (and the pool's widths when a LoraPool is
    given), ranks against the pool's capacity."""
    if T < 0 or P < 0:
        raise ValueError(f"lora_delta_apply_noalloc: T = {T} and P = {P} must be >= 0")
    for name, t, want in (("offsets", offsets, T + 1), ("ids", ids, P), ("alpha", alpha, P)):
        n = _numel(t)
        if n is not None and n != want:
            raise ValueError(f"lora_delta_apply_noalloc: {name} holds {n} entries, {want} expected "
                             f"(T = {T}, P = {P})")
    d_in, d_out, cap = (getattr(pool, "d_in", None), getattr(pool, "d_out", None),
                        getattr(pool, "capacity", None))
    for name, t, width in (("x", x, d_in), ("y", y, d_out)):
        rc = _rows_cols(t)
        if rc is None:
            continue
        if rc[0] < T:
            raise ValueError(f"lora_delta_apply_noalloc: {name} has {rc[0]} rows, at least T = {T} needed")
        if width is not None and rc[1] != width:
            raise ValueError(f"lora_delta_apply_noalloc: {name} has {rc[1]} columns, the pool's width is {width}")
    n = _numel(ranks)
    if n is not None and cap is not None and n < cap:
        raise ValueError(f"lora_delta_apply_noalloc: ranks holds {n} entries, the pool has {cap} slots")


def lora_delta_apply_noalloc(x, y, pool, ranks, offsets, ids, alpha, T: int, P: int,
                             status=None, stream=None):
    """pool: a pool handle, or an object with ``handle`` (and ``d_in``,
    ``d_out``, ``capacity``, which enable the width and rank-table checks),
    such as ``LoraPool``."""
    _noalloc_checks(x, y, pool, ranks, offsets, ids, alpha, T, P)
    handle = pool if pool is None or isinstance(pool, int) else pool.handle
    _check("lora_delta_apply_noalloc",
           load().lora_delta_apply_noalloc(_dptr(x, "x", "bf16"), _dptr(y, "y", "bf16"), handle,
                                           _dptr(ranks, "ranks", "int32"), _dptr(offsets, "offsets", "int32"),
                                           _dptr(ids, "ids", "int32"), _dptr(alpha, "alpha", "float32"), T, P,
                                           _dptr(status, "status", "int32"), _stream(stream)))


def lora_mapping_status(m: int, stream=None) -> int:
    v = ctypes.c_int()
    _check("lora_mapping_status", load().lora_mapping_status(m, _stream(stream), ctypes.byref(v)))
    return int(v.value)


def lora_mapping_export(m: int, P: int, capacity: int, stream=None) -> dict:
    """Copies the mapping to host numpy arrays (for checking)."""
    n = max(P, 1)
    tok = np.zeros(n, np.int32)
    adapter = np.zeros(n, np.int32)
    alpha = np.zeros(n, np.float32)
    src = np.zeros(n, np.int32)
    pos = np.zeros(n, np.int32)
    nseg = max(min(P, capacity), 1)
    seg_adapter = np.zeros(nseg, np.int32)
    seg_start = np.zeros(nseg + 1, np.int32)
    counts = np.zeros(3, np.int32)
    _check("lora_mapping_export",
           load().lora_mapping_export(m, _stream(stream), tok.ctypes.data, adapter.ctypes.data,
                                      alpha.ctypes.data, src.ctypes.data, pos.ctypes.data,
                                      seg_adapter.ctypes.data, seg_start.ctypes.data, counts.ctypes.data))
    U, Pv = int(counts[0]), int(counts[1])
    return {"tok": tok[:Pv], "adapter": adapter[:Pv], "alpha": alpha[:Pv], "src": src[:Pv],
            "pos": pos[:P], "seg_adapter": seg_adapter[:U], "seg_start": seg_start[:U + 1],
            "U": U, "P_valid": Pv, "status": int(counts[2])}


def lora_mapping_destroy(m: int):
    _check("lora_mapping_destroy", load().lora_mapping_destroy(m))


def lora_diag_wait_expiry(kind: int, limit_ns: int, words, stream=None):
    """words: device int32 [4] (words[1] = 0 for kind 1)."""
    _need("lora_diag_wait_expiry", "words", words, 4)
    _check("lora_diag_wait_expiry",
           load().lora_diag_wait_expiry(kind, limit_ns, _dptr(words, "words", "int32"), _stream(stream)))


def lora_version() -> str:
    return load().lora_version().decode()
