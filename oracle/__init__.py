"""fp64 CPU oracle for the composite multi-LoRA delta (plain C, loaded with ctypes).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  Nothing in the product library imports
it, and it imports nothing from the product library.

``compile_oracle()`` builds ``_build/liblora_oracle.so`` from
``lora_oracle.c`` with gcc (OpenMP when available, no FMA contraction, no
fast-math), on first use or when the source is newer than the library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liblora_oracle.so")
_lib = None

BAD_ID, BAD_OFFSETS, UNREGISTERED, BAD_RANK = 1, 2, 4, 8


def compile_oracle(force: bool = False) -> str:
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(compile_oracle())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.orc_delta_apply.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, I]
        lib.orc_delta_apply.restype = I
        lib.orc_build_mapping.argtypes = [I, I, I, P, P, P, P, P, P, P, P, P, P, P]
        lib.orc_build_mapping.restype = I
        lib.orc_round_bf16.argtypes = [ctypes.c_double]
        lib.orc_round_bf16.restype = ctypes.c_uint16
        lib.orc_gate_logits.argtypes = [I, I, I, P, P, P, P]
        lib.orc_gate_logits.restype = None
        lib.orc_gate_topk.argtypes = [I, I, I, P, P, P, P, P]
        lib.orc_gate_topk.restype = I
        lib.orc_max_threads.argtypes = []
        lib.orc_max_threads.restype = I
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().orc_max_threads())


def round_bf16(v: float) -> int:
    """bf16 bit pattern nearest to the fp64 value v (ties to even)."""
    return int(_load().orc_round_bf16(float(v)))


def delta_apply(offsets, ids, alpha, x, A, B, ranks, y_in, *, d_in, d_out, r_max, capacity,
                threads: int = 1, want_acc: bool = True):
    """Returns (y_out bf16 bits [T, d_out], acc fp64 [T, d_out] or None, status)."""
    offsets = _c(offsets, np.int32)
    ids = _c(ids, np.int32)
    alpha = _c(alpha, np.float32)
    x = _c(x, np.uint16)
    A = _c(A, np.uint16)
    B = _c(B, np.uint16)
    ranks = _c(ranks, np.int32)
    y_in = _c(y_in, np.uint16)
    T = offsets.shape[0] - 1
    P = ids.shape[0]
    assert x.shape == (T, d_in) and y_in.shape == (T, d_out)
    assert A.shape == (capacity, d_in, r_max) and B.shape == (capacity, r_max, d_out)
    assert ranks.shape == (capacity,) and alpha.shape == (P,)
    y_out = np.empty((T, d_out), dtype=np.uint16)
    acc = np.empty((T, d_out), dtype=np.float64) if want_acc else None
    st = _load().orc_delta_apply(T, P, d_in, d_out, r_max, capacity, _ptr(offsets), _ptr(ids),
                                 _ptr(alpha), _ptr(x), _ptr(A), _ptr(B), _ptr(ranks), _ptr(y_in),
                                 _ptr(y_out), _ptr(acc) if acc is not None else None, threads)
    return y_out, acc, int(st)


def build_mapping(offsets, ids, alpha, *, capacity):
    """Returns a dict with the ordered tuples, pos, segments, U, P_valid, status."""
    offsets = _c(offsets, np.int32)
    ids = _c(ids, np.int32)
    alpha = _c(alpha, np.float32)
    T = offsets.shape[0] - 1
    P = ids.shape[0]
    n = max(P, 1)
    s_tok = np.zeros(n, np.int32)
    s_adapter = np.zeros(n, np.int32)
    s_alpha = np.zeros(n, np.float32)
    s_src = np.zeros(n, np.int32)
    pos = np.zeros(n, np.int32)
    seg_adapter = np.zeros(max(min(P, capacity), 1), np.int32)
    seg_start = np.zeros(max(min(P, capacity), 1) + 1, np.int32)
    counts = np.zeros(2, np.int32)
    st = _load().orc_build_mapping(T, P, capacity, _ptr(offsets), _ptr(ids), _ptr(alpha),
                                   _ptr(s_tok), _ptr(s_adapter), _ptr(s_alpha), _ptr(s_src),
                                   _ptr(pos), _ptr(seg_adapter), _ptr(seg_start), _ptr(counts))
    U, Pv = int(counts[0]), int(counts[1])
    return {
        "tok": s_tok[:Pv].copy(), "adapter": s_adapter[:Pv].copy(),
        "alpha": s_alpha[:Pv].copy(), "src": s_src[:Pv].copy(), "pos": pos[:P].copy(),
        "seg_adapter": seg_adapter[:U].copy(), "seg_start": seg_start[:U + 1].copy(),
        "U": U, "P_valid": Pv, "status": int(st),
    }


def gate_logits(x, Wg, req):
    """fp64 logits [T, E]: x bf16 bits [T, d_in], Wg bf16 bits [R, E, d_in], req int32 [T]."""
    x = _c(x, np.uint16)
    Wg = _c(Wg, np.uint16)
    req = _c(req, np.int32)
    T, d_in = x.shape
    E = Wg.shape[1]
    out = np.empty((T, E), np.float64)
    _load().orc_gate_logits(T, E, d_in, _ptr(x), _ptr(Wg), _ptr(req), _ptr(out))
    return out


def gate_topk(logits, cand, top_k: int):
    """(offsets [T+1], ids [T*top_k], alpha [T*top_k], tokens without a
    valid candidate) from fp32 logits [T, E] and candidate ids [T, E]
    (-1 = padding)."""
    logits = _c(logits, np.float32)
    cand = _c(cand, np.int32)
    T, E = logits.shape
    offsets = np.empty(T + 1, np.int32)
    ids = np.empty(max(T * top_k, 1), np.int32)
    alpha = np.empty(max(T * top_k, 1), np.float32)
    empty = _load().orc_gate_topk(T, E, top_k, _ptr(logits), _ptr(cand), _ptr(offsets), _ptr(ids), _ptr(alpha))
    return offsets, ids[: T * top_k], alpha[: T * top_k], int(empty)


def apply_workload(wl, ranks=None, threads: int = 1, want_acc: bool = True, y_in=None):
    """Convenience: the oracle on a ``workloads.Workload``."""
    r = wl.ranks if ranks is None else ranks
    return delta_apply(wl.offsets, wl.ids, wl.alpha, wl.x, wl.A, wl.B, r,
                       wl.y if y_in is None else y_in, d_in=wl.d_in, d_out=wl.d_out,
                       r_max=wl.r_max, capacity=wl.capacity, threads=threads, want_acc=want_acc)


def apply_tokens(wl, tokens, ranks=None, threads: int = 1):
    """The oracle on a subset of tokens (their own pair lists); returns
    (y_out [len(tokens), d_out], acc, status).  Used for sampled parity at
    full size."""
    tokens = np.asarray(tokens, dtype=np.int64)
    lists_ids, lists_alpha = [], []
    for t in tokens:
        a, b = int(wl.offsets[t]), int(wl.offsets[t + 1])
        lists_ids.append(wl.ids[a:b])
        lists_alpha.append(wl.alpha[a:b])
    offs = np.zeros(len(tokens) + 1, np.int32)
    offs[1:] = np.cumsum([len(l) for l in lists_ids])
    ids = np.concatenate(lists_ids) if lists_ids else np.zeros(0, np.int32)
    al = np.concatenate(lists_alpha) if lists_alpha else np.zeros(0, np.float32)
    r = wl.ranks if ranks is None else ranks
    return delta_apply(offs, ids, al, wl.x[tokens], wl.A, wl.B, r, wl.y[tokens],
                       d_in=wl.d_in, d_out=wl.d_out, r_max=wl.r_max, capacity=wl.capacity, threads=threads)
