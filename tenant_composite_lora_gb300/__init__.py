"""GB300 (sm_103a) composite multi-LoRA delta.

    y_t += sum over token t's pairs (i, alpha) of alpha * (x_t A_i[:, :k_i]) B_i[:k_i, :]

The compute lives in libtclora.so (hand-written CUDA, C ABI in
include/lora.h).  ``native`` binds it with ctypes under the C names;
``LoraPool`` / ``LoraMapping`` / ``delta_apply`` are small conveniences over
torch tensors.  Importing this package does not load the library; the first
call does, and fails loudly if it has not been built.
"""
from __future__ import annotations

from . import native
from .native import (LoraError, lora_build_mapping, lora_delta_apply, lora_delta_apply_host,
                     lora_delta_apply_noalloc, lora_delta_apply_path, lora_dispatch_choose, lora_mapping_create,
                     lora_mapping_destroy, lora_mapping_export, lora_mapping_status,
                     lora_pool_create, lora_pool_destroy, lora_pool_register,
                     lora_pool_unregister, lora_version, lora_diag_wait_expiry, lora_delta_apply_multi,
                     lora_ablation_workspace_bytes, lora_delta_apply_ablation, lora_gate_logits, lora_gate_topk,
                     lora_recompress_workspace_bytes, lora_recompress, lora_rank_allocate)

__all__ = [
    "native", "LoraError", "LoraPool", "LoraMapping", "delta_apply",
    "lora_pool_create", "lora_pool_register", "lora_pool_unregister", "lora_pool_destroy",
    "lora_mapping_create", "lora_build_mapping", "lora_delta_apply", "lora_delta_apply_path",
    "lora_dispatch_choose", "lora_delta_apply_host", "lora_mapping_status", "lora_mapping_export",
    "lora_mapping_destroy", "lora_version", "lora_delta_apply_noalloc", "lora_diag_wait_expiry",
    "lora_delta_apply_multi", "lora_ablation_workspace_bytes", "lora_delta_apply_ablation",
    "lora_gate_logits", "lora_gate_topk", "lora_recompress_workspace_bytes", "lora_recompress",
    "lora_rank_allocate",
]


class LoraPool:
    """Owns a device adapter pool (lora_pool_create / lora_pool_destroy)."""

    def __init__(self, d_in: int, d_out: int, r_max: int, capacity: int):
        self.d_in, self.d_out, self.r_max, self.capacity = d_in, d_out, r_max, capacity
        self.handle = lora_pool_create(d_in, d_out, r_max, capacity)

    def register(self, slot: int, A, B, k: int, stream=None):
        """A: bf16 CUDA tensor [d_in, r_max]; B: bf16 CUDA tensor [r_max, d_out]."""
        assert tuple(A.shape) == (self.d_in, self.r_max) and tuple(B.shape) == (self.r_max, self.d_out)
        assert A.is_contiguous() and B.is_contiguous()
        lora_pool_register(self.handle, slot, A, B, int(k), stream)

    def unregister(self, slot: int, stream=None):
        lora_pool_unregister(self.handle, slot, stream)

    def close(self):
        if self.handle:
            lora_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass


class LoraMapping:
    """Owns a mapping workspace (lora_mapping_create / lora_mapping_destroy)."""

    def __init__(self, max_tokens: int, max_pairs: int, capacity: int):
        self.capacity = capacity
        self.handle = lora_mapping_create(max_tokens, max_pairs, capacity)
        self.T = self.P = 0

    def build(self, offsets, ids, alpha, stream=None):
        """offsets int32 [T+1], ids int32 [P], alpha float32 [P]: CUDA tensors."""
        if offsets.dim() != 1 or ids.dim() != 1 or alpha.dim() != 1 or offsets.shape[0] < 1:
            raise ValueError("build: offsets, ids and alpha are 1-D, offsets of length T + 1 >= 1")
        T, P = offsets.shape[0] - 1, ids.shape[0]
        if alpha.shape[0] != P:
            raise ValueError(f"build: alpha has {alpha.shape[0]} entries for {P} ids")
        lora_build_mapping(self.handle, offsets, ids, alpha, T, P, stream)
        self.T, self.P = T, P

    def status(self, stream=None) -> int:
        return lora_mapping_status(self.handle, stream)

    def export(self, stream=None) -> dict:
        return lora_mapping_export(self.handle, self.P, self.capacity, stream)

    def close(self):
        if self.handle:
            lora_mapping_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass


def delta_apply(x, y, pool: LoraPool, mapping: LoraMapping, ranks=None, path: int = 0, stream=None):
    """In place: y += composite delta (bf16 CUDA tensors [T, d_in], [T, d_out],
    T of the mapping's last build; ranks: None or int32 [capacity])."""
    T = mapping.T
    if x.dim() != 2 or x.shape[0] < T or x.shape[1] != pool.d_in:
        raise ValueError(f"delta_apply: x must be [>= {T}, {pool.d_in}], got {tuple(x.shape)}")
    if y.dim() != 2 or y.shape[0] < T or y.shape[1] != pool.d_out:
        raise ValueError(f"delta_apply: y must be [>= {T}, {pool.d_out}], got {tuple(y.shape)}")
    if ranks is not None and ranks.numel() < pool.capacity:
        raise ValueError(f"delta_apply: ranks must hold {pool.capacity} entries, got {ranks.numel()}")
    lora_delta_apply_path(x, y, pool.handle, ranks, mapping.handle, path, stream)
    return y
