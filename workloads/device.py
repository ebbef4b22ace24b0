"""Moves a seeded workload onto the GPU through the library's public API
(pool registration, mapping build).  Data movement only."""
from __future__ import annotations

import numpy as np


def _t(a, dtype, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device).view(dtype) \
        if dtype is torch.bfloat16 else torch.from_numpy(np.ascontiguousarray(a)).to(device=device)


def bf16_tensor(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_to_numpy_bits(t) -> np.ndarray:
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceWorkload:
    """A workload resident on the GPU: pool (all slots registered), pair
    lists, x, y, and a mapping object sized for it."""

    def __init__(self, wl, device="cuda", stream=None, register_ranks=None, max_tokens=None,
                 max_pairs=None, build=True):
        import torch
        import tenant_composite_lora_gb300 as tcl
        self.wl = wl
        self.device = device
        ranks = wl.ranks if register_ranks is None else register_ranks
        self.pool = tcl.LoraPool(wl.d_in, wl.d_out, wl.r_max, wl.capacity)
        for a in range(wl.capacity):
            if ranks[a] < 0:
                continue
            A = bf16_tensor(wl.A[a], device)
            B = bf16_tensor(wl.B[a], device)
            self.pool.register(a, A, B, int(ranks[a]), stream)
        torch.cuda.synchronize()
        self.offsets = torch.from_numpy(wl.offsets).to(device)
        self.ids = torch.from_numpy(wl.ids).to(device)
        self.alpha = torch.from_numpy(wl.alpha).to(device)
        self.x = bf16_tensor(wl.x, device)
        self.y0 = bf16_tensor(wl.y, device)
        self.mapping = tcl.LoraMapping(max(wl.T, max_tokens or 0), max(wl.P, max_pairs or 0), wl.capacity)
        if build:
            self.mapping.build(self.offsets, self.ids, self.alpha, stream)

    def apply(self, y=None, ranks=None, path=0, stream=None):
        """Returns a fresh y (copy of y_in) with the delta applied."""
        import tenant_composite_lora_gb300 as tcl
        y = self.y0.clone() if y is None else y
        tcl.delta_apply(self.x, y, self.pool, self.mapping, ranks=ranks, path=path, stream=stream)
        return y

    def close(self):
        self.mapping.close()
        self.pool.close()
