"""Torch-side convenience around the C ABI: owns the device arena and the base
buffer as torch tensors and marshals numpy inputs into library calls.
PyTorch provides device memory and streams only; all computation is libovl's."""
from __future__ import annotations

import numpy as np
import torch

from . import (OVL_BF16, OVL_F32, OVL_MODE_STACK, OVL_PATH_DUAL, OVL_SWITCH_REJECT, OvlError, check,
               ovl_activate, ovl_base_digest, ovl_check_device, ovl_create, ovl_destroy, ovl_get_state,
               ovl_linear_forward, ovl_load_base, ovl_rollback, ovl_stage_adapter, ovl_stage_sparse,
               ovl_unstage_adapter)


def stream_handle(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


class Runtime:
    """One context on one device with a caller-owned arena."""

    def __init__(self, arena_bytes: int = 256 << 20, device: int = 0, policy: int = OVL_SWITCH_REJECT):
        self.device = torch.device("cuda", device)
        self.arena = torch.empty(arena_bytes, dtype=torch.uint8, device=self.device)
        st, self.ctx = ovl_create(device, self.arena.data_ptr(), arena_bytes, policy)
        if st != 0:
            raise OvlError(st, "ovl_create failed")
        self.base = None
        self.tensors = []

    def close(self):
        if self.ctx:
            ovl_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_base(self, quant: int, tensors, buf: np.ndarray, digest: bytes, copies: int = 1) -> int:
        """Upload the base bytes and register them.  With copies > 1 extra
        identical device copies are kept (self.base_copies) for benchmarks that
        rotate among them."""
        self.base = torch.from_numpy(np.ascontiguousarray(buf)).to(self.device)
        self.base_copies = [self.base] + [self.base.clone() for _ in range(copies - 1)]
        self.tensors = [tuple(int(v) for v in t) for t in tensors]
        return ovl_load_base(self.ctx, quant, self.tensors, self.base.data_ptr(), self.base.numel(), digest,
                             stream_handle())

    def stage(self, ad, digest: bytes, required_base: bytes | None = None):
        return ovl_stage_adapter(self.ctx, ad.targets, ad.ranks, ad.a_off, ad.b_off, ad.payload, digest,
                                 required_base)

    def stage_sparse(self, sp, digest: bytes, required_base: bytes | None = None):
        return ovl_stage_sparse(self.ctx, sp.targets, sp.nnz, sp.idx_off, sp.val_off, sp.payload, digest,
                                required_base)

    def unstage(self, h):
        return ovl_unstage_adapter(self.ctx, h)

    def activate(self, handles, scales, mode: int = OVL_MODE_STACK):
        return ovl_activate(self.ctx, handles, scales, mode)

    def rollback(self):
        return ovl_rollback(self.ctx)

    def base_digest(self):
        return ovl_base_digest(self.ctx, stream_handle())

    def state(self):
        return ovl_get_state(self.ctx)[1]

    def check_device(self):
        return ovl_check_device(self.ctx, stream_handle())

    def forward(self, tensor: int, x: torch.Tensor, path: int = OVL_PATH_DUAL, scratch: torch.Tensor | None = None,
                y: torch.Tensor | None = None) -> torch.Tensor:
        """x: device tensor [T][d_in] float32 or bfloat16 -> y float32 [T][d_out]."""
        d_out = self.tensors[tensor][2]
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, d_out), dtype=torch.float32, device=self.device)
        xdt = OVL_BF16 if x.dtype == torch.bfloat16 else OVL_F32
        sp, sb = (scratch.data_ptr(), scratch.numel() * scratch.element_size()) if scratch is not None else (0, 0)
        check(ovl_linear_forward(self.ctx, tensor, x.data_ptr(), xdt, T, y.data_ptr(), path, sp, sb,
                                 stream_handle()), self.ctx)
        return y
