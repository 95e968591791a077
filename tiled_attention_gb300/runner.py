"""Run a seeded workload through the C ABI with torch-owned device (or pinned host) buffers.

Marshalling only: moves the workload's arrays to the device, allocates outputs and the decode
workspace, and calls attn_fwd. The arithmetic runs in the CUDA library.
"""
from __future__ import annotations

import numpy as np
import torch

from . import attn
from .inputs import MASK_PAGED_DECODE, MASK_PAGED_PREFILL, Workload


def bf16_tensor(a: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor (bit-exact)."""
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.to(device).view(torch.bfloat16)


class DeviceProblem:
    """A workload resident in device memory, with output and workspace buffers."""

    def __init__(self, w: Workload, device="cuda", fill_outputs=float("nan")):
        self.w = w
        self.device = torch.device(device)
        self.q = bf16_tensor(w.q, self.device)
        self.k = bf16_tensor(w.k, self.device)
        self.v = bf16_tensor(w.v, self.device)
        self.o = torch.full(w.out_shape, fill_outputs, dtype=torch.bfloat16, device=self.device)
        self.lse = torch.full(w.lse_shape, fill_outputs, dtype=torch.float32, device=self.device)
        self.cu = (None if w.cu_seqlens is None else
                   torch.from_numpy(np.ascontiguousarray(w.cu_seqlens, np.int32)).to(self.device))
        self.table = (None if w.block_table is None else
                      torch.from_numpy(np.ascontiguousarray(w.block_table, np.int32)).to(self.device))
        self.num_pages = (int(w.k.shape[0]) if w.mask_kind in (MASK_PAGED_DECODE,
                                                                 MASK_PAGED_PREFILL) else 0)
        self.seqlens_k = (None if w.seqlens_k is None else
                          torch.from_numpy(np.ascontiguousarray(w.seqlens_k, np.int32)).to(self.device))
        self.fp8 = w.q8 is not None
        if self.fp8:
            self.q8 = torch.from_numpy(np.ascontiguousarray(w.q8)).to(self.device)
            self.k8 = torch.from_numpy(np.ascontiguousarray(w.k8)).to(self.device)
            self.q_scales = torch.from_numpy(np.ascontiguousarray(w.q_scales, np.float32)).to(
                self.device)
            self.k_scales = torch.from_numpy(np.ascontiguousarray(w.k_scales, np.float32)).to(
                self.device)
        nbytes = (0 if w.mask_kind == MASK_PAGED_PREFILL else
                  attn.attn_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d, w.mask_kind, w.page_size))
        self.workspace = (torch.empty(max(nbytes, 16), dtype=torch.uint8, device=self.device)
                          if nbytes else None)

    def run(self, stream=None) -> int:
        w = self.w
        if self.fp8:
            return attn.attn_fwd_fp8(self.q8, self.k8, self.v, self.o, self.lse, self.q_scales,
                                     self.k_scales, w.B, w.Hq, w.Hkv, w.N, w.d, w.scale,
                                     w.mask_kind, w.window, stream)
        if w.mask_kind == MASK_PAGED_PREFILL:
            return attn.attn_fwd_paged_prefill(self.q, self.k, self.v, self.o, self.lse, w.B,
                                               w.Hq, w.Hkv, w.N, w.d, w.scale, self.cu,
                                               self.seqlens_k, self.table,
                                               int(w.block_table.shape[1]), w.page_size,
                                               self.num_pages, stream)
        return attn.attn_fwd(self.q, self.k, self.v, self.o, self.lse, w.B, w.Hq, w.Hkv, w.N, w.d,
                             w.scale, w.mask_kind, w.window, self.cu, self.table, w.page_size,
                             self.num_pages, self.workspace, stream)

    def outputs(self):
        """(O as float64 numpy [rows, d], LSE float64 [rows]) in the oracle's row order."""
        o = self.o.float().reshape(-1, self.w.d).cpu().numpy().astype(np.float64)
        lse = self.lse.reshape(-1).cpu().numpy().astype(np.float64)
        return o, lse
