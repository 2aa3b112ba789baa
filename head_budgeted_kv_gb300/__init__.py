"""hwkv: per-head budgeted KV residency on one GB300.

The grouped-cache runtime of "HeadWiseKV: Budgeted Per-Head Cache Residency for Hybrid
Long-Context Language Models" (blog summary; abstract and section "Grouped-Cache
Runtime"): every KV head of a global-attention layer keeps a static window of its most
recent tokens in ceil(w / block_size) paged blocks, and decode attention reads only that
resident window.

``binding`` exposes the C ABI of ``include/hwkv.h`` under the same names; ``Pool`` below
is a convenience wrapper that owns the device buffers (allocated with torch).
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding
from .binding import (HWKV_BF16, HWKV_F32, HWKV_KERNEL_AUTO, HWKV_KERNEL_SIMT, HWKV_KERNEL_TENSOR, DecodeLaunch, HwkvError,
                      hwkv_abi_version, hwkv_advance_positions, hwkv_append, hwkv_append_decode_attn, hwkv_block_table,
                      hwkv_check_device_errors, hwkv_kernel_launches,
                      hwkv_decode_attn, hwkv_decode_workspace_bytes, hwkv_materialize, hwkv_pool_bytes,
                      hwkv_pool_create, hwkv_pool_destroy, hwkv_pool_geometry, hwkv_prefill_attn,
                      hwkv_prefill_plan, hwkv_prefill_workspace_bytes, hwkv_set_block_table, hwkv_set_decode_config,
                      hwkv_set_prefill_config, hwkv_wait_selftest)

__all__ = [
    "Pool", "DecodeLaunch", "HwkvError", "binding", "HWKV_F32", "HWKV_BF16", "HWKV_KERNEL_AUTO", "HWKV_KERNEL_TENSOR",
    "HWKV_KERNEL_SIMT", "hwkv_abi_version", "hwkv_advance_positions", "hwkv_append", "hwkv_append_decode_attn", "hwkv_block_table",
    "hwkv_check_device_errors", "hwkv_kernel_launches",
    "hwkv_decode_attn", "hwkv_decode_workspace_bytes", "hwkv_materialize", "hwkv_pool_bytes", "hwkv_pool_create",
    "hwkv_pool_destroy", "hwkv_pool_geometry", "hwkv_prefill_attn", "hwkv_prefill_plan", "hwkv_prefill_workspace_bytes",
    "hwkv_set_block_table", "hwkv_set_decode_config", "hwkv_set_prefill_config", "hwkv_wait_selftest",
]


class Pool:
    """A per-head paged KV pool on the current CUDA device.

    The pool buffer is one torch uint8 allocation of exactly ``hwkv_pool_bytes`` bytes
    (the pre-serving prediction), bound with ``hwkv_pool_create``.
    """

    def __init__(self, layers: int, kv_heads: int, head_dim: int, block_size: int, windows, num_seqs: int,
                 dtype: torch.dtype, q_heads: Optional[int] = None, device=None, stream=None):
        self.layers, self.kv_heads, self.head_dim = layers, kv_heads, head_dim
        self.block_size, self.num_seqs, self.dtype = block_size, num_seqs, dtype
        self.q_heads = q_heads or kv_heads
        self.nbytes = hwkv_pool_bytes(layers, kv_heads, head_dim, block_size, windows, num_seqs, dtype)
        device = torch.device(device or "cuda")
        self.buffer = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.handle = hwkv_pool_create(layers, kv_heads, head_dim, block_size, windows, num_seqs, dtype,
                                       self.buffer, stream)
        self.workspace = None
        self.prefill_workspace = None
        self._size_workspace()

    def _size_workspace(self):
        need = hwkv_decode_workspace_bytes(self.handle, self.q_heads)
        if self.workspace is None or self.workspace.numel() < need:
            self.workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=self.buffer.device)

    def set_decode_config(self, split_tokens: int = 0, kernel: int = HWKV_KERNEL_AUTO, workers: int = 0):
        hwkv_set_decode_config(self.handle, split_tokens, workers, kernel)
        self._size_workspace()

    def geometry(self):
        return hwkv_pool_geometry(self.handle)

    def blocks(self) -> torch.Tensor:
        """View of the pool as [total_blocks][2][block_size][head_dim] elements."""
        _, total, _ = self.geometry()
        return self.buffer.view(self.dtype).view(total, 2, self.block_size, self.head_dim)

    def block_table(self, seq: int, layer: int, kv_head: int):
        return hwkv_block_table(self.handle, seq, layer, kv_head)

    def set_block_table(self, table, stream=None):
        hwkv_set_block_table(self.handle, table, stream)

    def materialize(self, layer: int, k_full, v_full, lens, stream=None):
        hwkv_materialize(self.handle, layer, k_full, v_full, lens, stream)

    def append(self, layer: int, k_new, v_new, pos, stream=None):
        hwkv_append(self.handle, layer, k_new, v_new, pos, stream)

    def decode(self, layer: int, q, scale: float, lens, out=None, stream=None, early_reads: bool = False):
        if out is None:
            out = torch.empty_like(q)
        if q.shape[1] != self.q_heads:
            self.q_heads = q.shape[1]
            self._size_workspace()
        hwkv_decode_attn(self.handle, layer, q, scale, lens, out, self.workspace, stream, early_reads)
        return out

    def append_decode(self, layer: int, q, scale: float, k_new, v_new, pos, out=None, stream=None,
                      early_reads: bool = False):
        """Append the new token (positions ``pos``) and decode at ``pos + 1`` in one call.
        early_reads: the caller's guarantee of HWKV_DECODE_EARLY_READS (lengths, block table
        and this layer's pool not written by the kernel just before in the stream)."""
        if out is None:
            out = torch.empty_like(q)
        if q.shape[1] != self.q_heads:
            self.q_heads = q.shape[1]
            self._size_workspace()
        hwkv_append_decode_attn(self.handle, layer, q, scale, k_new, v_new, pos, out, self.workspace, stream,
                                early_reads)
        return out

    def decode_launch(self, layer: int, q, scale: float, lens, out, k_new=None, v_new=None, stream=None,
                      early_reads: bool = False) -> DecodeLaunch:
        """A prepared launch of decode (k_new None, ``lens`` = lengths after the append) or of the
        fused append + decode (``lens`` = positions) on fixed buffers: calling it launches."""
        if q.shape[1] != self.q_heads:
            self.q_heads = q.shape[1]
            self._size_workspace()
        return DecodeLaunch(self.handle, layer, q, scale, lens, out, self.workspace, k_new, v_new, stream, early_reads)

    def prefill(self, layer: int, q, scale: float, k_new, v_new, pos, n, out=None, stream=None):
        """Chunked prefill: q [B][n_max][Hq][D], k_new/v_new [B][n_max][Hkv][D]; pos, n int32 [B].
        Keeps a workspace for the split of long key streams, grown on demand."""
        if out is None:
            out = torch.zeros_like(q)
        need = hwkv_prefill_workspace_bytes(self.handle, layer, q.shape[2], q.shape[1])
        if need and (self.prefill_workspace is None or self.prefill_workspace.numel() < need):
            self.prefill_workspace = torch.empty(need, dtype=torch.uint8, device=self.buffer.device)
        hwkv_prefill_attn(self.handle, layer, q, scale, k_new, v_new, pos, n, out,
                          self.prefill_workspace if need else None, stream)
        return out

    def set_prefill_config(self, max_stages: int = 0):
        hwkv_set_prefill_config(self.handle, max_stages)

    def advance_positions(self, pos, out=None, delta: int = 1, stream=None):
        """out = pos + delta on the device with a library kernel (in place when out is None)."""
        out = pos if out is None else out
        hwkv_advance_positions(self.handle, pos, out, delta, stream)
        return out

    def check_device_errors(self, stream=None) -> int:
        return hwkv_check_device_errors(self.handle, stream)

    def close(self):
        if getattr(self, "handle", None):
            hwkv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
