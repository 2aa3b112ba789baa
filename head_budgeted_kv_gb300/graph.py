"""A whole decode step captured in a CUDA graph.

The C ABI is capture-safe: lengths and positions are device tensors, launch shapes depend
only on the pool's static geometry, nothing is allocated inside a call, and the tensor-core
kernel launches as a programmatic dependent so consecutive layers keep their overlap inside
the graph.  ``DecodeStepGraph`` records, for every layer, the append of the new token and the
windowed attention (``hwkv_append_decode_attn``, or ``hwkv_append`` + ``hwkv_decode_attn``),
followed by the advance of the positions (``hwkv_advance_positions``), and replays that whole
step with one launch from the host: every kernel of a replayed step is the library's.
Inputs are read from, and outputs written to, the static buffers it owns.
"""
from __future__ import annotations

import torch


class DecodeStepGraph:
    """Captured decode step of every layer of ``pool``.

    Static buffers (fill them before ``replay``):
      q     [layers][B][q_heads][D]   queries of the step
      k_new [layers][B][kv_heads][D]  new keys, v_new likewise
      pos   [B] int32                 lengths before the append; the step adds 1 to them
    Output: out [layers][B][q_heads][D].
    """

    def __init__(self, pool, scale: float, q_heads: int, pos0, fused: bool = True):
        dev = pool.buffer.device
        L, B, H, D = pool.layers, pool.num_seqs, pool.kv_heads, pool.head_dim
        dt = pool.dtype
        self.pool = pool
        self.q = torch.zeros((L, B, q_heads, D), dtype=dt, device=dev)
        self.k_new = torch.zeros((L, B, H, D), dtype=dt, device=dev)
        self.v_new = torch.zeros_like(self.k_new)
        self.out = torch.zeros_like(self.q)
        self.pos = torch.as_tensor(pos0, dtype=torch.int32, device=dev).clone()
        self.lens = torch.empty_like(self.pos)
        if q_heads != pool.q_heads:
            pool.q_heads = q_heads
            pool._size_workspace()
        self.scale = float(scale)
        self.fused = fused
        self.graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            with torch.cuda.graph(self.graph, stream=side):
                self._record()
        torch.cuda.current_stream(dev).wait_stream(side)

    def _record(self):
        p = self.pool
        if not self.fused:
            p.advance_positions(self.pos, out=self.lens)  # lengths after the append
        for l in range(p.layers):
            if self.fused:
                # after layer 0 the kernel just before is the previous layer's attention, which
                # writes neither the positions nor this layer's pool
                p.append_decode(l, self.q[l], self.scale, self.k_new[l], self.v_new[l], self.pos, out=self.out[l],
                                early_reads=l > 0)
            else:
                p.append(l, self.k_new[l], self.v_new[l], self.pos)
                p.decode(l, self.q[l], self.scale, self.lens, out=self.out[l])
        p.advance_positions(self.pos)  # the next step's positions

    def replay(self):
        self.graph.replay()
