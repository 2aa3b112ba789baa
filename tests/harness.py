"""Drives a workload through the CUDA path and computes the oracle's answer for the
same seeded inputs.  Used by the GPU parity tests."""
from __future__ import annotations

import dataclasses
from typing import Dict, Iterable, Optional

import numpy as np
import torch

import oracle
import workloads
import head_budgeted_kv_gb300 as hw

BF16_ATOL = 2e-2
BF16_RTOL = 2e-2
F32_ATOL = 1e-5


def tolerance(cfg):
    """(atol, rtol): pass iff |gpu - ref| <= atol + rtol * |ref| elementwise."""
    return (F32_ATOL, 0.0) if cfg.dtype == "f32" else (BF16_ATOL, BF16_RTOL)


def assert_close(got: np.ndarray, ref: np.ndarray, cfg, what: str = ""):
    atol, rtol = tolerance(cfg)
    bad = np.abs(got - ref) > atol + rtol * np.abs(ref)
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; first at "
                             f"{tuple(idx)}: gpu {got[tuple(idx)]!r} oracle {ref[tuple(idx)]!r}; "
                             f"max |err| {np.abs(got - ref).max():.3e}")


def small_config(name="small", cfg_id=90, layers=1, kv_heads=2, group=4, head_dim=128, block_size=16,
                 dtype="bf16", windows=((64, 200),), prefill=(300,), steps=2, spike_frac=0.0):
    return workloads.Config(name, cfg_id, layers=layers, kv_heads=kv_heads, q_heads=kv_heads * group,
                            head_dim=head_dim, block_size=block_size, dtype=dtype, batch=len(prefill),
                            steps=steps, windows=tuple(tuple(int(x) for x in r) for r in windows),
                            prefill=tuple(int(x) for x in prefill), spike_frac=spike_frac)


class Run:
    """One pool driven through materialise, then append + decode per step."""

    def __init__(self, cfg, kernel=hw.HWKV_KERNEL_AUTO, split=0, canary: Optional[int] = None,
                 keep_host_steps=True, workers=0, fused=False):
        self.cfg = cfg
        self.dev = torch.device("cuda", torch.cuda.current_device())
        gen_dev = "cpu" if cfg.single_cpu_stream else self.dev
        self.wl = workloads.Workload(cfg, device=gen_dev)
        self.pool = hw.Pool(cfg.layers, cfg.kv_heads, cfg.head_dim, cfg.block_size, cfg.windows_array(), cfg.batch,
                            cfg.torch_dtype, q_heads=cfg.q_heads, device=self.dev)
        self.pool.set_decode_config(split, kernel, workers)
        self.fused = fused
        if canary is not None:
            self.pool.buffer.fill_(canary)
            torch.cuda.synchronize()
        self.prefill = torch.tensor(cfg.prefill, dtype=torch.int32, device=self.dev)
        self.steps_done = 0
        self.host_steps = [] if keep_host_steps else None
        self._pre_cache: Dict = {}

    # -- path --------------------------------------------------------------------------
    def materialize(self, layers: Optional[Iterable[int]] = None):
        for l in (range(self.cfg.layers) if layers is None else layers):
            K, V = self.wl.prefill_layer(l, self.dev)
            self.pool.materialize(l, K, V, self.prefill)
            del K, V

    def step(self, keep_layers: Iterable[int] = ()):
        """One decode step over all layers; returns {layer: (q raw host, out host float64)}."""
        i = self.steps_done
        q, kn, vn = self.wl.step_inputs(i, self.dev)
        if self.host_steps is not None:
            self.host_steps.append((None, kn.cpu(), vn.cpu()))
        pos = self.prefill + i
        lens = pos + 1
        keep = set(keep_layers)
        res = {}
        for l in range(self.cfg.layers):
            if self.fused:
                out = self.pool.append_decode(l, q[l], self.cfg.scale, kn[l], vn[l], pos)
            else:
                self.pool.append(l, kn[l], vn[l], pos)
                out = self.pool.decode(l, q[l], self.cfg.scale, lens)
            if l in keep:
                res[l] = (workloads.to_raw(q[l]), out.float().cpu().double().numpy())
        self.steps_done += 1
        return res

    def run_prepared(self, keep_steps: Iterable[int] = (), keep_layers: Iterable[int] = (), pairs=None):
        """All remaining steps as the decode benchmark issues them: every step's inputs and
        positions prepared first, then one prepared fused launch per layer with early reads,
        back to back with no host synchronisation.  Returns {(step, layer): (q raw, out)} for
        keep_steps x keep_layers, or for the (step, layer) pairs given."""
        cfg = self.cfg
        first = self.steps_done
        steps = range(first, cfg.steps)
        inputs = []
        for i in steps:
            q, kn, vn = self.wl.step_inputs(i, self.dev)
            if self.host_steps is not None:
                self.host_steps.append((None, kn.cpu(), vn.cpu()))
            inputs.append((q, kn, vn, (self.prefill + i).contiguous()))
        outs = torch.empty((len(inputs), cfg.layers, cfg.batch, cfg.q_heads, cfg.head_dim),
                           dtype=cfg.torch_dtype, device=self.dev)
        launches = [[self.pool.decode_launch(l, q[l], cfg.scale, pos, outs[j, l], kn[l], vn[l], early_reads=True)
                     for l in range(cfg.layers)] for j, (q, kn, vn, pos) in enumerate(inputs)]
        torch.cuda.synchronize()
        for step in launches:
            for launch in step:
                launch()
        torch.cuda.synchronize()
        self.steps_done = cfg.steps
        res = {}
        want = sorted(pairs) if pairs is not None else [(i, l) for i in keep_steps for l in keep_layers]
        for i, l in want:
            res[(i, l)] = (workloads.to_raw(inputs[i - first][0][l]),
                           outs[i - first, l].float().cpu().double().numpy())
        return res

    def device_errors(self) -> int:
        return self.pool.check_device_errors()

    # -- oracle side -------------------------------------------------------------------------
    def _prefill_host(self, l, s):
        key = (l, s)
        if key not in self._pre_cache:
            self._pre_cache = {k: v for k, v in self._pre_cache.items() if k[0] == l}
            self._pre_cache[key] = self.wl.prefill_seq(l, s, self.dev)
        return self._pre_cache[key]

    def history(self, l, s, h, lo, hi):
        if hi <= lo:
            empty = workloads.to_raw(torch.zeros((0, self.cfg.head_dim), dtype=self.cfg.torch_dtype))
            return empty, empty
        pre = self._prefill_host(l, s) if lo < self.cfg.prefill[s] else None
        return self.wl.history(l, s, h, lo, hi, prefill=pre, steps=self.host_steps)

    def reference(self, step: int, layer: int, q_raw: np.ndarray, seqs=None) -> np.ndarray:
        """Oracle output [B][Hq][D] (fp64) of decode step ``step`` (0-based) of ``layer``."""
        cfg = self.cfg
        lens = [cfg.prefill[s] + step + 1 for s in range(cfg.batch)]
        hist = {}
        for s in range(cfg.batch):
            for h in range(cfg.kv_heads):
                lo, hi = oracle.window_span(lens[s], int(cfg.windows[layer][h]))
                if seqs is not None and s not in seqs:
                    lo = hi  # empty: not checked
                hk, hv = self.history(layer, s, h, lo, hi)
                hist[(s, h)] = (lo, hk, hv)
        if seqs is None:
            return oracle.attention_jobs(q_raw, hist, lens, cfg.windows[layer], cfg.scale)
        lens_used = [lens[s] if s in seqs else 0 for s in range(cfg.batch)]
        return oracle.attention_jobs(q_raw, hist, lens_used, cfg.windows[layer], cfg.scale)

    def layer_histories(self, layer: int, seqs=None) -> dict:
        """Host rows of every (seq, kv head) of ``layer`` covering the windows of all steps done:
        {(s, h): (p_lo, K rows, V rows)} from the oldest position any step's window holds to the
        newest appended one (drawn once, then sliced per step by ``reference_hoisted``)."""
        cfg = self.cfg
        out = {}
        for s in range(cfg.batch):
            if seqs is not None and s not in seqs:
                continue
            hi = cfg.prefill[s] + self.steps_done
            for h in range(cfg.kv_heads):
                lo, _ = oracle.window_span(cfg.prefill[s] + 1, int(cfg.windows[layer][h]))
                hk, hv = self.history(layer, s, h, lo, hi)
                out[(s, h)] = (lo, hk, hv)
        return out

    def reference_hoisted(self, hist_all: dict, step: int, layer: int, q_raw: np.ndarray, seqs=None) -> np.ndarray:
        """As ``reference``, with each head's rows sliced out of ``layer_histories``."""
        cfg = self.cfg
        lens = [cfg.prefill[s] + step + 1 for s in range(cfg.batch)]
        hist = {}
        empty = workloads.to_raw(torch.zeros((0, cfg.head_dim), dtype=cfg.torch_dtype))
        for s in range(cfg.batch):
            for h in range(cfg.kv_heads):
                lo, hi = oracle.window_span(lens[s], int(cfg.windows[layer][h]))
                if seqs is not None and s not in seqs:
                    hist[(s, h)] = (hi, empty, empty)
                    continue
                p_lo, hk, hv = hist_all[(s, h)]
                hist[(s, h)] = (lo, hk[lo - p_lo:hi - p_lo], hv[lo - p_lo:hi - p_lo])
        lens_used = lens if seqs is None else [lens[s] if s in seqs else 0 for s in range(cfg.batch)]
        return oracle.attention_jobs(q_raw, hist, lens_used, cfg.windows[layer], cfg.scale)

    def expected_ring_blocks(self, l, s, h):
        """Oracle contents of the blocks of (layer, seq, head) after the steps so far."""
        cfg = self.cfg
        L = cfg.prefill[s]
        w = int(cfg.windows[l][h])
        C = int(oracle.ring_capacity([[w]], cfg.block_size)[0, 0])
        writes = list(oracle.materialized_positions(L, w)) + list(oracle.appended_positions(L, self.steps_done))
        lo = writes[0] if writes else 0
        hk, hv = self.history(l, s, h, lo, L + self.steps_done)
        rk, rv = oracle.ring_after_writes(hk, hv, lo, writes, C)
        return oracle.ring_to_blocks(rk, rv, cfg.block_size), writes, C

    def gpu_blocks(self, ids) -> np.ndarray:
        blocks = self.pool.blocks()
        idx = torch.as_tensor(np.asarray(ids, dtype=np.int64), device=self.dev)
        return workloads.to_raw(blocks.index_select(0, idx))

    def close(self):
        self.pool.close()


def oracle_table(cfg):
    return oracle.block_tables(cfg.windows_array(), cfg.batch, cfg.block_size)


def config_with(cfg, **kw):
    return dataclasses.replace(cfg, **kw)
