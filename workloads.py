"""Seeded synthetic inputs for the per-head windowed decode path.

This module is the only code that the CPU oracle (``oracle/``) and the CUDA path
(``head_budgeted_kv_gb300``) both consume.  It holds configuration constants and
random draws and nothing else: no slot mapping, no block counts, no attention.

The five workloads follow the shapes the HeadWiseKV blog summary
("HeadWiseKV: budgeted per-head cache residency for hybrid long-context models",
abstract and section "Grouped-Cache Runtime") gives for its serving experiments:

* ``tiny``     fp32, 1 layer, 2 KV heads, GQA 2, D 64, windows [32, 128], 256-token
               prefill, 8 decode steps; one CPU generator seeded 0.
* ``layer``    bf16, 1 layer, 8 KV heads, GQA 4, D 128, windows drawn from the
               level set {1024, 4096, 16384, 65536}, batch 8, 32768-token prefill,
               1 decode step.
* ``full``     bf16, 48 global layers, windows from the example policy YAML of the
               "Grouped-Cache Runtime" section (layer 0 / layer 1 rows repeated by
               layer parity), batch 4, 112K (114 688) prefill, 128 decode steps.
* ``ragged``   bf16, 64 sequences with prefill lengths uniform in [1K, 160K],
               16 layers, block size 64, windows from the level set (some larger
               than the context), 1% of keys scaled by 8, 32 decode steps.
* ``long``     bf16, batch 1, 161K (164 864) prefill, 48 layers, windows from the
               level set, 256 decode steps; ``long_full`` sets every window to the
               final context (full attention through the same path).

"K" is read as 1024 (112K = 114 688, 161K = 164 864, 160K = 163 840).

Every tensor is N(0, 1) drawn by torch's generator from a seed that depends only
on (workload, purpose, layer, sequence or step).  bf16 tensors are drawn in fp32
and rounded to bf16 with round-to-nearest-even.  Large workloads are drawn on the
GPU (torch's Philox generator); the oracle is handed host copies of exactly those
bytes.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

LEVELS = (1024, 4096, 16384, 65536)
# Example policy rows printed in the "Grouped-Cache Runtime" section (layer 0, layer 1).
POLICY_LAYER0 = (4096, 4096, 16384, 16384, 65536, 65536, 65536, 65536)
POLICY_LAYER1 = (1024, 4096, 4096, 16384, 16384, 65536, 65536, 65536)

# purposes folded into the seeds
_P_PREFILL_K, _P_PREFILL_V, _P_Q, _P_KNEW, _P_VNEW, _P_SPIKE_PRE, _P_SPIKE_NEW = range(1, 8)
_P_CHUNK_Q, _P_CHUNK_K, _P_CHUNK_V = 8, 9, 10


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    cfg_id: int
    layers: int
    kv_heads: int
    q_heads: int
    head_dim: int
    block_size: int
    dtype: str                 # "f32" or "bf16"
    batch: int
    steps: int
    windows: tuple             # [layers][kv_heads] ints
    prefill: tuple             # [batch] ints
    spike_frac: float = 0.0    # fraction of keys scaled by spike_mult
    spike_mult: float = 8.0
    single_cpu_stream: bool = False   # all draws from one CPU generator (tiny case)

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def max_prefill(self) -> int:
        return max(self.prefill)

    def windows_array(self) -> np.ndarray:
        return np.asarray(self.windows, dtype=np.int32).reshape(self.layers, self.kv_heads)

    def prefill_array(self) -> np.ndarray:
        return np.asarray(self.prefill, dtype=np.int32)

    def with_layers(self, layers: int, name: Optional[str] = None) -> "Config":
        """Same per-layer shape, fewer layers (the first ``layers`` rows of the policy)."""
        return dataclasses.replace(self, name=name or f"{self.name}_{layers}l", layers=layers,
                                   windows=tuple(self.windows[:layers]))

    def with_steps(self, steps: int) -> "Config":
        return dataclasses.replace(self, steps=steps)


def _level_windows(seed: int, layers: int, heads: int) -> tuple:
    rng = np.random.default_rng(seed)
    w = rng.choice(np.asarray(LEVELS), size=(layers, heads))
    return tuple(tuple(int(x) for x in row) for row in w)


def _make(name: str) -> Config:
    if name == "tiny":
        return Config("tiny", 1, layers=1, kv_heads=2, q_heads=4, head_dim=64, block_size=16,
                      dtype="f32", batch=1, steps=8, windows=((32, 128),), prefill=(256,),
                      single_cpu_stream=True)
    if name == "layer":
        return Config("layer", 2, layers=1, kv_heads=8, q_heads=32, head_dim=128, block_size=16,
                      dtype="bf16", batch=8, steps=1, windows=_level_windows(2001, 1, 8),
                      prefill=(32768,) * 8)
    if name == "full":
        rows = tuple(POLICY_LAYER0 if l % 2 == 0 else POLICY_LAYER1 for l in range(48))
        return Config("full", 3, layers=48, kv_heads=8, q_heads=32, head_dim=128, block_size=16,
                      dtype="bf16", batch=4, steps=128, windows=rows, prefill=(114688,) * 4)
    if name == "ragged":
        rng = np.random.default_rng(4002)
        lens = tuple(int(x) for x in rng.integers(1024, 163840, size=64, endpoint=True))
        return Config("ragged", 4, layers=16, kv_heads=8, q_heads=32, head_dim=128, block_size=64,
                      dtype="bf16", batch=64, steps=32, windows=_level_windows(4001, 16, 8),
                      prefill=lens, spike_frac=0.01)
    if name == "long":
        return Config("long", 5, layers=48, kv_heads=8, q_heads=32, head_dim=128, block_size=16,
                      dtype="bf16", batch=1, steps=256, windows=_level_windows(5001, 48, 8),
                      prefill=(164864,))
    if name == "long_full":
        w = 164864 + 256
        return Config("long_full", 6, layers=48, kv_heads=8, q_heads=32, head_dim=128,
                      block_size=16, dtype="bf16", batch=1, steps=256,
                      windows=tuple((w,) * 8 for _ in range(48)), prefill=(164864,))
    raise KeyError(name)


NAMES = ("tiny", "layer", "full", "ragged", "long", "long_full")


def config(name: str) -> Config:
    return _make(name)


def _seed(cfg: Config, purpose: int, a: int, b: int) -> int:
    return ((cfg.cfg_id * 16 + purpose) * 1024 + a) * 1_000_003 + b


def _randn(shape, seed: int, device, dtype) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return x.to(dtype)


def _spike(x32: torch.Tensor, seed: int, frac: float, mult: float) -> torch.Tensor:
    """Scale whole key rows (last dim) by ``mult`` with probability ``frac``."""
    g = torch.Generator(device=x32.device)
    g.manual_seed(seed)
    sel = torch.rand(x32.shape[:-1], generator=g, device=x32.device) < frac
    return torch.where(sel.unsqueeze(-1), x32 * mult, x32)


class Workload:
    """Deterministic inputs of one configuration.

    ``device`` is where large tensors are drawn (``"cuda"`` for the big workloads).
    The tiny fp32 case always draws on the CPU from one generator seeded 0 in the
    order: prefill K, prefill V, then per step (q, k_new, v_new).
    """

    def __init__(self, cfg: Config, device="cpu"):
        self.cfg = cfg
        self.device = torch.device(device)
        self._tiny = None
        if cfg.single_cpu_stream:
            g = torch.Generator(device="cpu")
            g.manual_seed(0)
            B, H, Hq, D, L = cfg.batch, cfg.kv_heads, cfg.q_heads, cfg.head_dim, cfg.max_prefill
            dt = cfg.torch_dtype
            kp = torch.randn((cfg.layers, B, H, L, D), generator=g).to(dt)
            vp = torch.randn((cfg.layers, B, H, L, D), generator=g).to(dt)
            steps = []
            for _ in range(cfg.steps):
                q = torch.randn((cfg.layers, B, Hq, D), generator=g).to(dt)
                kn = torch.randn((cfg.layers, B, H, D), generator=g).to(dt)
                vn = torch.randn((cfg.layers, B, H, D), generator=g).to(dt)
                steps.append((q, kn, vn))
            self._tiny = (kp, vp, steps)

    # ---- shapes -------------------------------------------------------------------
    def windows(self) -> np.ndarray:
        return self.cfg.windows_array()

    def prefill_lens(self) -> np.ndarray:
        return self.cfg.prefill_array()

    def lens_before_step(self, step: int) -> np.ndarray:
        """Sequence lengths before the append of decode step ``step``."""
        return (self.cfg.prefill_array().astype(np.int64) + step).astype(np.int32)

    # ---- prefill ------------------------------------------------------------------
    def prefill_seq(self, layer: int, s: int, device=None):
        """Prefill K, V of one sequence: [kv_heads][prefill_s][head_dim]."""
        cfg = self.cfg
        dev = torch.device(device) if device is not None else self.device
        if self._tiny is not None:
            kp, vp, _ = self._tiny
            L = cfg.prefill[s]
            return kp[layer, s, :, :L].to(dev), vp[layer, s, :, :L].to(dev)
        shape = (cfg.kv_heads, cfg.prefill[s], cfg.head_dim)
        k32 = _randn(shape, _seed(cfg, _P_PREFILL_K, layer, s), self.device, torch.float32)
        if cfg.spike_frac > 0:
            k32 = _spike(k32, _seed(cfg, _P_SPIKE_PRE, layer, s), cfg.spike_frac, cfg.spike_mult)
        k = k32.to(cfg.torch_dtype)
        del k32
        v = _randn(shape, _seed(cfg, _P_PREFILL_V, layer, s), self.device, cfg.torch_dtype)
        return k.to(dev), v.to(dev)

    def prefill_layer(self, layer: int, device=None, max_len: Optional[int] = None):
        """Contiguous full prefill K, V of one layer: [batch][kv_heads][max_len][head_dim].

        Rows at or past a sequence's prefill length are zero.
        """
        cfg = self.cfg
        dev = torch.device(device) if device is not None else self.device
        Lm = max_len or cfg.max_prefill
        K = torch.zeros((cfg.batch, cfg.kv_heads, Lm, cfg.head_dim), dtype=cfg.torch_dtype, device=dev)
        V = torch.zeros_like(K)
        for s in range(cfg.batch):
            k, v = self.prefill_seq(layer, s, dev)
            K[s, :, : k.shape[1]] = k
            V[s, :, : v.shape[1]] = v
            del k, v
        return K, V

    # ---- decode steps --------------------------------------------------------------
    def step_inputs(self, step: int, device=None):
        """(q [layers][B][Hq][D], k_new [layers][B][Hkv][D], v_new [layers][B][Hkv][D])."""
        cfg = self.cfg
        dev = torch.device(device) if device is not None else self.device
        if self._tiny is not None:
            q, kn, vn = self._tiny[2][step]
            return q.to(dev), kn.to(dev), vn.to(dev)
        L, B, H, Hq, D = cfg.layers, cfg.batch, cfg.kv_heads, cfg.q_heads, cfg.head_dim
        q = _randn((L, B, Hq, D), _seed(cfg, _P_Q, 0, step), self.device, cfg.torch_dtype)
        k32 = _randn((L, B, H, D), _seed(cfg, _P_KNEW, 0, step), self.device, torch.float32)
        if cfg.spike_frac > 0:
            k32 = _spike(k32, _seed(cfg, _P_SPIKE_NEW, 0, step), cfg.spike_frac, cfg.spike_mult)
        kn = k32.to(cfg.torch_dtype)
        vn = _randn((L, B, H, D), _seed(cfg, _P_VNEW, 0, step), self.device, cfg.torch_dtype)
        return q.to(dev), kn.to(dev), vn.to(dev)

    # ---- chunked prefill ----------------------------------------------------------
    def chunk_inputs(self, layer: int, chunk: int, n_max: int, device=None):
        """A prefill chunk of n_max token rows per sequence: (q [B][n_max][Hq][D],
        k [B][n_max][Hkv][D], v [B][n_max][Hkv][D]), N(0, 1)."""
        cfg = self.cfg
        dev = torch.device(device) if device is not None else self.device
        B, H, Hq, D = cfg.batch, cfg.kv_heads, cfg.q_heads, cfg.head_dim
        q = _randn((B, n_max, Hq, D), _seed(cfg, _P_CHUNK_Q, layer, chunk), self.device, cfg.torch_dtype)
        k = _randn((B, n_max, H, D), _seed(cfg, _P_CHUNK_K, layer, chunk), self.device, cfg.torch_dtype)
        v = _randn((B, n_max, H, D), _seed(cfg, _P_CHUNK_V, layer, chunk), self.device, cfg.torch_dtype)
        return q.to(dev), k.to(dev), v.to(dev)

    # ---- host copies for the oracle ------------------------------------------------
    def history(self, layer: int, s: int, h: int, p_lo: int, p_hi: int, prefill=None, steps=None):
        """Host rows of K and V for positions [p_lo, p_hi) of (layer, seq, kv head).

        Positions below the prefill length come from the prefill, the rest from the
        appended tokens of the decode steps (position prefill + i is step i).
        ``prefill`` may pass an already drawn ``prefill_seq(layer, s)`` pair and
        ``steps`` a list of already drawn ``step_inputs`` tuples.
        Returns raw host arrays: float32 for fp32 workloads, uint16 bit patterns for bf16.
        """
        cfg = self.cfg
        L = cfg.prefill[s]
        ks, vs = [], []
        if p_lo < L:
            if prefill is None:
                prefill = self.prefill_seq(layer, s)
            kp, vp = prefill
            ks.append(kp[h, p_lo:min(p_hi, L)])
            vs.append(vp[h, p_lo:min(p_hi, L)])
        for p in range(max(p_lo, L), p_hi):
            st = p - L
            _, kn, vn = steps[st] if steps is not None else self.step_inputs(st)
            ks.append(kn[layer, s, h][None])
            vs.append(vn[layer, s, h][None])
        K = torch.cat([k.to("cpu") for k in ks]) if ks else torch.zeros((0, cfg.head_dim), dtype=cfg.torch_dtype)
        V = torch.cat([v.to("cpu") for v in vs]) if vs else torch.zeros((0, cfg.head_dim), dtype=cfg.torch_dtype)
        return to_raw(K), to_raw(V)


def to_raw(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of a tensor's bits: float32 stays float32, bf16 becomes uint16."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)
