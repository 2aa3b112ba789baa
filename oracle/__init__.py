"""Oracle for the per-head windowed KV path -- TEST INFRASTRUCTURE ONLY.

Plain, slow CPU restatement of what the pages fix, written from

* "HeadWiseKV: Budgeted Per-Head Cache Residency for Hybrid Long-Context Language
  Models" (blog summary), abstract -- every physical KV head of a global-attention layer
  keeps a static window of its most recent tokens, the footprint is known before serving,
  and the runtime materialises the residency rather than masking a full cache;
* same page, section "Grouped-Cache Runtime" -- a paged block table gives each head
  ceil(window / block_size) blocks;
* same page, section "SeqCalib" -- the layer-by-layer greedy choice of window vectors under
  a memory budget (``seqcalib_greedy``);
* chunked prefill (``prefill_attention``): every new token attends to its own window of the
  full history, exactly as if the chunk had been appended and decoded token by token.

Where the pages are silent the oracle takes these readings:

* ring placement: position p of a head lives in ring slot p mod C, C = nblk * block_size;
* materialise copies only the last min(w, L) prefill positions; unwritten slots hold 0;
* physical block ids are handed out in (layer, sequence, kv head, logical block) order;
* attention at length ``len`` (after the append) covers positions [max(0, len-w), len);
* query head q reads kv head q // (q_heads / kv_heads);
* an empty window (len == 0) gives a zero output.

Only ``tests/``, the smoke check of ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library.

Parity status: every function here is pinned by a ``-m "not gpu"`` test (hand-derived
golden fixtures, closed forms, and torch's own scaled_dot_product_attention on
special cases); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Iterable, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "hwkv_oracle.c")

F32, BF16, F64 = 0, 1, 2
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C part of the oracle with gcc (plain -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Job(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("row_stride", ctypes.c_int64), ("p_lo", ctypes.c_int64), ("n_hist", ctypes.c_int64),
                ("len", ctypes.c_int64), ("window", ctypes.c_int64), ("scale", ctypes.c_double),
                ("out", ctypes.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_attention.argtypes = [ctypes.POINTER(_Job), ctypes.c_int64, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int]
            lib.oracle_attention.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return os.cpu_count() or 1


# ------------------------------------------------------------------------------------
# Pool geometry (section "Grouped-Cache Runtime": ceil(window / block_size) blocks per head)
# ------------------------------------------------------------------------------------
def blocks_per_head(windows, block_size: int) -> np.ndarray:
    """nblk[l][h] = ceil(w[l][h] / block_size)."""
    w = np.asarray(windows, dtype=np.int64)
    return -(-w // block_size)


def ring_capacity(windows, block_size: int) -> np.ndarray:
    """C[l][h] = nblk[l][h] * block_size tokens."""
    return blocks_per_head(windows, block_size) * block_size


def pool_bytes(windows, num_seqs: int, head_dim: int, block_size: int, elem_bytes: int) -> int:
    """Bytes of the whole pool, known before serving (abstract): for every sequence,
    layer and kv head, nblk blocks of block_size K rows and block_size V rows."""
    nblk = blocks_per_head(windows, block_size)
    total = 0
    for s in range(num_seqs):
        for l in range(nblk.shape[0]):
            for h in range(nblk.shape[1]):
                total += int(nblk[l, h]) * block_size * head_dim * 2 * elem_bytes
    return total


def block_tables(windows, num_seqs: int, block_size: int) -> dict:
    """{(layer, seq, kv_head): [physical block id per logical block]} with ids handed
    out consecutively in (layer, seq, kv_head, logical block) order."""
    nblk = blocks_per_head(windows, block_size)
    tables, nxt = {}, 0
    for l in range(nblk.shape[0]):
        for s in range(num_seqs):
            for h in range(nblk.shape[1]):
                n = int(nblk[l, h])
                tables[(l, s, h)] = list(range(nxt, nxt + n))
                nxt += n
    return tables


def total_blocks(windows, num_seqs: int, block_size: int) -> int:
    return int(blocks_per_head(windows, block_size).sum()) * num_seqs


# ------------------------------------------------------------------------------------
# Residency: which positions are written where (materialise + append)
# ------------------------------------------------------------------------------------
def materialized_positions(prefill_len: int, window: int) -> range:
    """Materialise copies the last min(w, L) prefill positions, oldest first."""
    return range(max(0, prefill_len - window), prefill_len)


def appended_positions(prefill_len: int, n_appends: int) -> range:
    """Decode step i appends the token at position prefill_len + i."""
    return range(prefill_len, prefill_len + n_appends)


def ring_after_writes(hist_k: np.ndarray, hist_v: np.ndarray, p_lo: int,
                      writes: Iterable[int], capacity: int):
    """Ring contents [capacity][D] after writing the given positions in order.

    ``hist_k[i]`` is the row of position ``p_lo + i``.  A position's row goes to slot
    ``p mod capacity``; a later write to the same slot replaces the earlier one; slots
    never written hold zero bits.
    """
    D = hist_k.shape[1]
    ring_k = np.zeros((capacity, D), dtype=hist_k.dtype)
    ring_v = np.zeros((capacity, D), dtype=hist_v.dtype)
    for p in writes:
        ring_k[p % capacity] = hist_k[p - p_lo]
        ring_v[p % capacity] = hist_v[p - p_lo]
    return ring_k, ring_v


def ring_to_blocks(ring_k: np.ndarray, ring_v: np.ndarray, block_size: int) -> np.ndarray:
    """Split a ring into physical blocks [nblk][2][block_size][D]: K rows then V rows."""
    C, D = ring_k.shape
    n = C // block_size
    out = np.zeros((n, 2, block_size, D), dtype=ring_k.dtype)
    for j in range(n):
        out[j, 0] = ring_k[j * block_size:(j + 1) * block_size]
        out[j, 1] = ring_v[j * block_size:(j + 1) * block_size]
    return out


def expected_pool(windows, num_seqs: int, block_size: int, head_dim: int, raw_dtype,
                  history_fn, prefill_lens: Sequence[int], n_appends: int) -> np.ndarray:
    """Whole expected pool [total_blocks][2][block_size][D] after materialising every
    layer's prefill and then appending ``n_appends`` tokens.

    ``history_fn(layer, seq, head, p_lo, p_hi) -> (K rows, V rows)``.
    """
    cap = ring_capacity(windows, block_size)
    tables = block_tables(windows, num_seqs, block_size)
    pool = np.zeros((total_blocks(windows, num_seqs, block_size), 2, block_size, head_dim), dtype=raw_dtype)
    w = np.asarray(windows)
    for (l, s, h), ids in tables.items():
        L = int(prefill_lens[s])
        writes = list(materialized_positions(L, int(w[l, h]))) + list(appended_positions(L, n_appends))
        if writes:
            p_lo = writes[0]
            hk, hv = history_fn(l, s, h, p_lo, L + n_appends)
        else:
            p_lo, hk, hv = 0, np.zeros((0, head_dim), raw_dtype), np.zeros((0, head_dim), raw_dtype)
        rk, rv = ring_after_writes(hk, hv, p_lo, writes, int(cap[l, h]))
        blocks = ring_to_blocks(rk, rv, block_size)
        for j, b in enumerate(ids):
            pool[b] = blocks[j]
    return pool


# ------------------------------------------------------------------------------------
# Attention (abstract + "Grouped-Cache Runtime": materialised window == masked full cache)
# ------------------------------------------------------------------------------------
def window_span(length: int, window: int):
    """Positions [lo, hi) that attention covers at sequence length ``length``."""
    return max(0, length - window), length


def _raw_code(arr: np.ndarray) -> int:
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    if arr.dtype == np.float64:
        return F64
    raise TypeError(arr.dtype)


def attention_jobs(q: np.ndarray, hist: dict, lens, windows_l, scale: float, threads=None) -> np.ndarray:
    """fp64 decode attention of one layer, GQA by consecutive groups.

    q       : [B][Hq][D] raw host array (float32, uint16 bf16 bits, or float64)
    hist    : {(seq, kv_head): (p_lo, K rows, V rows)} covering each head's window
    lens    : [B] sequence lengths after the append
    windows_l: [Hkv] windows of this layer
    returns : [B][Hq][D] float64
    """
    B, Hq, D = q.shape
    Hkv = len(windows_l)
    G = Hq // Hkv
    code = _raw_code(q)
    q = np.ascontiguousarray(q)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    keep = []
    jobs = (_Job * (B * Hq))()
    i = 0
    for s in range(B):
        for qh in range(Hq):
            h = qh // G
            p_lo, hk, hv = hist[(s, h)]
            hk = np.ascontiguousarray(hk)
            hv = np.ascontiguousarray(hv)
            if _raw_code(hk) != code or _raw_code(hv) != code:
                raise TypeError("q, K and V must share one raw dtype")
            keep += [hk, hv]
            jobs[i].q = q[s, qh].ctypes.data
            jobs[i].k = hk.ctypes.data
            jobs[i].v = hv.ctypes.data
            jobs[i].row_stride = D
            jobs[i].p_lo = int(p_lo)
            jobs[i].n_hist = int(hk.shape[0])
            jobs[i].len = int(lens[s])
            jobs[i].window = int(windows_l[h])
            jobs[i].scale = float(scale)
            jobs[i].out = out[s, qh].ctypes.data
            i += 1
    rc = _load().oracle_attention(jobs, B * Hq, D, code, int(threads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_attention failed ({rc}): history does not cover a window")
    return out


def attention_one(q_vec: np.ndarray, hist_k: np.ndarray, hist_v: np.ndarray, p_lo: int,
                  length: int, window: int, scale: float) -> np.ndarray:
    """fp64 attention of one query vector against one head's history."""
    D = q_vec.shape[-1]
    out = attention_jobs(np.asarray(q_vec).reshape(1, 1, D), {(0, 0): (p_lo, hist_k, hist_v)},
                         [length], [window], scale, threads=1)
    return out[0, 0]


def widen(raw: np.ndarray) -> np.ndarray:
    """Exact fp64 value of a raw host array (float32, or uint16 bf16 bit patterns)."""
    if raw.dtype == np.uint16:
        return (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return raw.astype(np.float64)



# ------------------------------------------------------------------------------------
# SeqCalib (section "SeqCalib"): greedy, layer by layer in execution order
# ------------------------------------------------------------------------------------
def layer_cost(window_vector, num_seqs: int, head_dim: int, block_size: int, elem_bytes: int) -> int:
    """R_i(w_i): bytes one layer's window vector occupies in the pool."""
    return pool_bytes([list(window_vector)], num_seqs, head_dim, block_size, elem_bytes)


def seqcalib_greedy(candidates, distortion_fn, budget: int, cost_fn):
    """Walks the layers in order; for each, among its candidate window vectors, keeps the one
    of smallest distortion (first one on ties) whose cost fits what is left of the budget,
    then charges its cost.  ``distortion_fn(layer, w, chosen_so_far)`` may depend on the
    vectors chosen for the earlier layers; ``cost_fn(layer, w)`` is the layer's memory.
    Returns (chosen vectors, chosen indices, total cost).  Raises ValueError when no candidate
    of a layer fits (the page's pseudocode would carry ``None`` on)."""
    policies, picks, remaining, total = [], [], budget, 0
    for layer, feasible in enumerate(candidates):
        best_w, best_i, min_distort = None, None, float("inf")
        for i, w in enumerate(feasible):
            d = distortion_fn(layer, list(w), [list(p) for p in policies])
            c = cost_fn(layer, list(w))
            if c <= remaining and d < min_distort:
                best_w, best_i, min_distort = list(w), i, d
        if best_w is None:
            raise ValueError(f"no candidate of layer {layer} fits the remaining budget {remaining}")
        policies.append(best_w)
        picks.append(best_i)
        cost = cost_fn(layer, best_w)
        remaining -= cost
        total += cost
    return policies, picks, total


# ------------------------------------------------------------------------------------
# Chunked prefill: token p0 + i attends to [max(0, p0 + i + 1 - w), p0 + i + 1)
# ------------------------------------------------------------------------------------
def prefill_attention(q: np.ndarray, hist: dict, p0: int, windows_l, scale: float, threads=None) -> np.ndarray:
    """fp64 windowed causal attention of a chunk of one sequence.

    q    : [n][Hq][D] raw host array, token i at position p0 + i
    hist : {kv_head: (p_lo, K rows, V rows)} covering every position the chunk's windows need
    returns [n][Hq][D] float64
    """
    n = q.shape[0]
    out = np.zeros(q.shape, dtype=np.float64)
    for i in range(n):
        per_tok = {(0, h): v for h, v in hist.items()}
        out[i] = attention_jobs(q[i][None], per_tok, [p0 + i + 1], windows_l, scale, threads=threads)[0]
    return out
