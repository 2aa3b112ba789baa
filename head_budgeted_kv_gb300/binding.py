"""Thin ctypes binding of the hwkv C ABI (``include/hwkv.h``).

Argument marshalling only: torch tensors become device pointers, torch streams become
``cudaStream_t``.  Every step of the path runs in libhwkv.so; when the library is missing
this module raises instead of computing anything itself.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

from . import _build

HWKV_OK = 0
HWKV_ERR_INVALID_ARG = -1
HWKV_ERR_ALIGNMENT = -2
HWKV_ERR_POOL_TOO_SMALL = -3
HWKV_ERR_CUDA = -4
HWKV_ERR_DEVICE_CHECK = -5
HWKV_ERR_UNSUPPORTED = -6
HWKV_ERR_WORKSPACE_TOO_SMALL = -7
HWKV_ERR_BUDGET = -8

DISTORTION_FN = ctypes.CFUNCTYPE(ctypes.c_double, ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
                                 ctypes.POINTER(ctypes.c_int32))

HWKV_F32 = 0
HWKV_BF16 = 1
HWKV_KERNEL_AUTO, HWKV_KERNEL_TENSOR, HWKV_KERNEL_SIMT = 0, 1, 2
HWKV_DEVERR_NEG_LENGTH, HWKV_DEVERR_BAD_BLOCK, HWKV_DEVERR_SRC_RANGE, HWKV_DEVERR_WAIT_TIMEOUT = 1, 2, 4, 8
HWKV_DECODE_EARLY_READS = 1

_c_i32p = ctypes.POINTER(ctypes.c_int32)
_c_u64p = ctypes.POINTER(ctypes.c_uint64)
_c_i64p = ctypes.POINTER(ctypes.c_int64)
_vp = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64

# (name, restype, argtypes) for every function declared in include/hwkv.h
SIGNATURES = [
    ("hwkv_abi_version", _i, []),
    ("hwkv_last_error", ctypes.c_char_p, []),
    ("hwkv_status_string", ctypes.c_char_p, [_i]),
    ("hwkv_pool_bytes", _i, [_i, _i, _i, _i, _c_i32p, _i, _i, _c_u64p]),
    ("hwkv_pool_create", _i, [_i, _i, _i, _i, _c_i32p, _i, _i, _vp, _u64, _vp, ctypes.POINTER(_vp)]),
    ("hwkv_pool_destroy", _i, [_vp]),
    ("hwkv_pool_geometry", _i, [_vp, _c_u64p, _c_i64p, _c_i64p]),
    ("hwkv_block_table", _i, [_vp, _i, _i, _i, _c_i32p, _i, ctypes.POINTER(_i)]),
    ("hwkv_set_block_table", _i, [_vp, _c_i32p, _i64, _vp]),
    ("hwkv_materialize", _i, [_vp, _i, _vp, _vp, _i64, _i64, _i64, _vp, _vp]),
    ("hwkv_append", _i, [_vp, _i, _vp, _vp, _vp, _vp]),
    ("hwkv_advance_positions", _i, [_vp, _vp, _vp, ctypes.c_int32, _vp]),
    ("hwkv_wait_selftest", _i, [ctypes.c_uint32, _vp, _vp]),
    ("hwkv_decode_workspace_bytes", _i, [_vp, _i, _c_u64p]),
    ("hwkv_decode_attn", _i, [_vp, _i, _vp, _i, ctypes.c_float, _vp, _vp, _vp, _u64, _vp]),
    ("hwkv_append_decode_attn", _i, [_vp, _i, _vp, _i, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _u64, _vp]),
    ("hwkv_decode_attn_ex", _i, [_vp, _i, _vp, _i, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _u64, _i, _vp]),
    ("hwkv_decode_attn_noalloc", _i, [_vp, _i, _vp, _i, ctypes.c_float, _vp, _vp, _vp]),
    ("hwkv_prefill_attn", _i, [_vp, _i, _vp, _i, ctypes.c_float, _vp, _vp, _i, _vp, _vp, _vp, _vp, _u64, _vp]),
    ("hwkv_prefill_workspace_bytes", _i, [_vp, _i, _i, _i, ctypes.POINTER(_u64)]),
    ("hwkv_prefill_plan", _i, [_i, _i, _i, _i, _c_i32p, _i, _i, _i, _i, _i, _i, _c_i32p, _c_i32p, _c_i32p, _c_u64p]),
    ("hwkv_set_prefill_config", _i, [_vp, _i]),
    ("hwkv_set_decode_config", _i, [_vp, _i, _i, _i]),
    ("hwkv_kernel_launches", _i, [_c_u64p]),
    ("hwkv_seqcalib", _i, [_i, _i, _i, _i, _i, _i, _i, _c_i32p, DISTORTION_FN, _vp, _u64, _c_i32p, _c_i32p, _c_u64p]),
    ("hwkv_check_device_errors", _i, [_vp, _vp, _c_i32p]),
]

_lib = None


class HwkvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{status_string(status)} ({status}): {msg}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libhwkv.so (building it with nvcc first when it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libhwkv.so not built ({path}); run __graft_entry__.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.hwkv_abi_version() != 3:
        raise RuntimeError("libhwkv.so ABI version mismatch")
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().hwkv_status_string(status).decode()


def last_error() -> str:
    return load().hwkv_last_error().decode()


def _check(status: int):
    if status != HWKV_OK:
        raise HwkvError(status, last_error())


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        return int(t)
    return t.data_ptr()


def _dtype_code(dtype) -> int:
    if dtype in (HWKV_F32, HWKV_BF16):
        return int(dtype)
    if dtype in (torch.float32, "f32", "float32"):
        return HWKV_F32
    if dtype in (torch.bfloat16, "bf16", "bfloat16"):
        return HWKV_BF16
    raise ValueError(f"unsupported dtype {dtype}")


def _windows(windows) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(windows, dtype=np.int32))


# ------------------------------------------------------------------------------------
# functions with the ABI's names
# ------------------------------------------------------------------------------------
def hwkv_abi_version() -> int:
    return load().hwkv_abi_version()


def hwkv_pool_bytes(layers, kv_heads, head_dim, block_size, windows, num_seqs, dtype) -> int:
    w = _windows(windows)
    out = ctypes.c_uint64(0)
    _check(load().hwkv_pool_bytes(layers, kv_heads, head_dim, block_size, w.ctypes.data_as(_c_i32p), num_seqs,
                                  _dtype_code(dtype), ctypes.byref(out)))
    return out.value


def hwkv_pool_create(layers, kv_heads, head_dim, block_size, windows, num_seqs, dtype, dev_pool: torch.Tensor,
                     stream=None) -> int:
    w = _windows(windows)
    handle = ctypes.c_void_p(0)
    nbytes = dev_pool.numel() * dev_pool.element_size()
    _check(load().hwkv_pool_create(layers, kv_heads, head_dim, block_size, w.ctypes.data_as(_c_i32p), num_seqs,
                                   _dtype_code(dtype), _ptr(dev_pool), nbytes, _stream_ptr(stream),
                                   ctypes.byref(handle)))
    return handle.value


def hwkv_pool_destroy(pool: int):
    _check(load().hwkv_pool_destroy(pool))


def hwkv_pool_geometry(pool: int):
    b, n, bb = ctypes.c_uint64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    _check(load().hwkv_pool_geometry(pool, ctypes.byref(b), ctypes.byref(n), ctypes.byref(bb)))
    return b.value, n.value, bb.value


def hwkv_block_table(pool: int, seq: int, layer: int, kv_head: int) -> np.ndarray:
    n = ctypes.c_int(0)
    _check(load().hwkv_block_table(pool, seq, layer, kv_head, None, 0, ctypes.byref(n)))
    out = np.zeros(n.value, dtype=np.int32)
    _check(load().hwkv_block_table(pool, seq, layer, kv_head, out.ctypes.data_as(_c_i32p), n.value, ctypes.byref(n)))
    return out


def hwkv_set_block_table(pool: int, table, stream=None):
    t = np.ascontiguousarray(np.asarray(table, dtype=np.int32))
    _check(load().hwkv_set_block_table(pool, t.ctypes.data_as(_c_i32p), t.size, _stream_ptr(stream)))


def hwkv_materialize(pool: int, layer: int, k_full: torch.Tensor, v_full: torch.Tensor, lens: torch.Tensor,
                     stream=None):
    """k_full, v_full: [B][H][max_len][D] with contiguous rows; lens: int32 [B] on the device."""
    if k_full.stride() != v_full.stride() or k_full.shape != v_full.shape:
        raise ValueError("k_full and v_full must share shape and strides")
    if k_full.stride(3) != 1 or k_full.stride(2) != k_full.shape[3]:
        raise ValueError("rows of k_full must be contiguous")
    _check(load().hwkv_materialize(pool, layer, _ptr(k_full), _ptr(v_full), k_full.stride(0), k_full.stride(1),
                                   k_full.shape[2], _ptr(lens), _stream_ptr(stream)))


def hwkv_append(pool: int, layer: int, k_new: torch.Tensor, v_new: torch.Tensor, pos: torch.Tensor, stream=None):
    """k_new, v_new: contiguous [B][H][D]; pos: int32 [B] lengths before the append."""
    if not (k_new.is_contiguous() and v_new.is_contiguous()):
        raise ValueError("k_new and v_new must be contiguous")
    _check(load().hwkv_append(pool, layer, _ptr(k_new), _ptr(v_new), _ptr(pos), _stream_ptr(stream)))


def hwkv_wait_selftest(limit_us: int, out: torch.Tensor, stream=None):
    """Runs the library's bounded wait on a completed and on a never-completing mbarrier phase;
    out: int32 [3] on the device (error bits, first wait succeeded, microseconds waited)."""
    _check(load().hwkv_wait_selftest(int(limit_us), _ptr(out), _stream_ptr(stream)))


def hwkv_advance_positions(pool: int, pos: torch.Tensor, out: torch.Tensor, delta: int = 1, stream=None):
    """out[s] = pos[s] + delta on the device (int32 [num_seqs]; out may be pos)."""
    if pos.dtype != torch.int32 or out.dtype != torch.int32:
        raise ValueError("positions must be int32")
    _check(load().hwkv_advance_positions(pool, _ptr(pos), _ptr(out), int(delta), _stream_ptr(stream)))


def hwkv_decode_workspace_bytes(pool: int, q_heads: int) -> int:
    out = ctypes.c_uint64(0)
    _check(load().hwkv_decode_workspace_bytes(pool, q_heads, ctypes.byref(out)))
    return out.value


def hwkv_decode_attn(pool: int, layer: int, q: torch.Tensor, scale: float, lens: torch.Tensor, out: torch.Tensor,
                     workspace: Optional[torch.Tensor], stream=None, early_reads: bool = False):
    """q, out: contiguous [B][Hq][D]; lens: int32 [B] lengths after the append.  early_reads sets
    HWKV_DECODE_EARLY_READS (see the header for the caller's guarantee)."""
    if not (q.is_contiguous() and out.is_contiguous()):
        raise ValueError("q and out must be contiguous")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if early_reads:
        _check(load().hwkv_decode_attn_ex(pool, layer, _ptr(q), q.shape[1], float(scale), None, None, _ptr(lens),
                                          _ptr(out), _ptr(workspace), ws_bytes, HWKV_DECODE_EARLY_READS,
                                          _stream_ptr(stream)))
        return
    _check(load().hwkv_decode_attn(pool, layer, _ptr(q), q.shape[1], float(scale), _ptr(lens), _ptr(out),
                                   _ptr(workspace), ws_bytes, _stream_ptr(stream)))


def hwkv_append_decode_attn(pool: int, layer: int, q: torch.Tensor, scale: float, k_new: torch.Tensor,
                            v_new: torch.Tensor, pos: torch.Tensor, out: torch.Tensor,
                            workspace: Optional[torch.Tensor], stream=None, early_reads: bool = False):
    """Append (k_new, v_new at positions pos) then decode at pos + 1, in one call.  early_reads
    sets HWKV_DECODE_EARLY_READS (see the header for the caller's guarantee)."""
    if not (q.is_contiguous() and out.is_contiguous() and k_new.is_contiguous() and v_new.is_contiguous()):
        raise ValueError("q, out, k_new and v_new must be contiguous")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if early_reads:
        _check(load().hwkv_decode_attn_ex(pool, layer, _ptr(q), q.shape[1], float(scale), _ptr(k_new), _ptr(v_new),
                                          _ptr(pos), _ptr(out), _ptr(workspace), ws_bytes, HWKV_DECODE_EARLY_READS,
                                          _stream_ptr(stream)))
        return
    _check(load().hwkv_append_decode_attn(pool, layer, _ptr(q), q.shape[1], float(scale), _ptr(k_new), _ptr(v_new),
                                          _ptr(pos), _ptr(out), _ptr(workspace), ws_bytes, _stream_ptr(stream)))


class DecodeLaunch:
    """One hwkv_decode_attn_ex launch whose arguments are checked and marshalled once; each call
    issues the launch again with the same buffers (a serving loop's static q / k_new / v_new /
    positions / output, or inputs prepared ahead of a timed loop).  k_new and v_new None: decode
    at lengths `lens` (after the append); given: append at positions `lens`, then decode.  The
    tensors are kept alive by the object.  Each call costs about one ctypes call plus the launch,
    against ~17 us for the checks, pointer reads and current-stream lookup of a plain call."""

    def __init__(self, pool: int, layer: int, q: torch.Tensor, scale: float, lens: torch.Tensor, out: torch.Tensor,
                 workspace: Optional[torch.Tensor], k_new: Optional[torch.Tensor] = None,
                 v_new: Optional[torch.Tensor] = None, stream=None, early_reads: bool = False):
        tensors = [t for t in (q, out, k_new, v_new) if t is not None]
        if not all(t.is_contiguous() for t in tensors):
            raise ValueError("q, out, k_new and v_new must be contiguous")
        if (k_new is None) != (v_new is None):
            raise ValueError("k_new and v_new go together")
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        self._keep = (q, lens, out, workspace, k_new, v_new)
        self._fn = load().hwkv_decode_attn_ex
        self._args = (pool, layer, _ptr(q), q.shape[1], float(scale), _ptr(k_new), _ptr(v_new), _ptr(lens), _ptr(out),
                      _ptr(workspace), ws_bytes, HWKV_DECODE_EARLY_READS if early_reads else 0, _stream_ptr(stream))

    def __call__(self):
        status = self._fn(*self._args)
        if status != HWKV_OK:
            raise HwkvError(status, last_error())


def hwkv_decode_attn_noalloc(pool: int, layer: int, q: torch.Tensor, scale: float, lens: torch.Tensor,
                             out: torch.Tensor, stream=None):
    """hwkv_decode_attn with the library's static scratch instead of a caller workspace."""
    if not (q.is_contiguous() and out.is_contiguous()):
        raise ValueError("q and out must be contiguous")
    _check(load().hwkv_decode_attn_noalloc(pool, layer, _ptr(q), q.shape[1], float(scale), _ptr(lens), _ptr(out),
                                           _stream_ptr(stream)))


def hwkv_prefill_attn(pool: int, layer: int, q: torch.Tensor, scale: float, k_new: torch.Tensor, v_new: torch.Tensor,
                      pos: torch.Tensor, n: torch.Tensor, out: torch.Tensor, workspace=None, stream=None):
    """q, out: [B][n_max][Hq][D]; k_new, v_new: [B][n_max][Hkv][D]; pos, n: int32 [B] on the device;
    workspace: optional device tensor of hwkv_prefill_workspace_bytes() bytes."""
    for t in (q, k_new, v_new, out):
        if not t.is_contiguous():
            raise ValueError("prefill tensors must be contiguous")
    ws, ws_bytes = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel() * workspace.element_size())
    _check(load().hwkv_prefill_attn(pool, layer, _ptr(q), q.shape[2], float(scale), _ptr(k_new), _ptr(v_new),
                                    q.shape[1], _ptr(pos), _ptr(n), _ptr(out), ws, ws_bytes, _stream_ptr(stream)))


def hwkv_prefill_workspace_bytes(pool: int, layer: int, q_heads: int, n_max: int) -> int:
    out = _u64(0)
    _check(load().hwkv_prefill_workspace_bytes(pool, layer, q_heads, n_max, ctypes.byref(out)))
    return out.value


def hwkv_prefill_plan(layers: int, kv_heads: int, head_dim: int, block_size: int, windows, num_seqs: int, layer: int,
                      q_heads: int, n_max: int, num_sms: int, max_stages: int = 0):
    """Host-only launch plan of hwkv_prefill_attn: (head_order, splits, split_stages) by launch
    position (int32 arrays of kv_heads entries) and the workspace bytes."""
    w = _windows(windows)
    order = np.zeros(kv_heads, dtype=np.int32)
    splits = np.zeros(kv_heads, dtype=np.int32)
    stages = np.zeros(kv_heads, dtype=np.int32)
    ws = _u64(0)
    _check(load().hwkv_prefill_plan(layers, kv_heads, head_dim, block_size, w.ctypes.data_as(_c_i32p), num_seqs, layer,
                                    q_heads, n_max, num_sms, max_stages, order.ctypes.data_as(_c_i32p),
                                    splits.ctypes.data_as(_c_i32p), stages.ctypes.data_as(_c_i32p), ctypes.byref(ws)))
    return order, splits, stages, ws.value


def hwkv_set_prefill_config(pool: int, max_stages: int = 0):
    _check(load().hwkv_set_prefill_config(pool, max_stages))


def hwkv_set_decode_config(pool: int, split_tokens: int = 0, workers: int = 0, kernel: int = HWKV_KERNEL_AUTO):
    _check(load().hwkv_set_decode_config(pool, split_tokens, workers, kernel))


def hwkv_seqcalib(candidates, distortion, budget_bytes: int, head_dim: int, block_size: int, num_seqs: int,
                  dtype):
    """SeqCalib greedy over candidate window vectors.

    candidates: int array [layers][num_candidates][kv_heads].
    distortion: either a float array [layers][num_candidates] (a fixed table) or a callable
    (layer, windows[kv_heads], chosen[layer][kv_heads]) -> float.
    Returns (windows [layers][kv_heads], choice [layers], pool bytes).
    """
    cand = np.ascontiguousarray(np.asarray(candidates, dtype=np.int32))
    L, C, H = cand.shape
    if callable(distortion):
        def cb(_user, layer, w_ptr, chosen_ptr):
            w = np.ctypeslib.as_array(w_ptr, shape=(H,)).copy()
            chosen = np.ctypeslib.as_array(chosen_ptr, shape=(L * H,)).reshape(L, H)[:layer].copy()
            return float(distortion(layer, w, chosen))
    else:
        table = np.asarray(distortion, dtype=np.float64)
        if table.shape != (L, C):
            raise ValueError("distortion table must be [layers][num_candidates]")

        base = cand.ctypes.data

        def cb(_user, layer, w_ptr, chosen_ptr):
            # the library passes a pointer into `cand`: its offset names the candidate
            row = (ctypes.cast(w_ptr, ctypes.c_void_p).value - base) // (4 * H)
            return float(table[layer, row % C])
    fn = DISTORTION_FN(cb)
    out_w = np.zeros((L, H), dtype=np.int32)
    choice = np.zeros(L, dtype=np.int32)
    nbytes = ctypes.c_uint64(0)
    _check(load().hwkv_seqcalib(L, H, head_dim, block_size, num_seqs, _dtype_code(dtype), C,
                                cand.ctypes.data_as(_c_i32p), fn, None, int(budget_bytes),
                                out_w.ctypes.data_as(_c_i32p), choice.ctypes.data_as(_c_i32p), ctypes.byref(nbytes)))
    return out_w, choice, nbytes.value


def hwkv_kernel_launches() -> int:
    out = ctypes.c_uint64(0)
    _check(load().hwkv_kernel_launches(ctypes.byref(out)))
    return out.value


def hwkv_check_device_errors(pool: int, stream=None) -> int:
    """Returns the device error bits (0 when clean) without raising."""
    bits = ctypes.c_int32(0)
    load().hwkv_check_device_errors(pool, _stream_ptr(stream), ctypes.byref(bits))
    return bits.value
