"""The C-ABI library without a GPU: it loads, exports every function include/hwkv.h
declares, predicts pool bytes exactly as the oracle does, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads
from head_budgeted_kv_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hwkv.h")


def _declared():
    text = open(HEADER).read()
    return set(re.findall(r"^\s*(?:int|const char\*)\s+(hwkv_\w+)\s*\(", text, flags=re.M))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load()


def test_every_declared_function_is_exported(lib):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert names == {s[0] for s in binding.SIGNATURES}


def test_abi_version_and_status_strings(lib):
    assert binding.hwkv_abi_version() == 3
    assert binding.status_string(0) == "HWKV_OK"
    assert binding.status_string(binding.HWKV_ERR_POOL_TOO_SMALL) == "HWKV_ERR_POOL_TOO_SMALL"


@pytest.mark.parametrize("name", workloads.NAMES)
def test_pool_bytes_match_oracle_on_every_workload(lib, name):
    c = workloads.config(name)
    w = c.windows_array()
    got = binding.hwkv_pool_bytes(c.layers, c.kv_heads, c.head_dim, c.block_size, w, c.batch, c.torch_dtype)
    assert got == oracle.pool_bytes(w, c.batch, c.head_dim, c.block_size, c.elem_bytes)


def test_pool_bytes_of_the_printed_policy(lib):
    c = workloads.config("full")
    got = binding.hwkv_pool_bytes(48, 8, 128, 16, c.windows_array(), 4, binding.HWKV_BF16)
    assert got == 26625441792


@pytest.mark.parametrize("seed", range(10))
def test_pool_bytes_random_geometry(lib, seed):
    rng = np.random.default_rng(seed)
    L, H, bs, B = int(rng.integers(1, 5)), int(rng.integers(1, 33)), int(rng.choice([1, 3, 16, 64])), int(rng.integers(1, 9))
    D = int(rng.choice([64, 128]))
    dt = int(rng.integers(0, 2))
    w = rng.integers(1, 5000, size=(L, H)).astype(np.int32)
    got = binding.hwkv_pool_bytes(L, H, D, bs, w, B, dt)
    assert got == oracle.pool_bytes(w, B, D, bs, 4 if dt == 0 else 2)


def _status(lib, *args):
    w = np.ascontiguousarray(np.asarray(args[4], dtype=np.int32))
    out = ctypes.c_uint64(0)
    return lib.hwkv_pool_bytes(args[0], args[1], args[2], args[3],
                               w.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if w.size else None,
                               args[5], args[6], ctypes.byref(out))


def test_invalid_geometry_is_rejected(lib):
    ok_w = [[16, 32]]
    assert _status(lib, 1, 2, 64, 16, ok_w, 1, 0) == binding.HWKV_OK
    assert _status(lib, 0, 2, 64, 16, ok_w, 1, 0) == binding.HWKV_ERR_INVALID_ARG
    assert _status(lib, 1, 2, 96, 16, ok_w, 1, 0) == binding.HWKV_ERR_UNSUPPORTED
    assert _status(lib, 1, 2, 64, 0, ok_w, 1, 0) == binding.HWKV_ERR_INVALID_ARG
    assert _status(lib, 1, 2, 64, 16, [[16, 0]], 1, 0) == binding.HWKV_ERR_INVALID_ARG
    assert _status(lib, 1, 2, 64, 16, [[16, -4]], 1, 0) == binding.HWKV_ERR_INVALID_ARG
    assert _status(lib, 1, 2, 64, 16, ok_w, 0, 0) == binding.HWKV_ERR_INVALID_ARG
    assert _status(lib, 1, 2, 64, 16, ok_w, 1, 7) == binding.HWKV_ERR_INVALID_ARG
    assert _status(lib, 1, 33, 64, 16, [[16] * 33], 1, 0) == binding.HWKV_ERR_UNSUPPORTED
    assert _status(lib, 1, 2, 64, 16, [], 1, 0) == binding.HWKV_ERR_INVALID_ARG
    # more than 2^31 rows of 2 x block_size
    assert _status(lib, 1, 1, 64, 16, [[2 ** 30]], 2, 0) == binding.HWKV_ERR_UNSUPPORTED
    assert "window" in binding.last_error() or "rows" in binding.last_error() or binding.last_error()


def test_pool_create_checks_size_and_alignment_before_any_launch(lib):
    w = np.asarray([[16, 32]], dtype=np.int32)
    wp = w.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    h = ctypes.c_void_p(0)
    need = oracle.pool_bytes(w, 1, 64, 16, 4)
    fake = 1 << 40  # never dereferenced: both checks come first
    rc = lib.hwkv_pool_create(1, 2, 64, 16, wp, 1, 0, fake, need - 1, None, ctypes.byref(h))
    assert rc == binding.HWKV_ERR_POOL_TOO_SMALL and not h.value
    assert str(need) in binding.last_error()
    rc = lib.hwkv_pool_create(1, 2, 64, 16, wp, 1, 0, fake + 128, need, None, ctypes.byref(h))
    assert rc == binding.HWKV_ERR_ALIGNMENT
    rc = lib.hwkv_pool_create(1, 2, 64, 16, wp, 1, 0, None, need, None, ctypes.byref(h))
    assert rc == binding.HWKV_ERR_INVALID_ARG


def test_null_pool_handles_are_rejected(lib):
    assert lib.hwkv_pool_destroy(None) == binding.HWKV_OK
    assert lib.hwkv_decode_attn(None, 0, None, 4, 1.0, None, None, None, 0, None) == binding.HWKV_ERR_INVALID_ARG
    assert lib.hwkv_append(None, 0, None, None, None, None) == binding.HWKV_ERR_INVALID_ARG
    assert lib.hwkv_set_decode_config(None, 0, 0, 0) == binding.HWKV_ERR_INVALID_ARG
    assert lib.hwkv_append_decode_attn(None, 0, None, 4, 1.0, None, None, None, None, None, 0, None) == binding.HWKV_ERR_INVALID_ARG


def test_wait_selftest_rejects_bad_arguments_before_any_launch(lib):
    # checked on the host: no device is touched (this runs without a GPU)
    assert lib.hwkv_wait_selftest(0, ctypes.c_void_p(16), None) == binding.HWKV_ERR_INVALID_ARG
    assert lib.hwkv_wait_selftest(2000001, ctypes.c_void_p(16), None) == binding.HWKV_ERR_INVALID_ARG
    assert lib.hwkv_wait_selftest(1000, None, None) == binding.HWKV_ERR_INVALID_ARG
    assert lib.hwkv_wait_selftest(1000, ctypes.c_void_p(18), None) == binding.HWKV_ERR_ALIGNMENT


def test_last_error_is_thread_local(lib):
    import threading
    _status(lib, 0, 2, 64, 16, [[16, 32]], 1, 0)
    msg = binding.last_error()
    seen = []
    t = threading.Thread(target=lambda: seen.append(binding.last_error()))
    t.start()
    t.join()
    assert msg and seen == [""]


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError):
        binding.load(build_if_missing=False)


def test_product_package_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "head_budgeted_kv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\boracle\b", text), f
