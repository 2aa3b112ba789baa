"""hwkv_decode_attn_noalloc: decode attention for callers that cannot allocate device memory
where they run attention (for example while a CUDA graph is being captured, or under an
allocator that owns all device memory).  Its split-K scratch is a fixed array inside the
library.  Decode launches are deterministic (no output depends on which CTA arrives last),
so it must give exactly the bits of hwkv_decode_attn, which takes a caller workspace -- here
on two calls in a row, each after an append, so the second call starts from the first call's
leftovers in the shared array -- and both must match the CPU oracle within the bf16
tolerance.

Kept in a file of its own, collected last."""
import ctypes

import numpy as np
import pytest
import torch

import head_budgeted_kv_gb300 as hw
import workloads
from harness import Run, assert_close, small_config

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hw.binding.load()
    yield
    torch.cuda.synchronize()


def _call_noalloc(lib, pool, layer, q, scale, lens, out):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.hwkv_decode_attn_noalloc(pool, layer, q.data_ptr(), q.shape[1], ctypes.c_float(scale),
                                        lens.data_ptr(), out.data_ptr(), stream)


@pytest.mark.parametrize("kernel", [hw.HWKV_KERNEL_AUTO, hw.HWKV_KERNEL_SIMT])
def test_noalloc_matches_decode_attn_on_two_consecutive_calls(kernel):
    lib = hw.binding.load()
    # heads shared by several CTAs (partials go through the scratch) and single-CTA heads
    cfg = small_config(name="noalloc", kv_heads=4, windows=((4096, 1024, 256, 2000),), prefill=(5000, 1500, 300))
    run = Run(cfg, kernel=kernel)
    run.materialize()
    need = hw.hwkv_decode_workspace_bytes(run.pool.handle, cfg.q_heads)
    assert 0 < need <= (4 << 20)  # the scratch is used, and fits the static array
    for step in range(2):
        q, kn, vn = run.wl.step_inputs(step, run.dev)
        run.host_steps.append((None, kn.cpu(), vn.cpu()))
        pos = run.prefill + step
        lens = pos + 1
        run.pool.append(0, kn[0], vn[0], pos)
        run.steps_done += 1
        ref = torch.empty_like(q[0])
        hw.hwkv_decode_attn(run.pool.handle, 0, q[0], cfg.scale, lens, ref, run.pool.workspace)
        got = torch.full_like(q[0], float("nan"))
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        rc = _call_noalloc(lib, run.pool.handle, 0, q[0], cfg.scale, lens, got)
        assert rc == hw.binding.HWKV_OK, hw.binding.last_error()
        torch.cuda.synchronize()
        if step == 1:
            # the first call on the device may load the module that holds the array; later
            # calls leave the device's free memory exactly as it was
            assert torch.cuda.mem_get_info()[0] == free0
        assert torch.equal(got, ref), f"noalloc call {step + 1} differs from hwkv_decode_attn"
        oracle_out = run.reference(step, 0, workloads.to_raw(q[0]))
        assert_close(got.float().cpu().double().numpy(), oracle_out, cfg, f"noalloc call {step + 1} vs the oracle")
    assert run.device_errors() == 0
    run.close()


def test_noalloc_rejects_scratch_beyond_its_array():
    lib = hw.binding.load()
    # 64 sequences x 32 kv heads x GQA 8: the split-K partials need more than 4 MiB
    B, H, G, D = 64, 32, 8, 128
    windows = np.full((1, H), 16, dtype=np.int32)
    pool = hw.Pool(1, H, D, 16, windows, B, torch.bfloat16, q_heads=H * G)
    need = hw.hwkv_decode_workspace_bytes(pool.handle, H * G)
    assert need > (4 << 20)
    q = torch.zeros(B, H * G, D, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    rc = _call_noalloc(lib, pool.handle, 0, q, 0.1, lens, out)
    assert rc == hw.binding.HWKV_ERR_WORKSPACE_TOO_SMALL
    msg = hw.binding.last_error()
    assert str(need) in msg and str(4 << 20) in msg
    torch.cuda.synchronize()
    assert not out.float().abs().sum().item()  # nothing was launched
    pool.close()
