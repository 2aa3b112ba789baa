"""The bounded waits.  Every mbarrier wait of every kernel gives up after a time limit and
records HWKV_DEVERR_WAIT_TIMEOUT in the error word instead of spinning forever.
hwkv_wait_selftest runs that same wait loop in one warp: on a phase that has completed (it must
return at once), then on one that nothing completes (it must run out).  The wait that runs out
must be reported with its status, take about its limit, and leave the context usable: a decode
launched afterwards in the same process matches the oracle with a clean error word."""
import pytest
import torch

import head_budgeted_kv_gb300 as hw
from harness import Run, assert_close, small_config

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hw.binding.load()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("limit_us", [500, 20000])
def test_a_wait_nothing_completes_runs_out_and_is_reported(limit_us):
    out = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    hw.hwkv_wait_selftest(limit_us, out)
    torch.cuda.synchronize()
    err, first, waited_us = out.tolist()
    assert err == hw.binding.HWKV_DEVERR_WAIT_TIMEOUT
    assert first == 1  # the completed phase was seen at once
    assert limit_us <= waited_us < limit_us + 200000  # gave up after its limit, not much later


def test_the_context_stays_usable_after_a_wait_ran_out():
    out = torch.zeros(3, dtype=torch.int32, device="cuda")
    hw.hwkv_wait_selftest(1000, out)
    torch.cuda.synchronize()
    assert out[0].item() == hw.binding.HWKV_DEVERR_WAIT_TIMEOUT
    cfg = small_config(name="after_wait", kv_heads=2, windows=((64, 300),), prefill=(500, 40), steps=2)
    run = Run(cfg)
    run.materialize()
    for i in range(cfg.steps):
        for l, (q_raw, got) in run.step(keep_layers=range(cfg.layers)).items():
            assert_close(got, run.reference(i, l, q_raw), cfg, f"step {i} layer {l}")
    assert run.device_errors() == 0  # the pool's own error word never saw the self-test
    run.close()
