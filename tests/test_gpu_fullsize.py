"""Parity at full size, in the launch configuration bench.py times (prepared fused append +
decode launches with early reads, back to back, automatic persistent grid), on sampled outputs
the oracle computes one by one.

Each workload runs all of its decode steps without a host synchronisation between them.  At the
first, middle and last step the outputs of layers {0, 1, last} are compared with the oracle
(every query head; for the 64-sequence ragged batch, 8 sequences spread over its length range).
After the last step the ring contents of sampled heads are compared bit for bit with the
oracle's ring model."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import head_budgeted_kv_gb300 as hw
from harness import Run, assert_close, oracle_table

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hw.binding.load()
    yield
    torch.cuda.synchronize()


def _sample_seqs(cfg, n=8):
    if cfg.batch <= n:
        return None
    order = np.argsort(np.asarray(cfg.prefill))
    pick = order[np.linspace(0, cfg.batch - 1, n).round().astype(int)]
    return sorted(int(s) for s in pick)


@pytest.mark.parametrize("name", ["full", "ragged", "long", "long_full"])
def test_full_size_sampled_parity(name):
    cfg = workloads.config(name)
    free, _ = torch.cuda.mem_get_info()
    need = oracle.pool_bytes(cfg.windows_array(), cfg.batch, cfg.head_dim, cfg.block_size, cfg.elem_bytes)
    if need * 1.6 > free:
        pytest.skip(f"needs ~{need * 1.6 / 1e9:.0f} GB of device memory")
    run = Run(cfg, fused=True)
    assert run.pool.nbytes == need
    run.materialize()
    seqs = _sample_seqs(cfg)
    check_steps = {0, cfg.steps // 2, cfg.steps - 1}
    check_layers = sorted({0, 1, cfg.layers - 1})
    res = run.run_prepared(sorted(check_steps), check_layers)
    for (i, l), (q_raw, got) in sorted(res.items()):
        ref = run.reference(i, l, q_raw, seqs=seqs)
        sel = slice(None) if seqs is None else seqs
        assert_close(got[sel], ref[sel], cfg, f"{name} step {i} layer {l}")
    assert run.device_errors() == 0

    # ring contents of sampled heads, bit for bit
    tables = oracle_table(cfg)
    rng = np.random.default_rng(7)
    heads = [(0, 0, 0), (cfg.layers - 1, cfg.batch - 1, cfg.kv_heads - 1)]
    heads += [(int(rng.integers(cfg.layers)), int(rng.integers(cfg.batch)), int(rng.integers(cfg.kv_heads)))
              for _ in range(4)]
    for (l, s, h) in heads:
        ids = tables[(l, s, h)]
        assert run.pool.block_table(s, l, h).tolist() == ids
        exp, _, _ = run.expected_ring_blocks(l, s, h)
        assert np.array_equal(run.gpu_blocks(ids), exp), f"{name}: ring of layer {l} seq {s} head {h}"
    run.close()
