"""A decode step captured in a CUDA graph gives bit-identical outputs and pool bytes to the
same step run eagerly through the C ABI, and matches the oracle."""
import numpy as np
import pytest
import torch

import head_budgeted_kv_gb300 as hw
from head_budgeted_kv_gb300.graph import DecodeStepGraph
from harness import Run, assert_close, small_config

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hw.binding.load()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("kernel", [hw.HWKV_KERNEL_AUTO, hw.HWKV_KERNEL_SIMT])
def test_graph_replay_equals_eager(fused, kernel):
    cfg = small_config(name="graph", layers=3, kv_heads=2, windows=((64, 512), (256, 32), (1024, 100)),
                       prefill=(600, 250, 1300), steps=3)
    eager = Run(cfg, kernel=kernel, fused=fused)
    graphed = Run(cfg, kernel=kernel, fused=fused)
    eager.materialize()
    graphed.materialize()
    g = DecodeStepGraph(graphed.pool, cfg.scale, cfg.q_heads, graphed.prefill, fused=fused)
    for i in range(cfg.steps):
        res = eager.step(keep_layers=range(cfg.layers))
        q, kn, vn = graphed.wl.step_inputs(i, graphed.dev)
        graphed.host_steps.append((None, kn.cpu(), vn.cpu()))
        g.q.copy_(q)
        g.k_new.copy_(kn)
        g.v_new.copy_(vn)
        g.replay()
        graphed.steps_done += 1
        torch.cuda.synchronize()
        for l in range(cfg.layers):
            got = g.out[l].float().cpu().double().numpy()
            assert np.array_equal(got, res[l][1]), f"step {i} layer {l}"
            assert_close(got, graphed.reference(i, l, res[l][0]), cfg, f"graph step {i} layer {l}")
    assert torch.equal(g.pos, graphed.prefill + cfg.steps)
    assert torch.equal(eager.pool.buffer, graphed.pool.buffer)
    assert eager.device_errors() == 0 and graphed.device_errors() == 0
    eager.close()
    graphed.close()


EARLY_CASES = {
    # about one tile per CTA: single segments, merges of contributors with empty ranges
    "small": dict(name="early", cfg_id=96, layers=3, kv_heads=2, windows=((4096, 64), (256, 1024), (32, 2048)),
                  prefill=(3000, 700, 90), steps=4),
    # ~100 line positions per CTA: boundary segments, bulk-copy and two-level merges, and the
    # L2 prefetch before the dependent-launch wait
    "long_ranges": dict(name="early_long", cfg_id=97, layers=2, kv_heads=4, windows=((65536, 65536, 65536, 65536),
                                                                                    (16384, 65536, 65536, 1024)),
                        prefill=(70000, 66000), steps=3),
}


@pytest.mark.parametrize("case", sorted(EARLY_CASES))
def test_early_reads_equal_default_bit_for_bit(case):
    """Chained fused launches with HWKV_DECODE_EARLY_READS (positions prepared up front, no
    synchronisation between launches, so each schedule may start while the previous launch
    finishes) give the same outputs and rings as the default launches.  Which CTA merges a
    group depends on timing; the outputs must not."""
    cfg = small_config(**EARLY_CASES[case])
    results = []
    for early in (False, True):
        run = Run(cfg, fused=True)
        run.materialize()
        dev = run.dev
        pre = torch.tensor(cfg.prefill, dtype=torch.int32, device=dev)
        pos = [(pre + i).contiguous() for i in range(cfg.steps)]
        ins = [run.wl.step_inputs(i, dev) for i in range(cfg.steps)]
        outs = torch.zeros((cfg.steps, cfg.layers, cfg.batch, cfg.q_heads, cfg.head_dim), dtype=torch.bfloat16,
                           device=dev)
        torch.cuda.synchronize()
        for i in range(cfg.steps):
            q, kn, vn = ins[i]
            for l in range(cfg.layers):
                run.pool.append_decode(l, q[l], cfg.scale, kn[l], vn[l], pos[i], out=outs[i, l], early_reads=early)
        torch.cuda.synchronize()
        assert run.device_errors() == 0
        results.append((outs.clone(), run.pool.buffer.clone()))
        run.close()
    assert torch.equal(results[0][0], results[1][0])
    assert torch.equal(results[0][1], results[1][1])


def test_prepared_launch_equals_plain_calls_bit_for_bit():
    """Pool.decode_launch (arguments marshalled once, then launched per step) gives the same
    outputs and rings as the plain append_decode calls, for the fused and the decode-only forms."""
    cfg = small_config(name="prepared", cfg_id=98, layers=2, kv_heads=2, windows=((1024, 64), (256, 2048)),
                       prefill=(1500, 300), steps=3)
    results = []
    for prepared in (False, True):
        run = Run(cfg, fused=True)
        run.materialize()
        dev = run.dev
        pre = torch.tensor(cfg.prefill, dtype=torch.int32, device=dev)
        pos = [(pre + i).contiguous() for i in range(cfg.steps)]
        ins = [run.wl.step_inputs(i, dev) for i in range(cfg.steps)]
        outs = torch.zeros((cfg.steps + 1, cfg.layers, cfg.batch, cfg.q_heads, cfg.head_dim), dtype=torch.bfloat16,
                           device=dev)
        torch.cuda.synchronize()
        for i in range(cfg.steps):
            q, kn, vn = ins[i]
            for l in range(cfg.layers):
                if prepared:
                    run.pool.decode_launch(l, q[l], cfg.scale, pos[i], outs[i, l], kn[l], vn[l])()
                else:
                    run.pool.append_decode(l, q[l], cfg.scale, kn[l], vn[l], pos[i], out=outs[i, l])
        # decode only (no append) at the lengths after the last step
        lens = (pre + cfg.steps).contiguous()
        q = ins[-1][0]
        for l in range(cfg.layers):
            if prepared:
                run.pool.decode_launch(l, q[l], cfg.scale, lens, outs[cfg.steps, l])()
            else:
                run.pool.decode(l, q[l], cfg.scale, lens, out=outs[cfg.steps, l])
        torch.cuda.synchronize()
        assert run.device_errors() == 0
        results.append((outs.clone(), run.pool.buffer.clone()))
        run.close()
    assert torch.equal(results[0][0], results[1][0])
    assert torch.equal(results[0][1], results[1][1])


def test_advance_positions_in_place_out_of_place_and_wrapping():
    windows = np.full((1, 2), 32, dtype=np.int32)
    pool = hw.Pool(1, 2, 64, 16, windows, 5, torch.bfloat16)
    pos = torch.tensor([0, 7, 2**31 - 1, -3, 1000], dtype=torch.int32, device="cuda")
    out = torch.full_like(pos, 12345)
    before = hw.binding.hwkv_kernel_launches()
    pool.advance_positions(pos, out=out)
    pool.advance_positions(pos, delta=-2)
    torch.cuda.synchronize()
    assert hw.binding.hwkv_kernel_launches() - before == 2
    assert out.cpu().tolist() == [1, 8, -2**31, -2, 1001]
    assert pos.cpu().tolist() == [-2, 5, 2**31 - 3, -5, 998]
    pool.close()


def test_replayed_step_launches_only_library_kernels():
    """Every kernel a captured step records is counted by the library: one per layer and the
    position advance (fused path)."""
    cfg = small_config(name="graph_count", layers=2, kv_heads=2, windows=((64, 512), (256, 32)), prefill=(300,),
                       steps=1)
    run = Run(cfg)
    run.materialize()
    before = hw.binding.hwkv_kernel_launches()
    g = DecodeStepGraph(run.pool, cfg.scale, cfg.q_heads, run.prefill, fused=True)
    assert hw.binding.hwkv_kernel_launches() - before == cfg.layers + 1
    g.replay()
    torch.cuda.synchronize()
    assert g.pos.cpu().tolist() == [cfg.prefill[0] + 1]
    run.close()
