"""Parity at full size, in the launch configuration bench.py times (prepared fused append +
decode launches with early reads, back to back, automatic persistent grid).

The runtime materialises each head's window instead of masking a full cache (HeadWiseKV blog
summary, abstract), so at full size -- where the stream-K partition, the two-level merges, the
overlap of dependent launches and many ring wraps all run -- every output must still equal the
masked attention over the full history, and every pool byte the ring model's.  Each workload
runs all of its decode steps without a host synchronisation between them, then:

* attention: every step of layers {0, 1} and steps {first, middle, last} of every layer are
  compared with the oracle (every query head; for the 64-sequence ragged batch, 8 sequences
  spread over its length range);
* copies: the whole pool region of layers {0, 1, last} is compared bit for bit with the
  oracle's expected pool, and for every (layer, seq, head) the slots of the newest appended
  position and of the oldest resident one hold exactly those positions' K and V rows."""
import dataclasses

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


def _layer_block_base(cfg, layer: int) -> int:
    """First physical block id of ``layer`` under the identity table ((layer, seq, head,
    block) order), from the oracle's block counts."""
    nblk = oracle.blocks_per_head(cfg.windows_array(), cfg.block_size)
    return int(nblk[:layer].sum()) * cfg.batch


def _check_layer_pool(run, cfg, layer: int, name: str):
    """The whole pool region of ``layer`` against oracle.expected_pool, one sequence at a time
    (a sequence's blocks of one layer are contiguous under the identity table)."""
    w = cfg.windows_array()[layer:layer + 1]
    raw_dtype = np.uint16 if cfg.dtype == "bf16" else np.float32
    per_seq = int(oracle.blocks_per_head(w, cfg.block_size).sum())
    base = _layer_block_base(cfg, layer)
    for s in range(cfg.batch):
        exp = oracle.expected_pool(w, 1, cfg.block_size, cfg.head_dim, raw_dtype,
                                   lambda _l, _s, h, lo, hi: run.history(layer, s, h, lo, hi), [cfg.prefill[s]],
                                   run.steps_done)
        first = base + s * per_seq
        ids = [b for h in range(cfg.kv_heads) for b in run.pool.block_table(s, layer, h)]
        assert ids == list(range(first, first + per_seq)) and exp.shape[0] == per_seq
        got = run.gpu_blocks(np.arange(first, first + per_seq))
        bad = np.argwhere((got != exp).reshape(per_seq, -1).any(axis=1))
        assert bad.size == 0, f"{name}: layer {layer} seq {s}: {bad.size} of {per_seq} blocks differ " \
                              f"(first {first + bad[0, 0]})"


def _check_newest_and_oldest_slots(run, cfg, name: str):
    """For every (layer, seq, head): the slot of the newest appended position and the slot of
    the oldest position the last step's window holds carry those positions' rows."""
    blocks = run.pool.blocks()
    tables = oracle_table(cfg)
    cap = oracle.ring_capacity(cfg.windows_array(), cfg.block_size)
    bs = cfg.block_size
    last_step = run.steps_done - 1
    for l in range(cfg.layers):
        rows_blk, rows_r, expect = [], [], []
        for s in range(cfg.batch):
            L = cfg.prefill[s]
            length = L + run.steps_done
            pre = run.wl.prefill_seq(l, s, run.dev) if length - max(cfg.windows[l]) < L else None
            for h in range(cfg.kv_heads):
                C = int(cap[l, h])
                newest = L + last_step
                oldest, _ = oracle.window_span(length, int(cfg.windows[l][h]))
                for p in (newest, oldest):
                    slot = p % C
                    rows_blk.append(tables[(l, s, h)][slot // bs])
                    rows_r.append(slot % bs)
                    if p >= L:
                        _, kn, vn = run.host_steps[p - L]
                        expect.append((workloads.to_raw(kn[l, s, h]), workloads.to_raw(vn[l, s, h])))
                    else:
                        expect.append((workloads.to_raw(pre[0][h, p]), workloads.to_raw(pre[1][h, p])))
        bi = torch.as_tensor(rows_blk, dtype=torch.int64, device=run.dev)
        ri = torch.as_tensor(rows_r, dtype=torch.int64, device=run.dev)
        got_k = workloads.to_raw(blocks[bi, 0, ri])
        got_v = workloads.to_raw(blocks[bi, 1, ri])
        for j, (ek, ev) in enumerate(expect):
            assert np.array_equal(got_k[j], ek) and np.array_equal(got_v[j], ev), \
                f"{name}: layer {l} slot check {j} (block {rows_blk[j]} row {rows_r[j]})"


@pytest.mark.parametrize("name", ["full", "ragged", "long", "long_full"])
def test_full_size_parity(name):
    cfg = workloads.config(name)
    free, _ = torch.cuda.mem_get_info()
    need = oracle.pool_bytes(cfg.windows_array(), cfg.batch, cfg.head_dim, cfg.block_size, cfg.elem_bytes)
    if need * 1.6 > free:
        pytest.skip(f"needs ~{need * 1.6 / 1e9:.0f} GB of device memory")
    run = Run(cfg, fused=True)
    assert run.pool.nbytes == need
    run.materialize()
    seqs = _sample_seqs(cfg)
    mid, last = cfg.steps // 2, cfg.steps - 1
    pairs = {(i, l) for i in range(cfg.steps) for l in (0, 1)}
    pairs |= {(i, l) for i in (0, mid, last) for l in range(cfg.layers)}
    res = run.run_prepared(pairs=pairs)
    assert run.device_errors() == 0
    sel = slice(None) if seqs is None else seqs
    for l in range(cfg.layers):
        hist = run.layer_histories(l, seqs)
        for i in sorted(i for (i, ll) in pairs if ll == l):
            q_raw, got = res.pop((i, l))
            ref = run.reference_hoisted(hist, i, l, q_raw, seqs=seqs)
            assert_close(got[sel], ref[sel], cfg, f"{name} step {i} layer {l}")
        del hist
    assert not res

    for l in sorted({0, 1, cfg.layers - 1}):
        _check_layer_pool(run, cfg, l, name)
    _check_newest_and_oldest_slots(run, cfg, name)
    run.close()


# the other decode shapes bench.py --mode shapes times, as it builds them
SHAPES = {"bf16_d64_gqa4": {"head_dim": 64}, "bf16_d64_gqa16": {"head_dim": 64, "q_heads": 128},
          "bf16_d128_gqa16": {"q_heads": 128}, "fp32_d128_gqa4": {"dtype": "f32"}}


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_decode_shapes_full_geometry_parity(shape):
    """The full geometry's first 8 layers (batch 4, 112K, the page's per-head windows) at another
    head_dim, GQA group or dtype, in the launch configuration the shapes benchmark times: every
    query head of steps {0, 2, 5} of layers {0, 1, 7} against the oracle; the pool of layers
    {0, 7} bit for bit; newest and oldest resident slots of every (layer, seq, head)."""
    cfg = dataclasses.replace(workloads.config("full").with_layers(8).with_steps(6), name="full_8l", **SHAPES[shape])
    free, _ = torch.cuda.mem_get_info()
    need = oracle.pool_bytes(cfg.windows_array(), cfg.batch, cfg.head_dim, cfg.block_size, cfg.elem_bytes)
    if need * 1.6 > free:
        pytest.skip(f"needs ~{need * 1.6 / 1e9:.0f} GB of device memory")
    run = Run(cfg, fused=True)
    run.materialize()
    pairs = {(i, l) for i in (0, 2, 5) for l in (0, 1, 7)}
    res = run.run_prepared(pairs=pairs)
    assert run.device_errors() == 0
    for l in (0, 1, 7):
        hist = run.layer_histories(l, None)
        for i in (0, 2, 5):
            q_raw, got = res.pop((i, l))
            assert_close(got, run.reference_hoisted(hist, i, l, q_raw), cfg, f"{shape} step {i} layer {l}")
        del hist
    assert not res
    for l in (0, 7):
        _check_layer_pool(run, cfg, l, shape)
    _check_newest_and_oldest_slots(run, cfg, shape)
    run.close()
