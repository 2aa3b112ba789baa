"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Copies and tables are compared bit for bit; attention within |gpu - ref| <= 1e-5 (fp32
inputs) or <= 2e-2 + 2e-2 |ref| (bf16 inputs, fp32 accumulation)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import head_budgeted_kv_gb300 as hw
from harness import Run, assert_close, oracle_table, small_config

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hw.binding.load()
    yield
    torch.cuda.synchronize()


def _check_all_pool_blocks(run: Run):
    cfg = run.cfg
    tables = oracle_table(cfg)
    for (l, s, h), ids in tables.items():
        assert run.pool.block_table(s, l, h).tolist() == ids
        exp, _, _ = run.expected_ring_blocks(l, s, h)
        got = run.gpu_blocks(ids)
        assert np.array_equal(got, exp), f"pool bytes of layer {l} seq {s} head {h}"


# ---------------------------------------------------------------------------------------
# the tiny fp32 workload: everything, every step
# ---------------------------------------------------------------------------------------
@pytest.mark.parametrize("kernel", [hw.HWKV_KERNEL_AUTO, hw.HWKV_KERNEL_SIMT])
def test_tiny_fp32_every_step_every_head(kernel):
    """The fp32 workload through the stream-K kernel (automatic choice) and the split kernel."""
    cfg = workloads.config("tiny")
    run = Run(cfg, kernel=kernel)
    exp_bytes = oracle.pool_bytes(cfg.windows_array(), cfg.batch, cfg.head_dim, cfg.block_size, cfg.elem_bytes)
    assert run.pool.nbytes == exp_bytes == 81920
    assert run.pool.geometry()[0] == exp_bytes
    run.materialize()
    _check_all_pool_blocks(run)
    for i in range(cfg.steps):
        res = run.step(keep_layers=[0])
        q_raw, got = res[0]
        ref = run.reference(i, 0, q_raw)
        assert_close(got, ref, cfg, f"tiny step {i}")
        _check_all_pool_blocks(run)
    assert run.device_errors() == 0
    run.close()


# ---------------------------------------------------------------------------------------
# the single-layer bf16 workload: whole pool bit-exact, every head's output
# ---------------------------------------------------------------------------------------
@pytest.mark.parametrize("kernel", [hw.HWKV_KERNEL_TENSOR, hw.HWKV_KERNEL_SIMT])
def test_layer_bf16_full(kernel):
    cfg = workloads.config("layer")
    run = Run(cfg, kernel=kernel)
    run.materialize()
    res = run.step(keep_layers=[0])
    q_raw, got = res[0]
    ref = run.reference(0, 0, q_raw)
    assert_close(got, ref, cfg, "layer bf16")
    if kernel == hw.HWKV_KERNEL_TENSOR:
        _check_all_pool_blocks(run)
    assert run.device_errors() == 0
    run.close()


# ---------------------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------------------
EDGE = {
    # windows larger than the context (clip to len), ragged lengths
    "clip": dict(kv_heads=3, windows=((1024, 16, 4096),), prefill=(5, 40, 300, 17)),
    # window not a multiple of the block size: ring of 48 slots holds a 40-token window
    "ring_c_gt_w": dict(kv_heads=2, windows=((40, 24),), prefill=(300, 47), steps=5),
    # windows of one token
    "w1": dict(kv_heads=2, windows=((1, 1),), prefill=(50, 3)),
    # GQA 1, 2, 8 and head_dim 64
    "g1_d64": dict(kv_heads=4, group=1, head_dim=64, windows=((64, 128, 32, 512),), prefill=(700, 90)),
    "g2": dict(kv_heads=2, group=2, windows=((256, 96),), prefill=(1000, 1000)),
    "g8": dict(kv_heads=2, group=8, windows=((2048, 160),), prefill=(3000, 100)),
    # groups past one 8-column n-tile (16, and 12 padded to 16), and padded small groups
    "g16": dict(kv_heads=2, group=16, windows=((4096, 96),), prefill=(5000, 300)),
    "g12_d64": dict(kv_heads=2, group=12, head_dim=64, windows=((512, 2048),), prefill=(1500, 2100)),
    "g3": dict(kv_heads=3, group=3, windows=((256, 64, 1024),), prefill=(900, 40)),
    "g6": dict(kv_heads=2, group=6, windows=((128, 700),), prefill=(800, 650)),
    # bigger block size, several layers
    "bs64_layers": dict(layers=3, kv_heads=2, block_size=64, windows=((128, 1024), (64, 256), (4096, 64)),
                        prefill=(5000, 700, 64)),
    # odd block size -> CUDA-core kernel
    "bs5": dict(kv_heads=2, block_size=5, windows=((23, 60),), prefill=(100, 9)),
    # fp32 with several layers and GQA 4 (stream-K tiles), GQA 8 (split kernel), head_dim 64
    "f32": dict(layers=2, kv_heads=2, dtype="f32", head_dim=128, windows=((100, 37), (16, 300)), prefill=(400, 20)),
    "f32_g8": dict(kv_heads=2, group=8, dtype="f32", head_dim=128, windows=((700, 48),), prefill=(900, 30)),
    "f32_d64_long": dict(kv_heads=3, group=3, dtype="f32", head_dim=64, windows=((4096, 64, 1000),),
                         prefill=(5000, 20)),
    # spiky keys (x8) as in the ragged workload
    "spikes": dict(kv_heads=2, windows=((1024, 512),), prefill=(2000, 1500), spike_frac=0.05),
    # more sequences than a CTA stages lengths for in shared memory (256): the lengths are read
    # from global memory; ragged, some prefills empty
    "many_seqs": dict(kv_heads=2, windows=((48, 200),), prefill=tuple((i * 37) % 400 for i in range(300))),
}


@pytest.mark.parametrize("name", sorted(EDGE))
@pytest.mark.parametrize("kernel", [hw.HWKV_KERNEL_AUTO, hw.HWKV_KERNEL_SIMT])
def test_edge_cases(name, kernel):
    spec = dict(EDGE[name])
    steps = spec.pop("steps", 3)
    cfg = small_config(name=name, steps=steps, **spec)
    run = Run(cfg, kernel=kernel)
    run.materialize()
    for i in range(steps):
        res = run.step(keep_layers=range(cfg.layers))
        for l, (q_raw, got) in res.items():
            ref = run.reference(i, l, q_raw)
            assert_close(got, ref, cfg, f"{name} step {i} layer {l}")
    _check_all_pool_blocks(run)
    assert run.device_errors() == 0
    run.close()


def test_window_one_returns_the_new_value_exactly():
    cfg = small_config(name="w1x", kv_heads=2, windows=((1, 1),), prefill=(50, 3))
    run = Run(cfg)
    run.materialize()
    _, kn, vn = run.wl.step_inputs(0, run.dev)
    res = run.step(keep_layers=[0])
    _, got = res[0]
    v = vn[0].float().cpu().double().numpy()          # [B][H][D]
    exp = np.repeat(v, cfg.group, axis=1)             # query head q reads kv head q // G
    assert np.array_equal(got, exp)
    run.close()


def test_empty_context_gives_zero_output():
    cfg = small_config(name="empty", kv_heads=2, windows=((64, 32),), prefill=(0, 0))
    run = Run(cfg)
    run.materialize()
    q = torch.randn(2, cfg.q_heads, cfg.head_dim, device=run.dev).to(torch.bfloat16)
    lens = torch.zeros(2, dtype=torch.int32, device=run.dev)
    out = torch.full_like(q, 7.0)
    run.pool.decode(0, q, cfg.scale, lens, out=out)
    torch.cuda.synchronize()
    assert not out.float().abs().sum().item()
    assert run.device_errors() == 0
    run.close()


@pytest.mark.parametrize("split", [16, 64, 256, 4096])
def test_simt_split_size_changes_rounding_only(split):
    cfg = small_config(name="split", kv_heads=4, windows=((4096, 1024, 256, 2000),), prefill=(5000, 1500, 300))
    run = Run(cfg, kernel=hw.HWKV_KERNEL_SIMT, split=split)
    run.materialize()
    res = run.step(keep_layers=[0])
    q_raw, got = res[0]
    assert_close(got, run.reference(0, 0, q_raw), cfg, f"split {split}")
    assert run.device_errors() == 0
    run.close()


@pytest.mark.parametrize("workers", [1, 2, 3, 7, 64, 1000, 5000])
def test_tensor_core_partition_changes_rounding_only(workers):
    """The persistent grid's size decides how the resident tiles are split into ranges and
    how many partials each head merges; more workers than tiles leaves some empty."""
    cfg = small_config(name="workers", kv_heads=4, windows=((4096, 1024, 256, 2000),), prefill=(5000, 1500, 300))
    run = Run(cfg, kernel=hw.HWKV_KERNEL_TENSOR, workers=workers)
    run.materialize()
    for i in range(2):
        res = run.step(keep_layers=[0])
        q_raw, got = res[0]
        assert_close(got, run.reference(i, 0, q_raw), cfg, f"workers {workers} step {i}")
    assert run.device_errors() == 0
    run.close()


@pytest.mark.parametrize("workers", [40, 60, 100, 160, 288])
def test_long_window_merge_at_batch_one(workers):
    """A 64K window at batch 1 spread over 40 .. 288 CTAs: its ~40 .. 280 contributors are
    merged in two levels (blocks of 8, then the blocks); every variant matches the oracle and
    repeats bit for bit."""
    cfg = small_config(name="merge1", kv_heads=2, windows=((65536, 1024),), prefill=(70000,))
    runs = [Run(cfg, kernel=hw.HWKV_KERNEL_TENSOR, workers=workers, fused=True) for _ in range(2)]
    for r in runs:
        r.materialize()
    for i in range(2):
        a, b = (r.step(keep_layers=[0]) for r in runs)
        assert np.array_equal(a[0][1], b[0][1]), f"workers {workers} step {i}"
        assert_close(a[0][1], runs[0].reference(i, 0, a[0][0]), cfg, f"workers {workers} step {i}")
    for r in runs:
        assert r.device_errors() == 0
        r.close()


@pytest.mark.parametrize("head_dim,workers", [(128, 40), (128, 56), (64, 48), (64, 64)])
def test_large_group_merge_in_head_passes(head_dim, workers):
    """GQA 16: a partial is 16 x head_dim floats, so a one-level merge of 13-24 partials exceeds
    the stage buffers and runs in passes over subsets of the query heads; it must match the
    oracle and repeat bit for bit."""
    cfg = small_config(name="bigg", kv_heads=2, group=16, head_dim=head_dim, windows=((8192, 4096),),
                       prefill=(9000, 9000))
    runs = [Run(cfg, kernel=hw.HWKV_KERNEL_TENSOR, workers=workers, fused=True) for _ in range(2)]
    for r in runs:
        r.materialize()
    for i in range(2):
        a, b = (r.step(keep_layers=[0]) for r in runs)
        assert np.array_equal(a[0][1], b[0][1]), f"D{head_dim} workers {workers} step {i}"
        assert_close(a[0][1], runs[0].reference(i, 0, a[0][0]), cfg, f"D{head_dim} workers {workers} step {i}")
    for r in runs:
        assert r.device_errors() == 0
        r.close()


@pytest.mark.parametrize("kernel", [hw.HWKV_KERNEL_TENSOR, hw.HWKV_KERNEL_SIMT])
def test_launches_are_deterministic(kernel):
    """No output depends on which CTA arrives last at a merge: two pools driven with the same
    inputs give the same bits (64K windows at batch 3 take the two-level merge)."""
    cfg = small_config(name="det", layers=2, kv_heads=4, windows=((65536, 1024, 256, 16384), (4096, 64, 8192, 2000)),
                       prefill=(70000, 1500, 20000))
    runs = [Run(cfg, kernel=kernel, fused=True) for _ in range(2)]
    for r in runs:
        r.materialize()
    for i in range(2):
        a, b = (r.step(keep_layers=range(cfg.layers)) for r in runs)
        for l in range(cfg.layers):
            assert np.array_equal(a[l][1], b[l][1]), f"step {i} layer {l}"
            assert_close(a[l][1], runs[0].reference(i, l, a[l][0]), cfg, f"step {i} layer {l}")
    for r in runs:
        assert r.device_errors() == 0
        r.close()


@pytest.mark.parametrize("name", ["clip", "ring_c_gt_w", "g8", "g16", "bs64_layers", "bs5", "f32"])
def test_fused_append_decode_equals_append_then_decode(name):
    """hwkv_append_decode_attn gives the same pool bytes and the same outputs as hwkv_append
    followed by hwkv_decode_attn, and matches the oracle."""
    spec = dict(EDGE[name])
    steps = spec.pop("steps", 3)
    cfg = small_config(name=name, steps=steps, **spec)
    split, fused = Run(cfg), Run(cfg, fused=True)
    split.materialize()
    fused.materialize()
    for i in range(steps):
        ra = split.step(keep_layers=range(cfg.layers))
        rb = fused.step(keep_layers=range(cfg.layers))
        for l in range(cfg.layers):
            assert np.array_equal(ra[l][1], rb[l][1]), f"{name} step {i} layer {l}"
            assert_close(rb[l][1], fused.reference(i, l, rb[l][0]), cfg, f"fused {name} step {i} layer {l}")
    torch.cuda.synchronize()
    assert torch.equal(split.pool.buffer, fused.pool.buffer)
    assert split.device_errors() == 0 and fused.device_errors() == 0
    split.close()
    fused.close()


def test_block_permutation_leaves_output_bit_identical():
    cfg = small_config(name="perm", layers=2, kv_heads=2, windows=((64, 512), (256, 32)), prefill=(600, 250))
    base = Run(cfg)
    base.materialize()
    out_a = base.step(keep_layers=[0, 1])
    # same inputs, then permute physical blocks: move the bytes and the table together
    perm_run = Run(cfg)
    perm_run.materialize()
    _, total, _ = perm_run.pool.geometry()
    rng = np.random.default_rng(0)
    perm = rng.permutation(total).astype(np.int32)         # logical entry i -> new physical id perm[i]
    blocks = perm_run.pool.blocks()
    moved = torch.empty_like(blocks)
    moved[torch.as_tensor(perm, device=perm_run.dev).long()] = blocks
    blocks.copy_(moved)
    perm_run.pool.set_block_table(perm)                    # identity table -> permuted ids
    out_b = perm_run.step(keep_layers=[0, 1])
    for l in (0, 1):
        assert np.array_equal(out_a[l][1], out_b[l][1])
    # the pool still decodes to the oracle's rings through the permuted table
    for (l, s, h), ids in oracle_table(cfg).items():
        exp, _, _ = perm_run.expected_ring_blocks(l, s, h)
        got = perm_run.gpu_blocks(perm[np.asarray(ids)])
        assert np.array_equal(got, exp)
    base.close()
    perm_run.close()


def test_canary_outside_written_slots_is_untouched():
    cfg = small_config(name="canary", kv_heads=2, windows=((40, 100),), prefill=(300, 30), steps=4)
    run = Run(cfg, canary=0xA5)
    run.materialize()
    for _ in range(cfg.steps):
        run.step()
    canary = np.uint16(0xA5A5)
    for (l, s, h), ids in oracle_table(cfg).items():
        exp, writes, C = run.expected_ring_blocks(l, s, h)
        got = run.gpu_blocks(ids)
        written = {p % C for p in writes}
        for t in range(C):
            j, r = divmod(t, cfg.block_size)
            if t in written:
                assert np.array_equal(got[j, :, r], exp[j, :, r])
            else:
                assert (got[j, :, r] == canary).all(), (l, s, h, t)
    run.close()


def test_pool_bytes_equal_allocation():
    cfg = small_config(name="alloc", layers=2, kv_heads=3, windows=((1024, 4096, 16), (64, 65536, 1)), prefill=(10,))
    before = torch.cuda.memory_allocated()
    pool = hw.Pool(cfg.layers, cfg.kv_heads, cfg.head_dim, cfg.block_size, cfg.windows_array(), cfg.batch,
                   torch.bfloat16, q_heads=cfg.q_heads)
    pred = oracle.pool_bytes(cfg.windows_array(), cfg.batch, cfg.head_dim, cfg.block_size, 2)
    assert pool.nbytes == pred
    assert pool.buffer.numel() == pred
    ws = pool.workspace.numel()
    assert torch.cuda.memory_allocated() - before == pred + ws or torch.cuda.memory_allocated() - before >= pred
    pool.close()


# ---------------------------------------------------------------------------------------
# failures are reported, never faulted
# ---------------------------------------------------------------------------------------
def test_negative_position_and_oversized_prefill_are_flagged():
    cfg = small_config(name="flags", kv_heads=2, windows=((64, 32),), prefill=(100,))
    run = Run(cfg)
    K = torch.zeros(1, 2, 100, cfg.head_dim, dtype=torch.bfloat16, device=run.dev)
    bad_len = torch.tensor([101], dtype=torch.int32, device=run.dev)   # above max_len = 100
    run.pool.materialize(0, K, K, bad_len)
    assert run.device_errors() & hw.binding.HWKV_DEVERR_SRC_RANGE
    kn = torch.zeros(1, 2, cfg.head_dim, dtype=torch.bfloat16, device=run.dev)
    run.pool.append(0, kn, kn, torch.tensor([-3], dtype=torch.int32, device=run.dev))
    assert run.device_errors() & hw.binding.HWKV_DEVERR_NEG_LENGTH
    assert run.device_errors() == 0   # cleared by the previous read
    assert not run.pool.buffer.any().item()  # nothing was written
    run.close()


def test_host_side_argument_errors():
    cfg = small_config(name="args", kv_heads=2, windows=((4096, 64),), prefill=(100,))
    run = Run(cfg)
    q = torch.zeros(1, cfg.q_heads, cfg.head_dim, dtype=torch.bfloat16, device=run.dev)
    lens = torch.ones(1, dtype=torch.int32, device=run.dev)
    out = torch.empty_like(q)
    small_ws = torch.empty(16, dtype=torch.uint8, device=run.dev)
    with pytest.raises(hw.HwkvError) as e:
        hw.hwkv_decode_attn(run.pool.handle, 0, q, cfg.scale, lens, out, small_ws)
    assert e.value.status == hw.binding.HWKV_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(hw.HwkvError) as e:
        hw.hwkv_decode_attn(run.pool.handle, 1, q, cfg.scale, lens, out, run.pool.workspace)
    assert e.value.status == hw.binding.HWKV_ERR_INVALID_ARG
    big = torch.zeros(2 * q.numel() + 8, dtype=torch.bfloat16, device=run.dev)
    qmis = big[1:1 + q.numel()].view_as(q)                     # 2-byte offset
    with pytest.raises(hw.HwkvError) as e:
        hw.hwkv_decode_attn(run.pool.handle, 0, qmis, cfg.scale, lens, out, run.pool.workspace)
    assert e.value.status == hw.binding.HWKV_ERR_ALIGNMENT
    q17 = torch.zeros(1, cfg.kv_heads * 17, cfg.head_dim, dtype=torch.bfloat16, device=run.dev)  # group 17
    with pytest.raises(hw.HwkvError) as e:
        hw.hwkv_decode_attn(run.pool.handle, 0, q17, cfg.scale, lens, torch.empty_like(q17), run.pool.workspace)
    assert e.value.status == hw.binding.HWKV_ERR_UNSUPPORTED
    with pytest.raises(hw.HwkvError) as e:
        hw.hwkv_set_block_table(run.pool.handle, np.zeros(run.pool.geometry()[1], np.int32))
    assert e.value.status == hw.binding.HWKV_ERR_INVALID_ARG
    buf = torch.empty(run.pool.nbytes - 256, dtype=torch.uint8, device=run.dev)
    with pytest.raises(hw.HwkvError) as e:
        hw.hwkv_pool_create(1, 2, cfg.head_dim, 16, cfg.windows_array(), 1, torch.bfloat16, buf)
    assert e.value.status == hw.binding.HWKV_ERR_POOL_TOO_SMALL
    assert run.device_errors() == 0
    run.close()


def _random_case(seed: int):
    """A seeded random small geometry: GQA group, head_dim, block size, per-head windows (some
    not multiples of the block size, some beyond the context), ragged lengths, fused or not,
    and a persistent grid from one CTA to more CTAs than tiles."""
    rng = np.random.default_rng(1000 + seed)
    kv_heads = int(rng.integers(1, 6))
    group = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16]))
    head_dim = int(rng.choice([64, 128]))
    block_size = int(rng.choice([16, 32, 64]))
    layers = int(rng.integers(1, 3))
    batch = int(rng.integers(1, 5))
    windows = tuple(tuple(int(rng.choice([int(rng.integers(1, 200)), 256, 1000, 2048, 4096, 8192]))
                          for _ in range(kv_heads)) for _ in range(layers))
    prefill = tuple(int(rng.integers(0, 9000)) for _ in range(batch))
    fused = bool(rng.integers(0, 2))
    workers = int(rng.choice([0, 0, 1, 3, 17, 100, 288, 1000]))
    cfg = small_config(name=f"random{seed}", cfg_id=200 + seed, layers=layers, kv_heads=kv_heads, group=group,
                       head_dim=head_dim, block_size=block_size, windows=windows, prefill=prefill, steps=2)
    return cfg, fused, workers


def _random_case_f32(seed: int):
    """As _random_case, fp32 pools: up to 4 query heads per KV head take the stream-K kernel
    (CUDA-core tiles), more the split kernel."""
    rng = np.random.default_rng(3000 + seed)
    kv_heads = int(rng.integers(1, 5))
    group = int(rng.choice([1, 2, 3, 4, 4, 6]))
    layers = int(rng.integers(1, 3))
    batch = int(rng.integers(1, 4))
    windows = tuple(tuple(int(rng.choice([int(rng.integers(1, 200)), 256, 1000, 4096]))
                          for _ in range(kv_heads)) for _ in range(layers))
    prefill = tuple(int(rng.integers(0, 5000)) for _ in range(batch))
    cfg = small_config(name=f"random_f32_{seed}", cfg_id=300 + seed, layers=layers, kv_heads=kv_heads, group=group,
                       head_dim=int(rng.choice([64, 128])), block_size=int(rng.choice([16, 32, 64])),
                       dtype="f32", windows=windows, prefill=prefill, steps=2)
    return cfg, bool(rng.integers(0, 2)), int(rng.choice([0, 0, 1, 5, 64, 500]))


@pytest.mark.parametrize("seed", range(8))
def test_random_f32_geometries_match_the_oracle(seed):
    cfg, fused, workers = _random_case_f32(seed)
    run = Run(cfg, fused=fused, workers=workers)
    run.materialize()
    for i in range(cfg.steps):
        res = run.step(keep_layers=range(cfg.layers))
        for l, (q_raw, got) in res.items():
            ref = run.reference(i, l, q_raw)
            assert_close(got, ref, cfg, f"random f32 {seed} (fused {fused}, workers {workers}) step {i} layer {l}")
    _check_all_pool_blocks(run)
    assert run.device_errors() == 0
    run.close()


@pytest.mark.parametrize("seed", range(16))
def test_random_geometries_match_the_oracle(seed):
    cfg, fused, workers = _random_case(seed)
    run = Run(cfg, fused=fused, workers=workers)
    run.materialize()
    for i in range(cfg.steps):
        res = run.step(keep_layers=range(cfg.layers))
        for l, (q_raw, got) in res.items():
            ref = run.reference(i, l, q_raw)
            assert_close(got, ref, cfg, f"random {seed} (fused {fused}, workers {workers}) step {i} layer {l}")
    _check_all_pool_blocks(run)
    assert run.device_errors() == 0
    run.close()


def test_many_sequences_through_prepared_fused_launches():
    """300 sequences (beyond the 256 whose lengths a CTA stages in shared memory) through the
    launches the benchmark issues: prepared fused append + decode with early reads, back to
    back; every step and layer against the oracle, every pool block bit for bit."""
    cfg = small_config(name="many_prep", layers=2, kv_heads=2, windows=((48, 200), (300, 16)),
                       prefill=tuple((i * 53) % 700 for i in range(300)), steps=3)
    run = Run(cfg, fused=True)
    run.materialize()
    res = run.run_prepared(keep_steps=range(cfg.steps), keep_layers=range(cfg.layers))
    assert run.device_errors() == 0
    for (i, l), (q_raw, got) in sorted(res.items()):
        assert_close(got, run.reference(i, l, q_raw), cfg, f"step {i} layer {l}")
    _check_all_pool_blocks(run)
    run.close()
