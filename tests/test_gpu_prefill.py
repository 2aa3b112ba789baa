"""Chunked prefill (hwkv_prefill_attn) against the oracle: every new token's output is the
windowed attention over the full history, the rings afterwards hold what appending the tokens
one by one would leave (bit for bit), and decoding continues correctly from there."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import head_budgeted_kv_gb300 as hw
from harness import assert_close, oracle_table, small_config

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hw.binding.load()
    yield
    torch.cuda.synchronize()


def _raw(t):
    return workloads.to_raw(t)


class History:
    """Host copy of every token of every (layer, seq, kv head), in position order."""

    def __init__(self, cfg):
        self.cfg = cfg
        self.k = {}
        self.v = {}

    def add(self, l, s, h, k_rows, v_rows):
        key = (l, s, h)
        self.k[key] = np.concatenate([self.k[key], k_rows]) if key in self.k else k_rows
        self.v[key] = np.concatenate([self.v[key], v_rows]) if key in self.v else v_rows

    def span(self, l, s, h, lo, hi):
        return lo, self.k[(l, s, h)][lo:hi], self.v[(l, s, h)][lo:hi]


def _run(cfg, chunks, seed_decode_steps=2, check_every_token=True, max_stages=0):
    """Materialise cfg.prefill, then prefill the given chunk lengths [[n_s per seq] per chunk],
    then decode a few steps; compare everything with the oracle.  max_stages > 0 splits every
    key stream longer than that many 64-key stages over several CTAs."""
    dev = torch.device("cuda")
    wl = workloads.Workload(cfg, device=dev)
    pool = hw.Pool(cfg.layers, cfg.kv_heads, cfg.head_dim, cfg.block_size, cfg.windows_array(), cfg.batch,
                   torch.bfloat16, q_heads=cfg.q_heads)
    pool.set_prefill_config(max_stages)
    hist = History(cfg)
    lens = np.asarray(cfg.prefill, dtype=np.int64)
    pre = torch.tensor(cfg.prefill, dtype=torch.int32, device=dev)
    for l in range(cfg.layers):
        K, V = wl.prefill_layer(l, dev)
        pool.materialize(l, K, V, pre)
        for s in range(cfg.batch):
            for h in range(cfg.kv_heads):
                hist.add(l, s, h, _raw(K[s, h, :lens[s]]), _raw(V[s, h, :lens[s]]))
    writes = {(l, s, h): list(oracle.materialized_positions(int(lens[s]), int(cfg.windows[l][h])))
              for l in range(cfg.layers) for s in range(cfg.batch) for h in range(cfg.kv_heads)}
    for ci, ns in enumerate(chunks):
        n_max = max(max(ns), 1)
        pos = torch.tensor(lens, dtype=torch.int32, device=dev)
        nt = torch.tensor(ns, dtype=torch.int32, device=dev)
        for l in range(cfg.layers):
            q, k, v = wl.chunk_inputs(l, ci, n_max, dev)
            out = torch.full_like(q, 3.0)
            pool.prefill(l, q, cfg.scale, k, v, pos, nt, out=out)
            torch.cuda.synchronize()
            got = out.float().cpu().double().numpy()
            for s in range(cfg.batch):
                n = ns[s]
                for h in range(cfg.kv_heads):
                    hist.add(l, s, h, _raw(k[s, :n, h]), _raw(v[s, :n, h]))
                    writes[(l, s, h)] += list(range(int(lens[s]), int(lens[s]) + n))
                if n == 0:
                    assert (got[s] == 3.0).all()  # untouched
                    continue
                spans = {}
                for h in range(cfg.kv_heads):
                    lo = max(0, int(lens[s]) + 1 - int(cfg.windows[l][h]))
                    spans[h] = hist.span(l, s, h, lo, int(lens[s]) + n)
                ref = oracle.prefill_attention(_raw(q[s, :n]), spans, int(lens[s]), cfg.windows[l], cfg.scale)
                assert_close(got[s, :n], ref, cfg, f"chunk {ci} layer {l} seq {s}")
                assert (got[s, n:] == 3.0).all()
        lens = lens + np.asarray(ns)
    # the rings hold exactly what the write sequence leaves
    blocks = pool.blocks()
    for (l, s, h), ids in oracle_table(cfg).items():
        w = int(cfg.windows[l][h])
        C = int(oracle.ring_capacity([[w]], cfg.block_size)[0, 0])
        wr = writes[(l, s, h)]
        if wr:
            p_lo = wr[0]
            rk, rv = oracle.ring_after_writes(hist.k[(l, s, h)][p_lo:], hist.v[(l, s, h)][p_lo:], p_lo, wr, C)
        else:
            rk = rv = np.zeros((C, cfg.head_dim), np.uint16)
        exp = oracle.ring_to_blocks(rk, rv, cfg.block_size)
        got = _raw(blocks[torch.as_tensor(ids, device=dev)])
        assert np.array_equal(got, exp), f"ring of layer {l} seq {s} head {h}"
    # decoding continues from the prefilled rings
    for step in range(seed_decode_steps):
        q, kn, vn = wl.step_inputs(100 + step, dev)
        pos = torch.tensor(lens, dtype=torch.int32, device=dev)
        for l in range(cfg.layers):
            out = pool.append_decode(l, q[l], cfg.scale, kn[l], vn[l], pos)
            torch.cuda.synchronize()
            for s in range(cfg.batch):
                for h in range(cfg.kv_heads):
                    hist.add(l, s, h, _raw(kn[l, s, h][None]), _raw(vn[l, s, h][None]))
            got = out.float().cpu().double().numpy()
            spans = {}
            for s in range(cfg.batch):
                for h in range(cfg.kv_heads):
                    L = int(lens[s]) + 1
                    lo = max(0, L - int(cfg.windows[l][h]))
                    spans[(s, h)] = hist.span(l, s, h, lo, L)
            ref = oracle.attention_jobs(_raw(q[l]), spans, [int(x) + 1 for x in lens], cfg.windows[l], cfg.scale)
            assert_close(got, ref, cfg, f"decode after prefill, layer {l}")
        lens = lens + 1
    assert pool.check_device_errors() == 0
    pool.close()


CASES = {
    # first chunk at p0 = 0, then a second one on top of it; C > w for the first head
    "from_empty": dict(kv_heads=2, windows=((40, 200),), prefill=(0, 0), chunks=[[37, 70], [50, 3]]),
    # prior context in the ring, chunk longer than the window and than the ring
    "long_chunk": dict(kv_heads=2, windows=((32, 96),), prefill=(300, 45), chunks=[[130, 64]]),
    # ragged chunk lengths with an empty one, several layers
    "ragged": dict(layers=2, kv_heads=3, windows=((64, 1024, 16), (256, 48, 500)), prefill=(700, 20, 130),
                   chunks=[[33, 0, 90]]),
    "g1_d64": dict(kv_heads=2, group=1, head_dim=64, windows=((128, 64),), prefill=(200, 10), chunks=[[75, 130]]),
    "g2": dict(kv_heads=2, group=2, windows=((1000, 160),), prefill=(1500, 300), chunks=[[40, 21]]),
    "g8": dict(kv_heads=1, group=8, windows=((256,),), prefill=(400, 5), chunks=[[20, 17]]),
    # group 16: four tokens per 64-row tile; groups 3 and 12 leave idle rows (21 and 5 tokens)
    "g16": dict(kv_heads=2, group=16, windows=((96, 512),), prefill=(600, 7), chunks=[[45, 9]]),
    "g3": dict(kv_heads=2, group=3, windows=((80, 300),), prefill=(350, 0), chunks=[[50, 64]]),
    "g12_d64": dict(kv_heads=1, group=12, head_dim=64, windows=((200,),), prefill=(260, 33), chunks=[[23, 18]]),
    "bs64": dict(kv_heads=2, block_size=64, windows=((128, 1000),), prefill=(900, 64), chunks=[[77, 129]]),
    # long key streams (about 130 stages of 64 keys per CTA), so the kernel's pipeline barriers
    # run through many phases
    "deep": dict(kv_heads=2, windows=((8192, 2048),), prefill=(9000, 2100), chunks=[[160, 70]]),
    # block sizes 32 and 128: whole-stage pool copies of two blocks x 32 rows and of 64 rows
    # inside one block (at several row offsets), plus the per-tile fallback where they do not fit
    "bs32": dict(kv_heads=2, block_size=32, windows=((200, 1000),), prefill=(700, 50), chunks=[[90, 40]]),
    "bs128": dict(kv_heads=2, block_size=128, windows=((256, 2048),), prefill=(3000, 129), chunks=[[100, 300]]),
    # key streams split over several CTAs and merged (forced by a small stage cap): long and
    # short streams, empty splits past short contexts, a zero-length chunk, group 16, two layers
    "split_deep": dict(kv_heads=2, windows=((8192, 2048),), prefill=(9000, 2100), chunks=[[160, 70]], max_stages=9),
    "split_ragged": dict(layers=2, kv_heads=3, windows=((64, 1024, 16), (256, 48, 500)), prefill=(700, 20, 130),
                         chunks=[[33, 0, 90]], max_stages=2),
    "split_g16": dict(kv_heads=2, group=16, windows=((900, 512),), prefill=(600, 7), chunks=[[45, 9]], max_stages=3),
    # 64 and 33 splits of one stream: the combine's lanes hold splits i and i + 32
    "split_wide": dict(kv_heads=2, windows=((4096, 2000),), prefill=(4500, 3000), chunks=[[50, 17]], max_stages=1),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_against_oracle(name):
    spec = dict(CASES[name])
    chunks = spec.pop("chunks")
    max_stages = spec.pop("max_stages", 0)
    cfg = small_config(name=name, cfg_id=91, steps=2, **spec)
    _run(cfg, chunks, max_stages=max_stages)


def test_split_streams_change_rounding_only():
    """The same chunk with and without the split of its key streams: outputs within rounding,
    rings bit-identical."""
    cfg = small_config(name="splitcmp", cfg_id=94, kv_heads=2, windows=((4096, 300),), prefill=(5000, 40))
    dev = torch.device("cuda")
    wl = workloads.Workload(cfg, device=dev)
    pre = torch.tensor(cfg.prefill, dtype=torch.int32, device=dev)
    K, V = wl.prefill_layer(0, dev)
    q, k, v = wl.chunk_inputs(0, 0, 200, dev)
    nt = torch.tensor([200, 130], dtype=torch.int32, device=dev)
    outs, pools = [], []
    for cap in (0, 4):
        pool = hw.Pool(1, 2, 128, 16, cfg.windows_array(), 2, torch.bfloat16, q_heads=cfg.q_heads)
        pool.set_prefill_config(cap)
        pool.materialize(0, K, V, pre)
        outs.append(pool.prefill(0, q, cfg.scale, k, v, pre, nt))
        pools.append(pool)
    torch.cuda.synchronize()
    assert hw.hwkv_prefill_workspace_bytes(pools[1].handle, 0, cfg.q_heads, 200) > 0
    for s, n in enumerate((200, 130)):
        assert_close(outs[1][s, :n].float().cpu().double().numpy(), outs[0][s, :n].float().cpu().double().numpy(),
                     cfg, f"seq {s}")
    assert torch.equal(pools[0].buffer, pools[1].buffer)
    for p in pools:
        assert p.check_device_errors() == 0
        p.close()


def test_prefill_equals_token_by_token_decode():
    """Prefilling a chunk leaves the same rings as appending its tokens one by one."""
    cfg = small_config(name="tbt", cfg_id=92, kv_heads=2, windows=((48, 160),), prefill=(100, 30))
    dev = torch.device("cuda")
    wl = workloads.Workload(cfg, device=dev)
    pools = [hw.Pool(1, 2, 128, 16, cfg.windows_array(), 2, torch.bfloat16, q_heads=8) for _ in range(2)]
    pre = torch.tensor(cfg.prefill, dtype=torch.int32, device=dev)
    K, V = wl.prefill_layer(0, dev)
    for p in pools:
        p.materialize(0, K, V, pre)
    n = 60
    q, k, v = wl.chunk_inputs(0, 0, n, dev)
    out = pools[0].prefill(0, q, cfg.scale, k, v, pre, torch.full((2,), n, dtype=torch.int32, device=dev))
    for i in range(n):
        o = pools[1].append_decode(0, q[:, i].contiguous(), cfg.scale, k[:, i].contiguous(), v[:, i].contiguous(),
                                   pre + i)
        assert_close(out[:, i].float().cpu().double().numpy(), o.float().cpu().double().numpy(), cfg, f"token {i}")
    torch.cuda.synchronize()
    assert torch.equal(pools[0].buffer, pools[1].buffer)
    for p in pools:
        assert p.check_device_errors() == 0
        p.close()


def test_prefill_rejects_unsupported_shapes():
    cfg = small_config(name="rej", cfg_id=93, kv_heads=2, group=3, windows=((64, 64),), prefill=(10,))
    pool = hw.Pool(1, 2, 128, 16, cfg.windows_array(), 1, torch.bfloat16, q_heads=6)
    q = torch.zeros(1, 4, 34, 128, dtype=torch.bfloat16, device="cuda")  # group 17
    k = torch.zeros(1, 4, 2, 128, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(hw.HwkvError) as e:
        pool.prefill(0, q, 0.1, k, k, pos, pos)
    assert e.value.status == hw.binding.HWKV_ERR_UNSUPPORTED
    pool.close()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["full", "long"])
def test_prefill_full_size_sampled(name):
    """One layer of the full-size geometry in the configuration bench.py's prefill mode times
    (a chunk of 2048 tokens per sequence on top of the context): sampled tokens of every
    sequence, all query heads, against the oracle; device error word clear."""
    cfg = workloads.config(name).with_layers(1)
    dev = torch.device("cuda")
    wl = workloads.Workload(cfg, device=dev)
    pool = hw.Pool(cfg.layers, cfg.kv_heads, cfg.head_dim, cfg.block_size, cfg.windows_array(), cfg.batch,
                   torch.bfloat16, q_heads=cfg.q_heads)
    pre = torch.tensor(cfg.prefill, dtype=torch.int32, device=dev)
    K, V = wl.prefill_layer(0, dev)
    pool.materialize(0, K, V, pre)
    n = 2048
    q, k, v = wl.chunk_inputs(0, 0, n, dev)
    out = pool.prefill(0, q, cfg.scale, k, v, pre, torch.full((cfg.batch,), n, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    assert pool.check_device_errors() == 0
    toks = [0, 1, 63, 64, 127, 1000, 2047]
    for s in range(cfg.batch):
        L = int(cfg.prefill[s])
        for t in toks:
            p = L + t
            spans = {}
            for h in range(cfg.kv_heads):
                lo = max(0, p + 1 - int(cfg.windows[0][h]))  # first position of the window
                c0 = max(0, lo - L)                           # first chunk row in it
                kh = np.concatenate([_raw(K[s, h, lo:L]), _raw(k[s, c0:t + 1, h])])
                vh = np.concatenate([_raw(V[s, h, lo:L]), _raw(v[s, c0:t + 1, h])])
                spans[(0, h)] = (lo, kh, vh)
            ref = oracle.attention_jobs(_raw(q[s, t])[None], spans, [p + 1], cfg.windows[0], cfg.scale)[0]
            got = out[s, t].float().cpu().double().numpy()
            assert_close(got, ref, cfg, f"{name} seq {s} token {t}")
    pool.close()


@pytest.mark.parametrize("block_size", [16, 64])
def test_prefill_block_permutation_leaves_output_bit_identical(block_size):
    """The same chunk through an identity and a permuted block table (blocks moved with it):
    outputs bit-identical, rings equal after moving back.  With permuted ids a stage's ring tiles
    are no longer consecutive blocks, so the kernel copies tile by tile instead of per stage."""
    cfg = small_config(name="pfperm", cfg_id=95, kv_heads=2, block_size=block_size, windows=((1024, 192),),
                       prefill=(1500, 300))
    dev = torch.device("cuda")
    wl = workloads.Workload(cfg, device=dev)
    pre = torch.tensor(cfg.prefill, dtype=torch.int32, device=dev)
    K, V = wl.prefill_layer(0, dev)
    q, k, v = wl.chunk_inputs(0, 0, 150, dev)
    nt = torch.tensor([150, 97], dtype=torch.int32, device=dev)
    pools = [hw.Pool(1, 2, 128, block_size, cfg.windows_array(), 2, torch.bfloat16, q_heads=cfg.q_heads)
             for _ in range(2)]
    for p in pools:
        p.materialize(0, K, V, pre)
    _, total, _ = pools[1].geometry()
    perm = np.random.default_rng(1).permutation(total).astype(np.int32)
    blocks = pools[1].blocks()
    moved = torch.empty_like(blocks)
    moved[torch.as_tensor(perm, device=dev).long()] = blocks
    blocks.copy_(moved)
    pools[1].set_block_table(perm)
    outs = [p.prefill(0, q, cfg.scale, k, v, pre, nt) for p in pools]
    torch.cuda.synchronize()
    for s, n in enumerate((150, 97)):
        assert torch.equal(outs[0][s, :n], outs[1][s, :n]), f"seq {s}"
    back = pools[1].blocks()[torch.as_tensor(perm, device=dev).long()]
    assert torch.equal(back, pools[0].blocks())
    for p in pools:
        assert p.check_device_errors() == 0
        p.close()


def _random_prefill_case(seed: int):
    """A seeded random chunked-prefill geometry: GQA group, head_dim, block size, per-head
    windows (some odd, some beyond the context), context from empty to a few thousand tokens,
    one or two ragged chunks (some empty), and a forced split of long key streams in some."""
    rng = np.random.default_rng(2000 + seed)
    kv_heads = int(rng.integers(1, 4))
    group = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16]))
    head_dim = int(rng.choice([64, 128]))
    block_size = int(rng.choice([16, 32, 64, 128]))
    layers = int(rng.integers(1, 3))
    batch = int(rng.integers(1, 4))
    windows = tuple(tuple(int(rng.choice([int(rng.integers(1, 130)), 64, 256, 1000, 4096])) for _ in range(kv_heads))
                    for _ in range(layers))
    prefill = tuple(int(rng.choice([0, int(rng.integers(1, 5000))])) for _ in range(batch))
    chunks = [[int(rng.choice([0, int(rng.integers(1, 200))])) for _ in range(batch)]
              for _ in range(int(rng.integers(1, 3)))]
    max_stages = int(rng.choice([0, 0, 2, 5]))
    cfg = small_config(name=f"pf_random{seed}", cfg_id=300 + seed, layers=layers, kv_heads=kv_heads, group=group,
                       head_dim=head_dim, block_size=block_size, windows=windows, prefill=prefill, steps=2)
    return cfg, chunks, max_stages


@pytest.mark.parametrize("seed", range(12))
def test_random_prefill_geometries_match_the_oracle(seed):
    cfg, chunks, max_stages = _random_prefill_case(seed)
    _run(cfg, chunks, max_stages=max_stages)
