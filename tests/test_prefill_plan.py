"""The chunked-prefill launch plan (host only, no GPU): every split key stream is covered.

hwkv_prefill_plan returns, per launch position, the KV head, its CTAs per (sequence, query-tile
pair) and the 64-key stages each CTA streams.  The kernel streams, for the tile pair starting at
chunk row qa, the 16-token ring tiles holding prior positions [lo, p0) (lo = max(0, p0 + qa + 1 - w))
and then the 16-row chunk tiles [clo, qb) (clo = max(0, qa + 1 - w), qb = min(n, qa + 2 * 128 / G)),
four tiles per stage.  CTA k of a split stream takes stages [k * split_stages, (k + 1) *
split_stages), so splits * split_stages must reach the stage count for every pair, sequence
position and chunk length; a plan short of it would drop keys.  The stage count below restates
that enumeration from the windowed-attention definition, independently of the library."""
import numpy as np
import pytest

import head_budgeted_kv_gb300 as hw

PF_M = 128  # query rows per tile


def stream_stages(w: int, C: int, G: int, p0: int, n: int, qa: int) -> int:
    """64-key stages of the key stream of the tile pair at chunk row qa (0 when it has no row)."""
    qb = min(n, qa + 2 * (PF_M // G))
    if qa >= qb:
        return 0
    lo = max(0, p0 + qa + 1 - w)
    need = p0 - lo  # prior positions visible to the pair's first query
    prior = 0
    if need > 0:
        first = lo % C
        prior = min(C // 16, (first + need - 1) // 16 - first // 16 + 1)
    clo = max(0, qa + 1 - w)
    chunk = (qb - 1) // 16 - clo // 16 + 1
    return -(-(prior + chunk) // 4)


def check_plan(windows, layer, num_seqs, block_size, head_dim, G, n_max, sms, max_stages, positions, rng):
    L, H = windows.shape
    order, splits, stages, ws = hw.hwkv_prefill_plan(L, H, head_dim, block_size, windows, num_seqs, layer, H * G,
                                                     n_max, sms, max_stages)
    assert sorted(order.tolist()) == list(range(H))
    assert ((splits >= 1) & (splits <= 64)).all()
    assert (stages >= 1).all()
    pairs = -(-n_max // (2 * (PF_M // G)))
    ctas = num_seqs * pairs * int(splits.sum())
    assert ws == (ctas * 2 * 128 * (head_dim + 2) * 4 if (splits > 1).any() else 0)
    if max_stages > 0:  # the configured cap holds wherever the split count is not at its limit
        assert (stages[splits < 64] <= max_stages).all()
    for i, h in enumerate(order.tolist()):
        w = int(windows[layer, h])
        C = -(-w // block_size) * block_size
        cover = int(splits[i]) * int(stages[i])
        for p0 in positions(w, C):
            for n in (n_max, int(rng.integers(1, n_max + 1))):
                for qt in range(pairs):
                    need = stream_stages(w, C, G, p0, n, qt * 2 * (PF_M // G))
                    assert need <= cover, (f"head {h} (w {w}, C {C}) p0 {p0} n {n} pair {qt}: {need} stages, "
                                           f"plan covers {splits[i]} x {stages[i]}")


def _positions(rng):
    def f(w, C):
        return sorted({0, 1, max(0, w - 1), w, C, C + 1, 2 * C + 7, int(rng.integers(0, 3 * C + 50))})
    return f


@pytest.mark.parametrize("seed", range(40))
def test_random_plans_cover_every_stream(seed):
    rng = np.random.default_rng(7000 + seed)
    H = int(rng.choice([1, 2, 3, 8, 16]))
    L = 2
    block_size = int(rng.choice([16, 32, 64, 128]))
    windows = rng.choice([16, 40, 100, 1000, 1024, 4096, 5000, 16384, 65536], size=(L, H)).astype(np.int32)
    G = int(rng.choice([1, 2, 3, 4, 8, 16]))
    num_seqs = int(rng.choice([1, 2, 4, 9]))
    n_max = int(rng.choice([1, 17, 64, 300, 2048]))
    sms = int(rng.choice([1, 20, 152]))
    max_stages = int(rng.choice([0, 0, 1, 3, 40]))
    head_dim = int(rng.choice([64, 128]))
    check_plan(windows, int(rng.integers(L)), num_seqs, block_size, head_dim, G, n_max, sms, max_stages,
               _positions(rng), rng)


def test_long_context_plans_cover_every_stream():
    """The 161K batch-1 geometry (windows from the level set), where the automatic plan splits
    64K-window streams and refines the split counts per head."""
    rng = np.random.default_rng(11)
    windows = rng.choice([1024, 4096, 16384, 65536], size=(4, 8)).astype(np.int32)
    windows[0] = [1024, 1024, 16384, 65536, 16384, 1024, 16384, 16384]
    for layer in range(4):
        order, splits, stages, ws = hw.hwkv_prefill_plan(4, 8, 128, 16, windows, 1, layer, 32, 2048, 152, 0)
        assert ws > 0 and splits.max() > 1  # long streams are split at batch 1
        # longest CTAs launch first
        assert all(stages[i] >= stages[i + 1] for i in range(7))
        check_plan(windows, layer, 1, 16, 128, 4, 2048, 152, 0,
                   lambda w, C: [164864, 164864 + 2048 * 3, int(rng.integers(0, 3 * C))], rng)


def test_plan_is_deterministic_and_matches_the_cap_rule():
    windows = np.array([[65536, 1024, 16384, 4096]], dtype=np.int32)
    a = hw.hwkv_prefill_plan(1, 4, 128, 16, windows, 1, 0, 16, 2048, 152, 0)
    b = hw.hwkv_prefill_plan(1, 4, 128, 16, windows, 1, 0, 16, 2048, 152, 0)
    assert all(np.array_equal(x, y) for x, y in zip(a[:3], b[:3])) and a[3] == b[3]
    # with an explicit cap every head is split to at most that many stages, by decreasing window
    order, splits, stages, _ = hw.hwkv_prefill_plan(1, 4, 128, 16, windows, 1, 0, 16, 2048, 152, 100)
    assert order.tolist() == [0, 2, 3, 1]
    assert (stages <= 100).all()
    # many sequences: enough CTAs that nothing is split
    _, splits, _, ws = hw.hwkv_prefill_plan(1, 4, 128, 16, windows, 64, 0, 16, 2048, 152, 0)
    assert (splits == 1).all() and ws == 0


def test_plan_rejects_bad_arguments():
    windows = np.array([[64, 64]], dtype=np.int32)
    for kw, status in ((dict(block_size=8), hw.binding.HWKV_ERR_UNSUPPORTED),
                       (dict(layer=1), hw.binding.HWKV_ERR_INVALID_ARG),
                       (dict(q_heads=3), hw.binding.HWKV_ERR_UNSUPPORTED),
                       (dict(n_max=0), hw.binding.HWKV_ERR_INVALID_ARG),
                       (dict(num_sms=0), hw.binding.HWKV_ERR_INVALID_ARG),
                       (dict(max_stages=-1), hw.binding.HWKV_ERR_INVALID_ARG)):
        args = dict(layers=1, kv_heads=2, head_dim=128, block_size=16, windows=windows, num_seqs=1, layer=0, q_heads=8,
                    n_max=10, num_sms=152, max_stages=0)
        args.update(kw)
        with pytest.raises(hw.HwkvError) as e:
            hw.hwkv_prefill_plan(**args)
        assert e.value.status == status
