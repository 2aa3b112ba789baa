"""Pins of the oracle's pool model (geometry, block tables, ring placement) against
hand-derived fixtures and closed forms.  CPU only."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_block_tables_match_hand_derived_fixture():
    g = _load("block_tables.json")
    w = np.asarray(g["windows"])
    assert oracle.blocks_per_head(w, g["block_size"]).tolist() == g["nblk"]
    tables = oracle.block_tables(w, g["num_seqs"], g["block_size"])
    assert len(tables) == len(g["tables"])
    for t in g["tables"]:
        assert tables[(t["layer"], t["seq"], t["head"])] == t["ids"]
    assert oracle.total_blocks(w, g["num_seqs"], g["block_size"]) == g["total_blocks"]
    assert oracle.pool_bytes(w, g["num_seqs"], g["head_dim"], g["block_size"], g["elem_bytes"]) == g["pool_bytes"]


def test_example_policy_pool_bytes():
    g = _load("example_policy.json")
    bs = g["block_size"]
    assert oracle.blocks_per_head([g["layer0_windows"]], bs)[0].tolist() == g["layer0_nblk"]
    assert oracle.blocks_per_head([g["layer1_windows"]], bs)[0].tolist() == g["layer1_nblk"]
    assert int(oracle.ring_capacity([g["layer0_windows"]], bs).sum()) == g["tokens_per_seq_layer0"]
    assert int(oracle.ring_capacity([g["layer1_windows"]], bs).sum()) == g["tokens_per_seq_layer1"]
    w = np.asarray([g["layer0_windows"] if l % 2 == 0 else g["layer1_windows"] for l in range(48)])
    assert oracle.pool_bytes(w, 1, 128, bs, 2) == g["pool_bytes_per_seq"]
    assert oracle.pool_bytes(w, g["num_seqs"], 128, bs, 2) == g["pool_bytes"]
    t = g["tiny_case"]
    assert oracle.pool_bytes(np.asarray(t["windows"]), t["num_seqs"], t["head_dim"], t["block_size"],
                             t["elem_bytes"]) == t["pool_bytes"]


def test_workload_policy_rows_are_the_printed_example():
    import workloads
    g = _load("example_policy.json")
    cfg = workloads.config("full")
    w = cfg.windows_array()
    assert w.shape == (48, 8)
    assert w[0].tolist() == g["layer0_windows"] and w[1].tolist() == g["layer1_windows"]
    assert all(w[l].tolist() == w[l % 2].tolist() for l in range(48))


@pytest.mark.parametrize("case", _load("ring_placement.json")["cases"], ids=lambda c: c["name"])
def test_ring_placement_fixture(case):
    w, bs, L, n = case["window"], case["block_size"], case["prefill"], case["appends"]
    C = int(oracle.ring_capacity([[w]], bs)[0, 0])
    hist = (np.arange(L + n, dtype=np.float32) + 1).reshape(-1, 1)
    writes = list(oracle.materialized_positions(L, w)) + list(oracle.appended_positions(L, n))
    rk, rv = oracle.ring_after_writes(hist, -hist, 0, writes, C)
    assert rk[:, 0].tolist() == case["ring"]
    assert (-rv[:, 0]).tolist() == case["ring"]
    blocks = oracle.ring_to_blocks(rk, rv, bs)
    assert blocks[:, 0, :, 0].tolist() == case["blocks"]
    lo, hi = oracle.window_span(case["attention_len"], w)
    assert list(range(lo, hi)) == case["attention_positions"]
    assert [p % C for p in range(lo, hi)] == case["attention_slots"]


@pytest.mark.parametrize("seed", range(6))
def test_block_table_is_a_bijection_with_ceil_counts(seed):
    rng = np.random.default_rng(seed)
    layers, heads, seqs, bs = rng.integers(1, 4), rng.integers(1, 5), rng.integers(1, 4), int(rng.choice([1, 4, 16]))
    w = rng.integers(1, 70, size=(layers, heads))
    tables = oracle.block_tables(w, seqs, bs)
    ids = sorted(i for t in tables.values() for i in t)
    assert ids == list(range(oracle.total_blocks(w, seqs, bs)))
    for (l, s, h), t in tables.items():
        assert len(t) * bs >= w[l, h] > (len(t) - 1) * bs


@pytest.mark.parametrize("seed", range(8))
def test_ring_holds_exactly_the_resident_positions(seed):
    """After materialise + appends, each position of the last min(C, written) positions is
    found at slot p mod C, and each slot holds the newest position congruent to it."""
    rng = np.random.default_rng(100 + seed)
    bs = int(rng.choice([2, 4, 16]))
    w = int(rng.integers(1, 60))
    L = int(rng.integers(0, 130))
    n = int(rng.integers(0, 40))
    D = 3
    C = int(oracle.ring_capacity([[w]], bs)[0, 0])
    hist = rng.standard_normal((L + n, D)).astype(np.float32)
    writes = list(oracle.materialized_positions(L, w)) + list(oracle.appended_positions(L, n))
    rk, _ = oracle.ring_after_writes(hist, hist, 0, writes, C)
    written = set(writes)
    for t in range(C):
        owners = [p for p in written if p % C == t]
        if owners:
            assert np.array_equal(rk[t], hist[max(owners)])
        else:
            assert not rk[t].any()
    # every position attention needs is still resident
    lo, hi = oracle.window_span(L + n, w)
    for p in range(lo, hi):
        if p in written:
            assert np.array_equal(rk[p % C], hist[p])


def test_expected_pool_places_rings_through_the_table():
    w = np.array([[5, 16], [1, 9]])
    seqs, bs, D = 2, 4, 2
    rng = np.random.default_rng(7)
    lens = [7, 13]
    n = 3
    hist = {(l, s, h): rng.standard_normal((lens[s] + n, D)).astype(np.float32)
            for l in range(2) for s in range(seqs) for h in range(2)}

    def history_fn(l, s, h, lo, hi):
        return hist[(l, s, h)][lo:hi], -hist[(l, s, h)][lo:hi]

    pool = oracle.expected_pool(w, seqs, bs, D, np.float32, history_fn, lens, n)
    assert pool.shape == (20, 2, bs, D)
    tables = oracle.block_tables(w, seqs, bs)
    # layer 1, seq 1, head 0: window 1 -> one block, C = 4; materialise writes position 12
    # (slot 0), the appends write 13, 14, 15 (slots 1, 2, 3)
    b = tables[(1, 1, 0)][0]
    for t in range(4):
        assert np.array_equal(pool[b, 0, t], hist[(1, 1, 0)][12 + t])
        assert np.array_equal(pool[b, 1, t], -hist[(1, 1, 0)][12 + t])
    # layer 0, seq 0, head 1: window 16 covers all 10 positions, slots 0..9 in order
    ids = tables[(0, 0, 1)]
    ring = np.concatenate([pool[i, 0] for i in ids])
    assert np.array_equal(ring[:10], hist[(0, 0, 1)][:10]) and not ring[10:].any()
    ringv = np.concatenate([pool[i, 1] for i in ids])
    assert np.array_equal(ringv[:10], -hist[(0, 0, 1)][:10])
