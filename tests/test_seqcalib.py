"""SeqCalib greedy (host tool): the oracle against a hand-derived example and invariants,
and the C-ABI implementation against the oracle.  CPU only."""
import json
import os

import numpy as np
import pytest

import oracle
from head_budgeted_kv_gb300 import _build, binding

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "seqcalib.json")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load()


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_layer_cost_is_pool_bytes():
    g = _golden()
    for l, row in enumerate(g["candidates"]):
        for c, w in enumerate(row):
            assert oracle.layer_cost(w, g["num_seqs"], g["head_dim"], g["block_size"], g["elem_bytes"]) == g["costs"][l][c]


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: str(c["budget"]))
def test_oracle_matches_hand_derived_choices(case):
    g = _golden()
    cost = lambda l, w: oracle.layer_cost(w, g["num_seqs"], g["head_dim"], g["block_size"], g["elem_bytes"])
    dist = lambda l, w, chosen: g["distortion"][l][g["candidates"][l].index(w)]
    if case["choice"] is None:
        with pytest.raises(ValueError):
            oracle.seqcalib_greedy(g["candidates"], dist, case["budget"], cost)
        return
    _, picks, total = oracle.seqcalib_greedy(g["candidates"], dist, case["budget"], cost)
    assert picks == case["choice"] and total == case["bytes"]


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: str(c["budget"]))
def test_library_matches_hand_derived_choices(lib, case):
    g = _golden()
    cand = np.asarray(g["candidates"], dtype=np.int32)
    if case["choice"] is None:
        with pytest.raises(binding.HwkvError) as e:
            binding.hwkv_seqcalib(cand, g["distortion"], case["budget"], g["head_dim"], g["block_size"],
                                  g["num_seqs"], binding.HWKV_F32)
        assert e.value.status == binding.HWKV_ERR_BUDGET and "layer 1" in str(e.value)
        return
    w, choice, total = binding.hwkv_seqcalib(cand, g["distortion"], case["budget"], g["head_dim"], g["block_size"],
                                             g["num_seqs"], binding.HWKV_F32)
    assert choice.tolist() == case["choice"] and total == case["bytes"]
    assert w.tolist() == [g["candidates"][l][c] for l, c in enumerate(case["choice"])]


def test_unlimited_budget_picks_each_layers_minimum():
    rng = np.random.default_rng(3)
    cand = rng.choice([1024, 4096, 16384, 65536], size=(5, 4, 8))
    table = rng.random((5, 4))
    cost = lambda l, w: oracle.layer_cost(w, 2, 128, 16, 2)
    dist = lambda l, w, chosen: table[l][[list(x) for x in cand[l]].index(w)]
    _, picks, _ = oracle.seqcalib_greedy(cand.tolist(), dist, 10 ** 15, cost)
    assert picks == [int(np.argmin(table[l])) for l in range(5)]


def test_distortion_sees_the_lower_layers_choices():
    cand = [[[16, 32], [64, 64]], [[16, 32], [64, 64]], [[16, 32], [64, 64]]]
    seen = []

    def dist(layer, w, chosen):
        seen.append((layer, [list(c) for c in chosen]))
        # prefer to alternate with the layer below
        return 0.0 if (not chosen or chosen[-1] != w) else 1.0

    cost = lambda l, w: oracle.layer_cost(w, 1, 64, 16, 4)
    pol, picks, _ = oracle.seqcalib_greedy(cand, dist, 10 ** 9, cost)
    assert picks == [0, 1, 0]
    assert all(len(ch) == layer for layer, ch in seen)


@pytest.mark.parametrize("seed", range(12))
def test_library_matches_oracle_on_random_problems(lib, seed):
    rng = np.random.default_rng(seed)
    L, C, H = int(rng.integers(1, 7)), int(rng.integers(1, 5)), int(rng.integers(1, 9))
    bs, D, B, dt = int(rng.choice([16, 64])), int(rng.choice([64, 128])), int(rng.integers(1, 5)), int(rng.integers(0, 2))
    eb = 4 if dt == 0 else 2
    cand = rng.choice([1024, 4096, 16384, 65536, 100, 7], size=(L, C, H)).astype(np.int32)
    weights = rng.random(H)

    def dist(layer, w, chosen):  # depends on the layer below: rewards windows above it
        below = np.asarray(chosen[-1]) if len(chosen) else np.zeros(H)
        return float(np.dot(weights, 1.0 / np.asarray(w, dtype=float)) - 1e-6 * np.sum(np.asarray(w) > below))

    cost = lambda l, w: oracle.layer_cost(w, B, D, bs, eb)
    budget = int(sum(min(cost(l, list(c)) for c in cand[l]) for l in range(L)) * rng.uniform(0.9, 3.0))
    try:
        ref = oracle.seqcalib_greedy(cand.tolist(), dist, budget, cost)
    except ValueError:
        ref = None
    if ref is None:
        with pytest.raises(binding.HwkvError) as e:
            binding.hwkv_seqcalib(cand, dist, budget, D, bs, B, dt)
        assert e.value.status == binding.HWKV_ERR_BUDGET
        return
    w, choice, total = binding.hwkv_seqcalib(cand, dist, budget, D, bs, B, dt)
    assert choice.tolist() == ref[1] and total == ref[2] and w.tolist() == ref[0]
    assert total == oracle.pool_bytes(w, B, D, bs, eb) <= budget
