"""Pins of the oracle's fp64 windowed attention.  CPU only.

The oracle is checked against torch's scaled_dot_product_attention (an independent
library routine) with an explicit boolean window mask and GQA expansion, and against
closed forms: a one-token window returns that token's value exactly, constant keys give
the mean of the resident values, two tokens give a logistic weighting.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _sdpa_masked(q, K, V, lens, windows, scale):
    """torch SDPA in fp64 with a boolean mask keeping positions [len - w, len)."""
    B, Hq, D = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for s in range(B):
        Lfull = K.shape[2]
        qq = torch.from_numpy(q[s]).double()[None, :, None, :]               # [1, Hq, 1, D]
        kk = torch.from_numpy(K[s]).double().repeat_interleave(G, dim=0)[None]  # [1, Hq, L, D]
        vv = torch.from_numpy(V[s]).double().repeat_interleave(G, dim=0)[None]
        mask = torch.zeros((1, Hq, 1, Lfull), dtype=torch.bool)
        for qh in range(Hq):
            w = int(windows[qh // G])
            mask[0, qh, 0, max(0, lens[s] - w):lens[s]] = True
        o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
        out[s] = o[0, :, 0, :].numpy()
    return out


def _run_oracle(q, K, V, lens, windows, scale, threads=2, p_lo=None):
    B, Hkv = K.shape[:2]
    hist = {}
    for s in range(B):
        for h in range(Hkv):
            lo = 0 if p_lo is None else p_lo[s][h]
            hist[(s, h)] = (lo, K[s, h, lo:lens[s]], V[s, h, lo:lens[s]])
    return oracle.attention_jobs(q, hist, lens, windows, scale, threads=threads)


@pytest.mark.parametrize("seed", range(6))
def test_windowed_attention_matches_masked_sdpa(seed):
    rng = np.random.default_rng(seed)
    B, Hkv, G, D = 2, 3, int(rng.choice([1, 2, 4])), int(rng.choice([8, 16, 64]))
    L = 50
    K = rng.standard_normal((B, Hkv, L, D)).astype(np.float32)
    V = rng.standard_normal((B, Hkv, L, D)).astype(np.float32)
    q = rng.standard_normal((B, Hkv * G, D)).astype(np.float32)
    lens = [int(rng.integers(1, L + 1)) for _ in range(B)]
    windows = [int(x) for x in rng.choice([1, 3, 17, 49, 50, 1000], size=Hkv)]
    scale = 1 / math.sqrt(D)
    got = _run_oracle(q, K, V, lens, windows, scale)
    ref = _sdpa_masked(q, K, V, lens, windows, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_full_window_is_plain_attention():
    """w >= len: the windowed result is full (unmasked) attention."""
    rng = np.random.default_rng(11)
    B, Hkv, G, D, L = 1, 2, 4, 32, 40
    K = rng.standard_normal((B, Hkv, L, D)).astype(np.float32)
    V = rng.standard_normal((B, Hkv, L, D)).astype(np.float32)
    q = rng.standard_normal((B, Hkv * G, D)).astype(np.float32)
    got = _run_oracle(q, K, V, [L], [L, 10 * L], 0.125)
    qq = torch.from_numpy(q).double()[:, :, None, :]
    kk = torch.from_numpy(K).double()
    vv = torch.from_numpy(V).double()
    ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=0.125, enable_gqa=True)
    np.testing.assert_allclose(got, ref[:, :, 0, :].numpy(), rtol=1e-12, atol=1e-12)


def test_window_one_returns_last_value_exactly():
    rng = np.random.default_rng(3)
    D = 64
    K = rng.standard_normal((1, 1, 9, D)).astype(np.float32)
    V = rng.standard_normal((1, 1, 9, D)).astype(np.float32)
    q = rng.standard_normal((1, 2, D)).astype(np.float32)
    got = _run_oracle(q, K, V, [9], [1], 0.3)
    assert np.array_equal(got[0, 0], V[0, 0, 8].astype(np.float64))
    assert np.array_equal(got[0, 1], V[0, 0, 8].astype(np.float64))


def test_length_one_returns_first_value_exactly():
    rng = np.random.default_rng(4)
    K = rng.standard_normal((1, 1, 1, 16)).astype(np.float32)
    V = rng.standard_normal((1, 1, 1, 16)).astype(np.float32)
    q = rng.standard_normal((1, 1, 16)).astype(np.float32)
    got = _run_oracle(q, K, V, [1], [4096], 0.25)
    assert np.array_equal(got[0, 0], V[0, 0, 0].astype(np.float64))


def test_constant_keys_give_mean_of_resident_values():
    rng = np.random.default_rng(5)
    L, D, w = 30, 8, 7
    K = np.tile(rng.standard_normal(D).astype(np.float32), (1, 1, L, 1))
    V = rng.standard_normal((1, 1, L, D)).astype(np.float32)
    q = rng.standard_normal((1, 1, D)).astype(np.float32)
    got = _run_oracle(q, K, V, [L], [w], 1.0)
    np.testing.assert_allclose(got[0, 0], V[0, 0, L - w:].astype(np.float64).mean(axis=0), rtol=1e-13, atol=1e-14)


def test_two_tokens_logistic_weights():
    D = 4
    K = np.zeros((1, 1, 5, D), np.float32)
    V = np.zeros((1, 1, 5, D), np.float32)
    K[0, 0, 3] = [1, 0, 0, 0]
    K[0, 0, 4] = [0, 2, 0, 0]
    V[0, 0, 3] = [1, 0, 0, 0]
    V[0, 0, 4] = [0, 1, 0, 0]
    q = np.array([[[0.5, 1.5, 0, 0]]], np.float32)
    got = _run_oracle(q, K, V, [5], [2], 0.5)
    s3, s4 = 0.5 * 0.5, 0.5 * 3.0
    w4 = 1 / (1 + math.exp(s3 - s4))
    np.testing.assert_allclose(got[0, 0], [1 - w4, w4, 0, 0], rtol=1e-15, atol=1e-15)


def test_empty_window_is_zero():
    K = np.ones((1, 1, 4, 8), np.float32)
    q = np.ones((1, 1, 8), np.float32)
    got = _run_oracle(q, K, K, [0], [4], 1.0)
    assert not got.any()


def test_history_tail_equals_full_history_and_uncovered_window_is_rejected():
    rng = np.random.default_rng(8)
    L, D = 80, 16
    K = rng.standard_normal((1, 1, L, D)).astype(np.float32)
    V = rng.standard_normal((1, 1, L, D)).astype(np.float32)
    q = rng.standard_normal((1, 2, D)).astype(np.float32)
    full = _run_oracle(q, K, V, [L], [20], 0.25)
    tail = _run_oracle(q, K, V, [L], [20], 0.25, p_lo=[[60]])
    assert np.array_equal(full, tail)
    with pytest.raises(ValueError):
        _run_oracle(q, K, V, [L], [20], 0.25, p_lo=[[61]])


def test_bf16_bits_are_widened_exactly():
    rng = np.random.default_rng(9)
    L, D = 33, 16
    t = torch.from_numpy(rng.standard_normal((3, L, D)).astype(np.float32)).to(torch.bfloat16)
    raw = t.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.widen(raw), t.double().numpy())
    q = raw[0, :2][None]
    got = _run_oracle(q, raw[1][None, None], raw[2][None, None], [L], [L], 0.25)
    ref = _run_oracle(t[0, :2].double().numpy()[None], t[1].double().numpy()[None, None],
                      t[2].double().numpy()[None, None], [L], [L], 0.25)
    assert np.array_equal(got, ref)


def test_gqa_groups_are_consecutive():
    """Query heads g*G .. g*G+G-1 read kv head g (values of kv head h are all h)."""
    Hkv, G, D, L = 3, 4, 8, 5
    rng = np.random.default_rng(10)
    K = rng.standard_normal((1, Hkv, L, D)).astype(np.float32)
    V = np.zeros((1, Hkv, L, D), np.float32)
    for h in range(Hkv):
        V[0, h] = h
    q = rng.standard_normal((1, Hkv * G, D)).astype(np.float32)
    got = _run_oracle(q, K, V, [L], [L] * Hkv, 0.3)
    for qh in range(Hkv * G):
        np.testing.assert_allclose(got[0, qh], qh // G, rtol=0, atol=1e-15)


def test_thread_count_does_not_change_bits():
    rng = np.random.default_rng(12)
    B, Hkv, G, D, L = 2, 2, 2, 32, 300
    K = rng.standard_normal((B, Hkv, L, D)).astype(np.float32)
    V = rng.standard_normal((B, Hkv, L, D)).astype(np.float32)
    q = rng.standard_normal((B, Hkv * G, D)).astype(np.float32)
    a = _run_oracle(q, K, V, [L, 200], [64, 1000], 0.2, threads=1)
    b = _run_oracle(q, K, V, [L, 200], [64, 1000], 0.2, threads=4)
    assert np.array_equal(a, b)


def test_large_scores_are_stable():
    """Keys scaled x8 (the ragged workload's spikes) must not overflow the softmax."""
    rng = np.random.default_rng(13)
    L, D = 64, 128
    K = (rng.standard_normal((1, 1, L, D)) * 8).astype(np.float32)
    V = rng.standard_normal((1, 1, L, D)).astype(np.float32)
    q = (rng.standard_normal((1, 4, D)) * 8).astype(np.float32)
    got = _run_oracle(q, K, V, [L], [48], 1 / math.sqrt(D))
    ref = _sdpa_masked(q, K, V, [L], [48], 1 / math.sqrt(D))
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-11)
