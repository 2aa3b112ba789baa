"""Pins of the oracle's chunked-prefill attention (``oracle.prefill_attention``).  CPU only.

What a prefill token attends to is read from the HeadWiseKV blog summary, section
"Grouped-Cache Runtime": every KV head keeps only its window of the newest tokens, so the
token at position p sees, per KV head, the positions [max(0, p + 1 - w), p] -- exactly what a
decode step at length p + 1 would see.  These tests fix that against things that do not go
through the oracle's own code:

* torch's scaled_dot_product_attention in fp64 with an explicit boolean mask written from
  the inequality max(0, p + 1 - w) <= j <= p and an explicit GQA expansion of K and V;
* closed forms: a window of one returns the token's own value row exactly; two tokens give
  logistic weights whose offset would change if the window ended one position early.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _masked_sdpa(q, K, V, p0, windows, G, scale):
    """q [n][Hq][D] (positions p0 .. p0+n-1), K/V [Hkv][Ltot][D] (positions 0 .. Ltot-1)."""
    n, Hq, D = q.shape
    Ltot = K.shape[1]
    kk = torch.from_numpy(K).double().repeat_interleave(G, dim=0)  # [Hq][Ltot][D]
    vv = torch.from_numpy(V).double().repeat_interleave(G, dim=0)
    qq = torch.from_numpy(q).double().permute(1, 0, 2)            # [Hq][n][D]
    mask = torch.zeros((Hq, n, Ltot), dtype=torch.bool)
    for qh in range(Hq):
        w = int(windows[qh // G])
        for i in range(n):
            p = p0 + i
            for j in range(Ltot):
                mask[qh, i, j] = max(0, p + 1 - w) <= j <= p
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
    return o.permute(1, 0, 2).numpy()


def _oracle(q, K, V, p0, windows, scale, lo=None):
    """Hands the oracle each head's history from ``lo[h]`` (default 0) to the chunk's end."""
    n = q.shape[0]
    hist = {}
    for h in range(K.shape[0]):
        a = 0 if lo is None else lo[h]
        hist[h] = (a, K[h, a:p0 + n], V[h, a:p0 + n])
    return oracle.prefill_attention(q, hist, p0, windows, scale, threads=2)


@pytest.mark.parametrize("seed,p0,n,windows,G", [
    (0, 37, 12, (5, 64), 2),          # one window shorter than the chunk, one covering all
    (1, 0, 9, (3, 1, 100), 1),        # chunk at the start of the sequence
    (2, 20, 25, (7, 30), 4),          # both windows shorter than the chunk (w < n)
    (3, 50, 6, (50, 51, 2, 57), 2),   # windows around the context length
])
def test_chunk_matches_masked_sdpa(seed, p0, n, windows, G):
    rng = np.random.default_rng(seed)
    Hkv, D = len(windows), 16
    K = rng.standard_normal((Hkv, p0 + n, D))
    V = rng.standard_normal((Hkv, p0 + n, D))
    q = rng.standard_normal((n, Hkv * G, D))
    scale = 1 / math.sqrt(D)
    got = _oracle(q, K, V, p0, windows, scale)
    ref = _masked_sdpa(q, K, V, p0, windows, G, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_history_trimmed_to_the_windows_gives_the_same_bits():
    """Only [max(0, p0 + 1 - w), p0 + n) is needed: a history trimmed there changes nothing,
    and one missing the oldest needed position is rejected."""
    rng = np.random.default_rng(4)
    p0, n, windows, D = 40, 10, (8, 33), 8
    K = rng.standard_normal((2, p0 + n, D))
    V = rng.standard_normal((2, p0 + n, D))
    q = rng.standard_normal((n, 4, D))
    full = _oracle(q, K, V, p0, windows, 0.3)
    lo = [p0 + 1 - w for w in windows]
    assert np.array_equal(full, _oracle(q, K, V, p0, windows, 0.3, lo=lo))
    with pytest.raises(ValueError):
        _oracle(q, K, V, p0, windows, 0.3, lo=[lo[0] + 1, lo[1]])


def test_window_one_returns_each_tokens_own_value():
    rng = np.random.default_rng(5)
    p0, n, D = 13, 7, 32
    K = rng.standard_normal((1, p0 + n, D)).astype(np.float32)
    V = rng.standard_normal((1, p0 + n, D)).astype(np.float32)
    q = rng.standard_normal((n, 3, D)).astype(np.float32)
    got = _oracle(q, K, V, p0, (1,), 0.2)
    for i in range(n):
        for qh in range(3):
            assert np.array_equal(got[i, qh], V[0, p0 + i].astype(np.float64))


def test_two_token_window_logistic_weights_pin_the_offset():
    """Window 2 at positions p0 = 3 and p0 + 1 = 4, worked by hand.

    Keys: position 2 -> e1, 3 -> 2*e2, 4 -> 3*e3; values: position j -> j * e1 (a single
    column).  q = (1, 1, 1), scale 1.  Token 3 sees positions {2, 3}: scores 1 and 2, so its
    output is (2 e^1 + 3 e^2) / (e^1 + e^2).  Token 4 sees {3, 4}: scores 2 and 3, output
    (3 e^2 + 4 e^3) / (e^2 + e^3).  A window shifted by one position (ending before the token
    itself) would give (1 e^0 + 2 e^1) / (e^0 + e^1) for token 3 instead.
    """
    D = 3
    K = np.zeros((1, 5, D))
    V = np.zeros((1, 5, D))
    K[0, 2] = [1, 0, 0]
    K[0, 3] = [0, 2, 0]
    K[0, 4] = [0, 0, 3]
    for j in range(5):
        V[0, j, 0] = j
    q = np.ones((2, 1, D))
    got = _oracle(q, K, V, 3, (2,), 1.0)
    e = math.exp
    t3 = (2 * e(1) + 3 * e(2)) / (e(1) + e(2))
    t4 = (3 * e(2) + 4 * e(3)) / (e(2) + e(3))
    np.testing.assert_allclose(got[:, 0, 0], [t3, t4], rtol=1e-15, atol=1e-15)
    assert not got[:, 0, 1:].any()


def test_chunk_equals_tokens_appended_and_decoded_one_by_one():
    """The chunk's token i is a decode step at length p0 + i + 1 over the same history."""
    rng = np.random.default_rng(6)
    p0, n, windows, D, G = 25, 9, (4, 17, 200), 8, 2
    K = rng.standard_normal((3, p0 + n, D))
    V = rng.standard_normal((3, p0 + n, D))
    q = rng.standard_normal((n, 6, D))
    got = _oracle(q, K, V, p0, windows, 0.4)
    for i in range(n):
        hist = {(0, h): (0, K[h, :p0 + i + 1], V[h, :p0 + i + 1]) for h in range(3)}
        ref = oracle.attention_jobs(q[i][None], hist, [p0 + i + 1], windows, 0.4, threads=1)[0]
        assert np.array_equal(got[i], ref)
