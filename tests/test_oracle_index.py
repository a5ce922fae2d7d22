"""Pins for the oracle's indexer score, block means, Top-K, pool and Reindex.

Pinned against pure-Python loops on tiny inputs, exact rational means with
nearest-value enumeration, structural invariants of Top-K (every chosen
score >= every unchosen one; ties broken toward lower positions) and
special cases where the hierarchical pool must reproduce the Full result.
"""
from fractions import Fraction

import numpy as np
import torch

import oracle


def e4m3_bytes(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def e4m3_val(b):
    return float(torch.tensor([int(b)], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item())


def test_indexer_loops_tiny():
    rng = np.random.default_rng(0)
    H, dI, n = 3, 8, 17
    q = e4m3_bytes(rng.standard_normal((H, dI)))
    k = e4m3_bytes(rng.standard_normal((n, dI)))
    w = rng.random(H)
    got = oracle.indexer_scores(q, w, k)
    for t in range(n):
        s = 0.0
        for h in range(H):
            dot = sum(e4m3_val(q[h, c]) * e4m3_val(k[t, c]) for c in range(dI))
            s += w[h] * (dot if dot > 0 else 0.0)
        assert abs(got[t] - s) <= 1e-12 * max(1.0, abs(s))


def test_indexer_permutation_and_onehot():
    rng = np.random.default_rng(1)
    q = e4m3_bytes(rng.standard_normal((8, 128)))
    k = e4m3_bytes(rng.standard_normal((300, 128)))
    w = rng.random(8)
    s = oracle.indexer_scores(q, w, k)
    perm = rng.permutation(300)
    np.testing.assert_array_equal(oracle.indexer_scores(q, w, k[perm]), s[perm])
    # one-hot weight picks relu of a single head's dot product
    Q = oracle.e4m3_decode(q)
    K = oracle.e4m3_decode(k)
    for h in (0, 5):
        oh = np.zeros(8)
        oh[h] = 1.0
        np.testing.assert_allclose(oracle.indexer_scores(q, oh, k), np.maximum(K @ Q[h], 0), rtol=0, atol=1e-12)
    assert np.all(s >= 0)


def test_block_means_exact():
    rng = np.random.default_rng(2)
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    table = [(c, Fraction(float(v))) for c, v in enumerate(vals)]
    for n in (1, 7, 8, 9, 23, 24):
        k = e4m3_bytes(rng.standard_normal((n, 4)) * 3)
        got = oracle.block_means(k, n)
        assert got.shape == ((n + 7) // 8, 4)
        for j in range(got.shape[0]):
            rows = range(8 * j, min(8 * j + 8, n))
            for c in range(4):
                m = sum(Fraction(e4m3_val(k[t, c])) for t in rows) / len(rows)
                mag = abs(m)
                best = None
                for code, v in table:
                    d = abs(mag - v)
                    if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
                        best = (d, code)
                exp = best[1] | (0x80 if m < 0 else 0)
                if m == 0:
                    assert got[j, c] & 0x7F == 0
                else:
                    assert got[j, c] == exp, (n, j, c)


def test_block_means_identical_keys():
    rng = np.random.default_rng(3)
    base = e4m3_bytes(rng.standard_normal((5, 16)))
    k = np.repeat(base, 8, axis=0)
    np.testing.assert_array_equal(oracle.block_means(k, 40), base)


def _check_topk_invariants(scores, positions, k, idx):
    valid = positions >= 0
    s_of = dict(zip(positions[valid].tolist(), scores[valid].tolist()))
    chosen = [int(i) for i in idx if i >= 0]
    assert chosen == sorted(chosen) and len(set(chosen)) == len(chosen)
    assert all(i == -1 for i in idx[len(chosen):])
    assert len(chosen) == min(k, len(s_of))
    rest = set(s_of) - set(chosen)
    if chosen and rest:
        for p in rest:
            for c in chosen:
                # chosen beats unchosen: higher score, or equal score and lower position
                assert (s_of[c] > s_of[p]) or (s_of[c] == s_of[p] and c < p)


def test_topk_invariants_with_ties():
    rng = np.random.default_rng(4)
    for trial in range(20):
        m = int(rng.integers(1, 80))
        scores = rng.integers(0, 6, m).astype(np.float64)      # many exact ties
        positions = rng.permutation(1000)[:m]
        positions[rng.random(m) < 0.1] = -1
        k = int(rng.integers(1, 40))
        idx = oracle.topk_select(scores, positions, k)
        _check_topk_invariants(scores, positions, k, idx)


def test_topk_k_ge_n_returns_all():
    rng = np.random.default_rng(5)
    s = rng.random(30)
    idx = oracle.topk_select(s, np.arange(30), 512)
    assert list(idx[:30]) == list(range(30)) and np.all(idx[30:] == -1)
    assert np.all(oracle.topk_select(s[:0], np.arange(0), 4) == -1)


def test_full_topk_matches_sorted_scores():
    rng = np.random.default_rng(6)
    q = e4m3_bytes(rng.standard_normal((4, 64)))
    k = e4m3_bytes(rng.standard_normal((2048, 64)))
    w = rng.random(4)
    idx, s = oracle.full_topk(q, w, k, 2048, 512)
    _check_topk_invariants(s, np.arange(2048), 512, idx)


def test_pool_all_blocks_when_small():
    rng = np.random.default_rng(7)
    n = 1000
    k = e4m3_bytes(rng.standard_normal((n, 32)))
    kbar = oracle.block_means(k, n)
    q = e4m3_bytes(rng.standard_normal((2, 32)))
    pool, _ = oracle.form_pool(q, rng.random(2), kbar, P=2048)
    nb = (n + 7) // 8
    assert list(pool[:nb]) == list(range(nb)) and np.all(pool[nb:] == -1)
    np.testing.assert_array_equal(oracle.pool_positions(pool, n), np.arange(n))


def test_reindex_equals_full_for_blockwise_constant_keys():
    """Keys constant within each block: mean = key, so block score = token score.
    With the pool formed by the same indexer query that rescores it, the pool's
    Top-512 equals the Full Top-512 (pool holds the best 2048 blocks)."""
    rng = np.random.default_rng(8)
    nb = 5000
    base = e4m3_bytes(rng.standard_normal((nb, 32)))
    k = np.repeat(base, 8, axis=0)
    n = nb * 8 - 3                                      # ragged last block
    q = e4m3_bytes(rng.standard_normal((4, 32)))
    w = rng.random(4)
    kbar = oracle.block_means(k, n)
    pool, _ = oracle.form_pool(q, w, kbar, P=2048)
    full_idx, _ = oracle.full_topk(q, w, k, n, 512)
    re_idx, _, pos = oracle.reindex_topk(q, w, k, pool, n, 512)
    np.testing.assert_array_equal(re_idx, full_idx)
    assert pos.size <= 2048 * 8 and np.all(pos < n)


def test_pool_recall_tiny():
    """On inputs with at most 2048 blocks the pool holds every block of the
    brute-force Top-512 (the pool is then the whole context)."""
    rng = np.random.default_rng(9)
    n = 16000
    k = e4m3_bytes(rng.standard_normal((n, 16)))
    q = e4m3_bytes(rng.standard_normal((2, 16)))
    w = rng.random(2)
    pool, _ = oracle.form_pool(q, w, oracle.block_means(k, n))
    full_idx, _ = oracle.full_topk(q, w, k, n, 512)
    assert set((full_idx // 8).tolist()) <= set(pool.tolist())


def test_block_max_pool_brute_force_and_small_context():
    """Block maxima against explicit loops over ragged rows; with at most P
    blocks the pool is every block."""
    rng = np.random.default_rng(21)
    for n in (1, 7, 8, 9, 63, 1000):
        s = rng.standard_normal(n + 5)
        pool, bmax = oracle.form_pool_block_max(s, n, P=4096)
        nb = (n + 7) // 8
        for j in range(nb):
            m = -np.inf
            for t in range(8 * j, min(8 * j + 8, n)):
                m = max(m, s[t])
            assert bmax[j] == m
        assert pool[:nb].tolist() == list(range(nb)) and np.all(pool[nb:] == -1)


def test_block_max_pool_recall_guarantee_with_ties():
    """For P >= k every Full Top-k position lies in a pool block, including
    integer scores with massive ties and the Top-k tie-break by position."""
    rng = np.random.default_rng(22)
    for n, k, P in ((5000, 64, 64), (20000, 512, 512), (20000, 512, 2048), (3000, 100, 150)):
        for s in (rng.standard_normal(n), rng.integers(0, 5, n).astype(np.float64)):
            pool, _ = oracle.form_pool_block_max(s, n, P)
            top = oracle.topk_select(s, np.arange(n), k)
            assert set((top[top >= 0] // 8).tolist()) <= set(pool[pool >= 0].tolist())


def test_mean_key_pool_can_miss_a_top_position():
    """The mean-key rule gives no such guarantee: a block whose keys point in
    opposite directions has a near-zero mean key although one of its
    positions has the largest score."""
    d = 16
    q = e4m3_bytes(np.eye(1, d)[0:1] * 4.0)                  # one head on channel 0
    w = np.array([1.0])
    k = np.zeros((8 * 4, d))
    k[0, 0], k[1, 0] = 4.0, -4.0                             # block 0: +4 and -4 -> mean 0
    for j in range(1, 4):
        k[8 * j:8 * j + 8, 0] = 1.0                          # blocks 1..3: all +1
    kb = e4m3_bytes(k)
    n = 32
    full_top, s = oracle.full_topk(q, w, kb, n, 1)
    assert full_top[0] == 0                                  # position 0 has the best score
    pool_mean, _ = oracle.form_pool(q, w, oracle.block_means(kb, n), P=1)
    pool_max, _ = oracle.form_pool_block_max(s, n, P=1)
    assert pool_max[0] == 0 and pool_mean[0] != 0


def test_prefill_visible_brute_force():
    for r in (1, 2, 4):
        for p in range(0, 50):
            brute = sum(1 for j in range(100) if r * j + r - 1 <= p)
            assert oracle.prefill_visible(p, r) == brute
    assert list(oracle.prefill_swa_rows(3)) == [0, 1, 2, 3]
    assert list(oracle.prefill_swa_rows(300))[:2] == [173, 174] and len(oracle.prefill_swa_rows(300)) == 128
