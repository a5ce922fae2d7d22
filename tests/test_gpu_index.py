"""GPU parity of the indexer scan, Top-K, pool formation and Reindex against
the oracle (scores to fp32 accuracy; index sets equal outside the 1e-5
relative tie band around the k-th score)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp4_kv_cache_06_b300 import csa2
from tests._parity import check_topk, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(B, n_cap, H_I, d_I, seed, bias=0.0):
    kI = synth.indexer_keys_e4m3((B, n_cap, d_I), seed=seed, bias_prob=bias)
    qI = synth.normal_e4m3((B, H_I, d_I), seed=seed, stream="qI")
    w = synth.uniform_f32((B, H_I), seed=seed, stream="w")
    return kI, qI, w


def _ws(op, B, n_max, k=512, P=2048, H=64):
    return csa2.alloc_workspace(csa2.workspace_size(op, B, n_max, k, P, H))


@pytest.mark.parametrize("H_I,d_I", [(4, 64), (8, 128), (3, 128), (8, 64)])
def test_scores_match_oracle(H_I, d_I):
    B, n_cap = 4, 9000
    ns = [9000, 1, 4097, 0]
    kI, qI, w = _inputs(B, n_cap, H_I, d_I, seed=11, bias=0.05)
    scores = torch.full((B, n_cap), -7.0, dtype=torch.float32, device=DEV)
    n = torch.tensor(ns, dtype=torch.int64, device=DEV)
    csa2.csa2_index_scores(qI.to(DEV), w.to(DEV), kI.to(DEV), n, n_cap, scores)
    torch.cuda.synchronize()
    s = scores.cpu().numpy()
    for b in range(B):
        ref = oracle.indexer_scores(u8(qI)[b], w.numpy()[b], u8(kI)[b, :ns[b]])
        np.testing.assert_allclose(s[b, :ns[b]], ref, rtol=2e-6, atol=1e-6)
        assert np.all(s[b, ns[b]:] == -7.0)


@pytest.mark.parametrize("n_list,k", [([2048], 512), ([131072, 5000, 511, 0], 512), ([70000, 300], 2048), ([600], 512)])
def test_index_full_topk(n_list, k):
    B, n_cap = len(n_list), max(n_list) + 13
    kI, qI, w = _inputs(B, n_cap, 8, 128, seed=21, bias=0.05)
    n = torch.tensor(n_list, dtype=torch.int64, device=DEV)
    idx = torch.empty((B, k), dtype=torch.int32, device=DEV)
    scores = torch.empty((B, n_cap), dtype=torch.float32, device=DEV)
    ws = _ws(csa2.OP_INDEX_FULL, B, n_cap, k)
    csa2.csa2_index_full(qI.to(DEV), w.to(DEV), kI.to(DEV), n, n_cap, k, idx, ws, scores_out=scores)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    for b in range(B):
        ref_idx, ref_s = oracle.full_topk(u8(qI)[b], w.numpy()[b], u8(kI)[b], n_list[b], k)
        check_topk(gi[b], ref_idx, ref_s, np.arange(n_list[b]), k)


def test_topk_exact_ties_deterministic():
    """Integer scores with massive ties: the selection is unique (lower
    positions win) and must match bit for bit, including the slow path when
    more than 8192 candidates share the threshold bin."""
    rng = np.random.default_rng(0)
    cases = [rng.integers(0, 50, 100000), np.zeros(30000), rng.integers(0, 3, 20000), np.arange(5000)[::-1] % 7]
    for sv in cases:
        m = sv.size
        for k in (1, 512, 2048):
            scores = torch.tensor(sv, dtype=torch.float32, device=DEV).reshape(1, m)
            n = torch.tensor([m], dtype=torch.int64, device=DEV)
            idx = torch.empty((1, k), dtype=torch.int32, device=DEV)
            ws = _ws(csa2.OP_TOPK, 1, m, k)
            csa2.csa2_topk(scores, n, m, k, idx, ws)
            torch.cuda.synchronize()
            ref = oracle.topk_select(sv.astype(np.float64), np.arange(m), k)
            np.testing.assert_array_equal(idx.cpu().numpy()[0], ref)


def test_topk_candidate_positions_and_absent():
    rng = np.random.default_rng(1)
    B, m, k = 3, 16384, 512
    s = rng.standard_normal((B, m)).astype(np.float32)
    pos = rng.permutation(10 ** 6)[:B * m].reshape(B, m).astype(np.int32)
    pos[rng.random((B, m)) < 0.3] = -1
    pos[2, 100:] = -1                # a row with fewer candidates than k
    idx = torch.empty((B, k), dtype=torch.int32, device=DEV)
    ws = _ws(csa2.OP_TOPK, B, m, k)
    csa2.csa2_topk(torch.from_numpy(s).to(DEV), None, m, k, idx, ws, cand_pos=torch.from_numpy(pos).to(DEV))
    torch.cuda.synchronize()
    for b in range(B):
        ref = oracle.topk_select(s[b].astype(np.float64), pos[b], k)
        np.testing.assert_array_equal(idx.cpu().numpy()[b], ref)


@pytest.mark.parametrize("m", [40000, 8_400_000])
def test_topk_long_rows_and_unordered_positions(m):
    """Rows past the short-row limit go through the ordered compaction; rows
    past the chunk table's reach (8M entries) and candidates whose positions do
    not increase with the index take the exact 64-bit select and a sort."""
    rng = np.random.default_rng(m)
    k = 512
    s = rng.standard_normal((1, m)).astype(np.float32)
    idx = torch.empty((1, k), dtype=torch.int32, device=DEV)
    ws = _ws(csa2.OP_TOPK, 1, m, k)
    csa2.csa2_topk(torch.from_numpy(s).to(DEV), None, m, k, idx, ws)
    torch.cuda.synchronize()
    ref = oracle.topk_select(s[0].astype(np.float64), np.arange(m), k)
    np.testing.assert_array_equal(idx.cpu().numpy()[0], ref)
    if m < 10 ** 6:
        pos = rng.permutation(10 ** 7)[:m].reshape(1, m).astype(np.int32)
        csa2.csa2_topk(torch.from_numpy(s).to(DEV), None, m, k, idx, ws, cand_pos=torch.from_numpy(pos).to(DEV))
        torch.cuda.synchronize()
        ref = oracle.topk_select(s[0].astype(np.float64), pos[0], k)
        np.testing.assert_array_equal(idx.cpu().numpy()[0], ref)


def test_form_pool_and_reindex():
    B, d_I, P, k = 3, 128, 2048, 512
    n_list = [40000, 16384, 3001]
    n_cap = 40008
    kI, qI, w = _inputs(B, n_cap, 8, d_I, seed=31)
    qP = synth.normal_e4m3((B, 8, d_I), seed=31, stream="qI_pool")
    wP = synth.uniform_f32((B, 8), seed=31, stream="w_pool")
    kI_d = kI.to(DEV)
    kbar = torch.zeros((B, n_cap // 8, d_I), dtype=torch.uint8, device=DEV)
    n = torch.tensor(n_list, dtype=torch.int64, device=DEV)
    csa2.csa2_block_means(kI_d, n, kbar, n_max=max(n_list))
    pool = torch.empty((B, P), dtype=torch.int32, device=DEV)
    csa2.csa2_form_pool(qP.to(DEV), wP.to(DEV), kbar, n, max(n_list), P, pool, _ws(csa2.OP_FORM_POOL, B, n_cap, P=P))
    idx = torch.empty((B, k), dtype=torch.int32, device=DEV)
    csa2.csa2_index_reindex(qI.to(DEV), w.to(DEV), kI_d, n, pool, k, idx, _ws(csa2.OP_INDEX_REINDEX, B, 0, k, P))
    torch.cuda.synchronize()
    gp, gi = pool.cpu().numpy(), idx.cpu().numpy()
    for b in range(B):
        kb_ref = oracle.block_means(u8(kI)[b], n_list[b])
        np.testing.assert_array_equal(u8(kbar)[b, :kb_ref.shape[0]], kb_ref)
        ref_pool, ref_bs = oracle.form_pool(u8(qP)[b], wP.numpy()[b], kb_ref, P)
        check_topk(gp[b], ref_pool, ref_bs, np.arange(kb_ref.shape[0]), P)
        # rescore the oracle's own pool; compare Top-K when the pools agree
        ref_idx, ref_s, ref_pos = oracle.reindex_topk(u8(qI)[b], w.numpy()[b], u8(kI)[b], ref_pool, n_list[b], k)
        if np.array_equal(gp[b], ref_pool):
            check_topk(gi[b], ref_idx, ref_s, ref_pos, k)


def test_reindex_on_oracle_pool():
    """Reindex given the oracle's pool as input (isolates the rescoring)."""
    B, d_I, P, k = 2, 64, 700, 512
    n_list = [20000, 5555]
    kI, qI, w = _inputs(B, 20000, 4, d_I, seed=41, bias=0.05)
    rng = np.random.default_rng(2)
    pools = np.full((B, P), -1, dtype=np.int32)
    for b in range(B):
        nb = (n_list[b] + 7) // 8
        pools[b, :min(P, nb)] = np.sort(rng.permutation(nb)[:min(P, nb)])
    idx = torch.empty((B, k), dtype=torch.int32, device=DEV)
    n = torch.tensor(n_list, dtype=torch.int64, device=DEV)
    csa2.csa2_index_reindex(qI.to(DEV), w.to(DEV), kI.to(DEV), n, torch.from_numpy(pools).to(DEV), k, idx,
                            _ws(csa2.OP_INDEX_REINDEX, B, 0, k, P))
    torch.cuda.synchronize()
    for b in range(B):
        ref_idx, ref_s, ref_pos = oracle.reindex_topk(u8(qI)[b], w.numpy()[b], u8(kI)[b], pools[b], n_list[b], k)
        check_topk(idx.cpu().numpy()[b], ref_idx, ref_s, ref_pos, k)


def test_form_pool_block_max_matches_oracle():
    """Pool by the max-of-token rule from given scores, ragged rows, P < and >= #blocks."""
    rng = np.random.default_rng(5)
    n_list = [131072, 40000, 9000, 15]
    B, m = len(n_list), max(n_list)
    s = rng.standard_normal((B, m)).astype(np.float32)
    s[1, :5000] = np.round(s[1, :5000])            # ties on block maxima
    n = torch.tensor(n_list, dtype=torch.int64, device=DEV)
    for P in (2048, 512):
        pool = torch.empty((B, P), dtype=torch.int32, device=DEV)
        ws = _ws(csa2.OP_FORM_POOL_BLOCK_MAX, B, m)
        csa2.csa2_form_pool_block_max(torch.from_numpy(s).to(DEV), n, m, P, pool, ws)
        torch.cuda.synchronize()
        gp = pool.cpu().numpy()
        for b in range(B):
            ref_pool, ref_bs = oracle.form_pool_block_max(s[b].astype(np.float64), n_list[b], P)
            check_topk(gp[b], ref_pool, ref_bs, np.arange(ref_bs.size), P)


def test_full_group_block_max_pool_holds_every_top_position():
    """A Full layer forming its pool by the block maxima of its own scores:
    the pool matches the oracle and contains the block of every Top-512
    position the layer selected."""
    B, n, H, P = 2, 150000, 64, 2048
    kI, qI, w = _inputs(B, n, 8, 128, seed=31, bias=0.05)
    codes = torch.zeros((B, n, 256), dtype=torch.uint8, device=DEV)
    scales = torch.zeros((B, n, 32), dtype=torch.uint8, device=DEV)
    nt = torch.full((B,), n, dtype=torch.int64, device=DEV)
    idx = torch.empty((B, 512), dtype=torch.int32, device=DEV)
    pool = torch.full((B, P), -1, dtype=torch.int32, device=DEV)
    q = [torch.zeros((B, H, 512), dtype=torch.bfloat16, device=DEV)]
    swa = [torch.zeros((B, 128, 512), dtype=torch.bfloat16, device=DEV)]
    out = [torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV)]
    swa_len = torch.zeros((B,), dtype=torch.int32, device=DEV)
    ws = _ws(csa2.OP_LAYER_GROUP, B, n, 512, P, H)
    csa2.csa2_layer_group(csa2.MODE_FULL, nt, n, codes, scales, kI.to(DEV), qI.to(DEV), w.to(DEV), idx, q, swa,
                          swa_len, out, ws, pool=pool, form_pool=csa2.POOL_BLOCK_MAX, P=P)
    torch.cuda.synchronize()
    gi, gp = idx.cpu().numpy(), pool.cpu().numpy()
    for b in range(B):
        ref_idx, ref_s = oracle.full_topk(u8(qI)[b], w.numpy()[b], u8(kI)[b], n)
        check_topk(gi[b], ref_idx, ref_s, np.arange(n), 512)
        ref_pool, ref_bs = oracle.form_pool_block_max(ref_s, n, P)
        check_topk(gp[b], ref_pool, ref_bs, np.arange(ref_bs.size), P)
        assert set((gi[b] // 8).tolist()) <= set(gp[b].tolist())


@pytest.mark.parametrize("k", [512, 2048])
def test_topk_many_long_rows(k):
    """Many position rows longer than 32K entries (ordered compaction, chunk
    table, ordered select): rows with heavy exact ties, an all-tied row (more
    than 8192 candidates in the threshold bin: the slow path), ragged and empty
    rows; every row exact."""
    rng = np.random.default_rng(k)
    B, m = 20, 70000
    s = rng.standard_normal((B, m)).astype(np.float32)
    s[1] = rng.integers(0, 50, m)
    s[2] = 0.0
    s[3] = rng.integers(0, 3, m)
    n_list = [m] * B
    n_list[4], n_list[5], n_list[6], n_list[7] = 100, 0, 511, 33000
    n = torch.tensor(n_list, dtype=torch.int64, device=DEV)
    idx = torch.empty((B, k), dtype=torch.int32, device=DEV)
    ws = _ws(csa2.OP_TOPK, B, m, k)
    csa2.csa2_topk(torch.from_numpy(s).to(DEV), n, m, k, idx, ws)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    for b in range(B):
        ref = oracle.topk_select(s[b, :n_list[b]].astype(np.float64), np.arange(n_list[b]), k)
        np.testing.assert_array_equal(gi[b], ref)


@pytest.mark.parametrize("k", [512, 2048])
def test_index_full_many_long_rows_topk(k):
    """The Full scan's fused histogram feeding Top-K on many rows past the
    short-row limit."""
    B, n_cap = 17, 40000
    n_list = [40000] * 16 + [35001]
    kI, qI, w = _inputs(B, n_cap, 8, 128, seed=33, bias=0.05)
    n = torch.tensor(n_list, dtype=torch.int64, device=DEV)
    idx = torch.empty((B, k), dtype=torch.int32, device=DEV)
    ws = _ws(csa2.OP_INDEX_FULL, B, n_cap, k)
    csa2.csa2_index_full(qI.to(DEV), w.to(DEV), kI.to(DEV), n, n_cap, k, idx, ws)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    for b in range(0, B, 4):
        ref_idx, ref_s = oracle.full_topk(u8(qI)[b], w.numpy()[b], u8(kI)[b], n_list[b], k)
        check_topk(gi[b], ref_idx, ref_s, np.arange(n_list[b]), k)
