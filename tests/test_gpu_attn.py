"""GPU parity of the sparse attention (gathered FP4 rows + SWA rows, split-K
with log-sum-exp merge) against the float64 oracle: max-abs <= 2e-3 and
mean-abs <= 2e-4 on the bf16 output."""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp4_kv_cache_06_b300 import csa2
from tests._parity import bits16, check_attn, u8, vmax_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cache(B, n_cap, seed):
    kv = synth.normal_bf16((B, n_cap, 512), seed=seed, stream="kv").to(DEV)
    codes = torch.empty((B, n_cap, 256), dtype=torch.uint8, device=DEV)
    scales = torch.empty((B, n_cap, 32), dtype=torch.uint8, device=DEV)
    csa2.csa2_quantize_kv_fp4(kv, codes, scales)
    return kv, codes, scales


def _oracle_cache(kv_cpu_bits):
    return oracle.quantize_fp4(kv_cpu_bits)


@pytest.mark.parametrize("B,H,k,n", [(1, 16, 512, 2048), (3, 64, 512, 3000), (2, 64, 512, 400), (5, 32, 256, 1000), (8, 48, 64, 100)])
def test_sparse_attn_matches_oracle(B, H, k, n):
    W = 128
    kv, codes, scales = _cache(B, n, seed=B * 100 + H)
    rng = np.random.default_rng(B + H)
    idx = np.full((B, k), -1, dtype=np.int32)
    for b in range(B):
        m = min(k, n) if b % 2 == 0 else min(k, n) // 2       # some rows partly absent
        idx[b, :m] = np.sort(rng.permutation(n)[:m])
    swa_len = np.array([W if b % 3 != 1 else 17 for b in range(B)], dtype=np.int32)
    q = synth.normal_bf16((B, H, 512), seed=7, stream="q").to(DEV)
    swa = synth.normal_bf16((B, W, 512), seed=7, stream="swa").to(DEV)
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_SPARSE_ATTN, B, 0, k, 2048, H))
    csa2.csa2_sparse_attn(q, codes, scales, torch.from_numpy(idx).to(DEV), swa,
                          torch.from_numpy(swa_len).to(DEV), out, ws)
    torch.cuda.synchronize()
    kvb, qb, swab = bits16(kv), bits16(q), bits16(swa)
    ref = np.zeros((B, H, 512))
    vmax = np.zeros((B, 1, 512))
    for b in range(B):
        c, s = oracle.quantize_fp4(kvb[b])
        np.testing.assert_array_equal(u8(codes)[b], c)
        ref[b] = oracle.sparse_attention(qb[b], c, s, idx[b], swab[b], swa_len[b])
        sel = idx[b][idx[b] >= 0]
        vmax[b, 0] = vmax_of(np.concatenate([oracle.dequant_fp4(c[sel], s[sel]),
                                             oracle.bf16_bits_to_f64(swab[b][:swa_len[b]])]))
    few_keys = (idx >= 0).sum(1).min() + swa_len.min() < 300
    check_attn(out, ref, vmax=vmax if few_keys else None)


def test_sparse_attn_empty_and_swa_only():
    B, H, k, n, W = 2, 64, 512, 100, 128
    kv, codes, scales = _cache(B, n, seed=9)
    idx = torch.full((B, k), -1, dtype=torch.int32, device=DEV)
    swa_len = torch.tensor([0, 5], dtype=torch.int32, device=DEV)
    q = synth.normal_bf16((B, H, 512), seed=9, stream="q").to(DEV)
    swa = synth.normal_bf16((B, W, 512), seed=9, stream="swa").to(DEV)
    out = torch.full((B, H, 512), 7.0, dtype=torch.bfloat16, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_SPARSE_ATTN, B, 0, k, 2048, H))
    csa2.csa2_sparse_attn(q, codes, scales, idx, swa, swa_len, out, ws)
    torch.cuda.synchronize()
    assert torch.all(out[0] == 0)
    ref = oracle.sparse_attention(bits16(q)[1], np.zeros((0, 256), np.uint8), np.zeros((0, 32), np.uint8),
                                  np.full(k, -1), bits16(swa)[1], 5)
    check_attn(out[1:], ref[None], vmax=vmax_of(oracle.bf16_bits_to_f64(bits16(swa)[1][:5])))


def test_sparse_attn_out_of_range_index_is_reported_and_skipped():
    B, H, k, n, W = 1, 16, 64, 50, 128
    kv, codes, scales = _cache(B, n, seed=4)
    idxn = np.arange(k, dtype=np.int32)[None]              # 50..63 are >= n_cap
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q = synth.normal_bf16((B, H, 512), seed=4, stream="q").to(DEV)
    swa = synth.normal_bf16((B, W, 512), seed=4, stream="swa").to(DEV)
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_SPARSE_ATTN, B, 0, k, 2048, H))
    csa2.csa2_sparse_attn(q, codes, scales, torch.from_numpy(idxn).to(DEV), swa,
                          torch.tensor([W], dtype=torch.int32, device=DEV), out, ws, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 6
    c, s = oracle.quantize_fp4(bits16(kv)[0])
    ref = oracle.sparse_attention(bits16(q)[0], c, s, np.where(idxn[0] < n, idxn[0], -1), bits16(swa)[0], W)
    keys = np.concatenate([oracle.dequant_fp4(c, s), oracle.bf16_bits_to_f64(bits16(swa)[0])])
    check_attn(out, ref[None], vmax=vmax_of(keys))


def test_prefill_layout_shared_cache_and_sliding_rows():
    """Prefill form: every query reads one shared cache (stride 0) and its own
    window of a chunk's SWA rows (stride 1 row)."""
    Q, H, k, n, W = 40, 64, 512, 1500, 128
    kv, codes, scales = _cache(1, n, seed=12)
    rng = np.random.default_rng(12)
    idx = np.stack([np.sort(rng.permutation(n)[:k]) for _ in range(Q)]).astype(np.int32)
    q = synth.normal_bf16((Q, H, 512), seed=12, stream="q").to(DEV)
    swa_rows = synth.normal_bf16((Q + W - 1, 512), seed=12, stream="swa").to(DEV)
    swa_len = torch.full((Q,), W, dtype=torch.int32, device=DEV)
    out = torch.empty((Q, H, 512), dtype=torch.bfloat16, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_SPARSE_ATTN, Q, 0, k, 2048, H))
    csa2.csa2_sparse_attn(q, codes, scales, torch.from_numpy(idx).to(DEV), swa_rows, swa_len, out, ws,
                          kv_seq_stride=0, swa_seq_stride=1, W=W)
    torch.cuda.synchronize()
    c, s = oracle.quantize_fp4(bits16(kv)[0])
    sb, qb = bits16(swa_rows), bits16(q)
    ref = np.stack([oracle.sparse_attention(qb[i], c, s, idx[i], sb[i:i + W], W) for i in range(Q)])
    check_attn(out, ref)


@pytest.mark.parametrize("W", [0, 17, 64, 100])
def test_sparse_attn_window_sizes(W):
    """Windows that are not a multiple of the 64-key tile: a tile then holds
    window rows and gathered rows together (W = 17, 100), one tile is window
    only (W = 64), or there is no window (W = 0). The window rows of a tile
    are loaded whole by TMA; the rows past the window or past the ring's
    filled slots must not leak into the result."""
    B, H, k, n = 3, 32, 256, 700
    kv, codes, scales = _cache(B, n, seed=300 + W)
    rng = np.random.default_rng(300 + W)
    idx = np.stack([np.sort(rng.permutation(n)[:k]) for _ in range(B)]).astype(np.int32)
    idx[1, k // 2:] = -1                                      # a partly absent row
    swa_len = np.array([W, min(W, 5), W // 2], dtype=np.int32)
    q = synth.normal_bf16((B, H, 512), seed=31, stream="q").to(DEV)
    # ring slots past swa_len hold other data, which must be ignored
    swa = (synth.normal_bf16((B, max(W, 1), 512), seed=32, stream="swa") * 3).to(DEV)[:, :W]
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_SPARSE_ATTN, B, 0, k, 2048, H))
    csa2.csa2_sparse_attn(q, codes, scales, torch.from_numpy(idx).to(DEV), swa.contiguous(),
                          torch.from_numpy(swa_len).to(DEV), out, ws, W=W)
    torch.cuda.synchronize()
    kvb, qb, swab = bits16(kv), bits16(q), bits16(swa.contiguous())
    ref = np.stack([oracle.sparse_attention(qb[b], *oracle.quantize_fp4(kvb[b]), idx[b], swab[b], swa_len[b])
                    for b in range(B)])
    check_attn(out, ref)


def test_prefill_layout_window_not_a_tile_multiple():
    """Prefill form with W = 100 and short windows at the start of a chunk:
    query i's window is the last swa_len of rows i .. i + W - 1."""
    Q, H, k, n, W = 24, 64, 256, 900, 100
    kv, codes, scales = _cache(1, n, seed=41)
    rng = np.random.default_rng(41)
    idx = np.stack([np.sort(rng.permutation(n)[:k]) for _ in range(Q)]).astype(np.int32)
    q = synth.normal_bf16((Q, H, 512), seed=41, stream="q").to(DEV)
    swa_rows = synth.normal_bf16((Q + W - 1, 512), seed=41, stream="swa").to(DEV)
    slen = np.minimum(np.arange(Q) * 9 + 1, W).astype(np.int32)
    out = torch.empty((Q, H, 512), dtype=torch.bfloat16, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_SPARSE_ATTN, Q, 0, k, 2048, H))
    csa2.csa2_sparse_attn(q, codes, scales, torch.from_numpy(idx).to(DEV), swa_rows, torch.from_numpy(slen).to(DEV),
                          out, ws, kv_seq_stride=0, swa_seq_stride=1, W=W, swa_tail=True)
    torch.cuda.synchronize()
    c, s = oracle.quantize_fp4(bits16(kv)[0])
    sb, qb = bits16(swa_rows), bits16(q)
    ref = np.stack([oracle.sparse_attention(qb[i], c, s, idx[i], sb[i + W - slen[i]:i + W], slen[i])
                    for i in range(Q)])
    check_attn(out, ref)


def test_sparse_attn_exact_over_the_bf16_range():
    """Queries and SWA rows far outside fp16's range (|x| up to 1e5) and far
    below it (|x| ~ 1e-6), mixed per head and per row. Each query head is
    brought into fp16's range by an exact power of two folded into its
    softmax scale, and SWA rows beyond it by one folded into their logits and
    probabilities, so the result follows the float64 oracle within the usual
    bound (2e-3 plus the bf16 rounding of the output); no range error is
    reported."""
    B, H, k, n, W = 3, 64, 512, 2500, 128
    kv, codes, scales = _cache(B, n, seed=77)
    rng = np.random.default_rng(77)
    idx = np.stack([np.sort(rng.permutation(n)[:k]) for _ in range(B)]).astype(np.int32)
    g = torch.Generator().manual_seed(77)
    head_scale = torch.tensor([1e5 if h % 3 == 0 else (1e-6 if h % 3 == 1 else 1.0) for h in range(H)])
    row_scale = torch.tensor([1e5 if r % 4 == 0 else (1e-6 if r % 4 == 1 else 1.0) for r in range(W)])
    q = (torch.randn((B, H, 512), generator=g) * head_scale[None, :, None]).to(torch.bfloat16).to(DEV)
    swa = (torch.randn((B, W, 512), generator=g) * row_scale[None, :, None]).to(torch.bfloat16).to(DEV)
    swa_len = torch.tensor([W, 77, 1], dtype=torch.int32, device=DEV)
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_SPARSE_ATTN, B, 0, k, 2048, H))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa2.csa2_sparse_attn(q, codes, scales, torch.from_numpy(idx).to(DEV), swa, swa_len, out, ws, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    kvb, qb, swab = bits16(kv), bits16(q), bits16(swa)
    ref = np.zeros((B, H, 512))
    for b in range(B):
        c, s = oracle.quantize_fp4(kvb[b])
        ref[b] = oracle.sparse_attention(qb[b], c, s, idx[b], swab[b], int(swa_len[b]))
    assert np.abs(ref).max() > 1e4                 # some outputs are dominated by the large rows
    # heads with |q| ~ 1e5 have one-hot softmaxes: P is exactly 1 and 0, so
    # the output is a key row itself and the strict bound applies
    big = np.arange(H) % 3 == 0
    hb, hs = torch.from_numpy(np.nonzero(big)[0]).to(DEV), torch.from_numpy(np.nonzero(~big)[0]).to(DEV)
    check_attn(out[:, hb], ref[:, big])
    # elsewhere large rows carry weight, and rounding P to bf16 moves the
    # output by up to 2^-9 max_j |v_jd| per dim (the bound the library states)
    vmax = np.zeros((B, 1, 512))
    for b in range(B):
        c, s = oracle.quantize_fp4(kvb[b])
        sel = idx[b][idx[b] >= 0]
        vmax[b, 0] = vmax_of(np.concatenate([oracle.dequant_fp4(c[sel], s[sel]),
                                             oracle.bf16_bits_to_f64(swab[b][:int(swa_len[b])])]))
    check_attn(out[:, hs], ref[:, ~big], vmax=vmax)


def test_sparse_attn_reports_swa_rows_beyond_its_range():
    """An SWA row reaching 2^23 (past the 2^7 scale-down) is reported as
    CSA2_ERR_DEVICE_RANGE; the call still completes."""
    B, H, k, n, W = 1, 16, 64, 200, 128
    kv, codes, scales = _cache(B, n, seed=78)
    idx = torch.arange(k, dtype=torch.int32, device=DEV)[None]
    q = synth.normal_bf16((B, H, 512), seed=78, stream="q").to(DEV)
    swa = synth.normal_bf16((B, W, 512), seed=78, stream="swa").to(DEV)
    swa[0, 3, 7] = 1e8
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_SPARSE_ATTN, B, 0, k, 2048, H))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa2.csa2_sparse_attn(q, codes, scales, idx, swa, torch.tensor([W], dtype=torch.int32, device=DEV), out, ws,
                          d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 7
