"""Pins for the oracle's sparse attention (gathered FP4 rows + SWA rows).

Pinned against torch's scaled_dot_product_attention in float64 on the
CPU (library routine) when Top-K covers every position, the log-sum-exp
merge identity, and closed forms (single key, zero query, identical keys).
"""
import numpy as np
import torch

import oracle


def bf16_bits(x):
    return (torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def make_cache(rng, n, d=512):
    kv = bf16_bits(rng.standard_normal((n, d)))
    codes, scales = oracle.quantize_fp4(kv)
    return codes, scales


def test_dense_equivalence_with_sdpa():
    rng = np.random.default_rng(0)
    n, H, W = 300, 16, 128
    codes, scales = make_cache(rng, n)
    q = bf16_bits(rng.standard_normal((H, 512)))
    swa = bf16_bits(rng.standard_normal((W, 512)))
    idx = np.arange(512, dtype=np.int32)
    idx[n:] = -1                                       # k >= n: every position chosen
    got = oracle.sparse_attention(q, codes, scales, idx, swa, 100)
    X = np.concatenate([oracle.dequant_fp4(codes, scales), oracle.bf16_bits_to_f64(swa[:100])])
    Q = torch.from_numpy(oracle.bf16_bits_to_f64(q))[None, :, None, :].transpose(1, 2)  # [1,1,H,d]
    K = torch.from_numpy(X)[None, None]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, K, scale=1.0 / np.sqrt(512))
    np.testing.assert_allclose(got, ref[0, 0].numpy(), rtol=1e-12, atol=1e-13)


def test_lse_merge_identity():
    rng = np.random.default_rng(1)
    codes, scales = make_cache(rng, 700)
    q = bf16_bits(rng.standard_normal((4, 512)))
    swa = bf16_bits(rng.standard_normal((128, 512)))
    idx = np.sort(rng.permutation(700)[:512]).astype(np.int32)
    full = oracle.sparse_attention(q, codes, scales, idx, swa, 128)
    # the two parts separately, merged with their log-sum-exp weights
    Qf = oracle.bf16_bits_to_f64(q)
    parts = []
    for X in (oracle.dequant_fp4(codes[idx], scales[idx]), oracle.bf16_bits_to_f64(swa)):
        L = Qf @ X.T / np.sqrt(512)
        m = L.max(1, keepdims=True)
        p = np.exp(L - m)
        parts.append((m, p.sum(1, keepdims=True), p @ X))
    M = np.maximum(parts[0][0], parts[1][0])
    num = sum(np.exp(m - M) * o for m, l, o in parts)
    den = sum(np.exp(m - M) * l for m, l, o in parts)
    np.testing.assert_allclose(full, num / den, rtol=1e-12, atol=1e-14)


def test_closed_forms():
    rng = np.random.default_rng(2)
    codes, scales = make_cache(rng, 50)
    swa = bf16_bits(rng.standard_normal((128, 512)))
    q = bf16_bits(rng.standard_normal((3, 512)))
    idx = np.full(512, -1, dtype=np.int32)
    idx[0] = 17
    # single key: the output is that key's dequantised row for every head
    out = oracle.sparse_attention(q, codes, scales, idx, swa, 0)
    row = oracle.dequant_fp4(codes[17], scales[17])
    np.testing.assert_array_equal(out, np.broadcast_to(row, out.shape))
    # zero query: uniform weights -> mean of the keys
    q0 = np.zeros((2, 512), dtype=np.uint16)
    idx2 = np.arange(512, dtype=np.int32)
    idx2[50:] = -1
    out0 = oracle.sparse_attention(q0, codes, scales, idx2, swa, 10)
    X = np.concatenate([oracle.dequant_fp4(codes, scales), oracle.bf16_bits_to_f64(swa[:10])])
    np.testing.assert_allclose(out0, np.broadcast_to(X.mean(0), out0.shape), rtol=1e-13, atol=1e-15)
    # no key at all -> zeros
    assert np.all(oracle.sparse_attention(q, codes, scales, np.full(512, -1), swa, 0) == 0)


def test_reuse_equals_recompute_on_group_indices():
    rng = np.random.default_rng(3)
    n = 3000
    kv = bf16_bits(rng.standard_normal((n, 512)))
    codes, scales = oracle.quantize_fp4(kv)
    kI = torch.from_numpy(rng.standard_normal((n, 64)).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    qI = torch.from_numpy(rng.standard_normal((4, 64)).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    w = rng.random(4)
    L = 4
    q = bf16_bits(rng.standard_normal((L, 16, 512)))
    swa = bf16_bits(rng.standard_normal((L, 128, 512)))
    idx, outs = oracle.layer_group("full", q, swa, 128, codes, scales, n, kI=kI, qI=qI, w=w)
    full_idx, _ = oracle.full_topk(qI, w, kI, n, 512)
    np.testing.assert_array_equal(idx, full_idx)
    for l in range(L):
        np.testing.assert_array_equal(outs[l], oracle.sparse_attention(q[l], codes, scales, full_idx, swa[l], 128))


def test_swa_ring_after_brute_force():
    """The ring after n appends holds the last min(n, W) tokens, token t at
    slot t mod W, against an explicit window of the last W tokens."""
    rng = np.random.default_rng(3)
    W = 16
    rows = rng.integers(1, 1 << 15, (70, 4))
    for n in (0, 1, 15, 16, 17, 40, 70):
        ring = oracle.swa_ring_after(rows, n, W)
        window = list(range(max(0, n - W), n))
        for t in window:
            assert (ring[t % W] == rows[t]).all()
        filled = {t % W for t in window}
        for slot in range(W):
            if slot not in filled:
                assert (ring[slot] == 0).all()
