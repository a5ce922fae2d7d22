"""The CSA2 step, written out plainly in float64 (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring for the page
citations [CSA2], [FP4], [CED], [TG] and the readings taken where the pages
are silent).

Array conventions (numpy):
  bf16 tensors are given as uint16 bit patterns; E4M3 tensors as uint8;
  the FP4 main-KV cache as ``codes`` [n, 256] uint8 (two E2M1 codes per
  byte, channel 2i in the low nibble) and ``scales`` [n, 32] uint8 (E4M3,
  one per 16 channels).
"""
from __future__ import annotations

import numpy as np

from .formats import E2M1_GRID, bf16_bits_to_f64, e2m1_encode_mag, e4m3_decode, e4m3_encode

GROUP = 16  # channels per E4M3 scale [FP4]


# --------------------------------------------------------------------------
# FP4 main KV [FP4]
# --------------------------------------------------------------------------
def quantize_fp4(x_bits):
    """Quantise bf16 rows [..., d] to E2M1 codes + one E4M3 scale per 16 channels.

    [FP4]: E2M1 values, one E4M3 scale per 16 channels, no global scale.
    The pages do not state how the scale is chosen; the reading taken is the
    plainest NVFP4-style rule without a global factor: scale = E4M3(amax/6)
    (6 = largest E2M1 magnitude), round-to-nearest-even, saturating. Each
    value is coded as E2M1(|x| / scale) with the sign of x; a group whose
    scale rounds to zero stores +0 codes.
    Returns (codes [..., d/2] uint8, scales [..., d/16] uint8).
    """
    x = bf16_bits_to_f64(x_bits)
    d = x.shape[-1]
    assert d % GROUP == 0
    xg = x.reshape(x.shape[:-1] + (d // GROUP, GROUP))
    amax = np.max(np.abs(xg), axis=-1)
    sc = e4m3_encode(amax / 6.0)
    s = e4m3_decode(sc)
    live = s > 0
    ratio = np.abs(xg) / np.where(live, s, 1.0)[..., None]
    mag = e2m1_encode_mag(ratio).astype(np.int64)
    sign = np.signbit(xg).astype(np.int64)
    code = np.where(live[..., None], mag | (sign << 3), 0)
    code = code.reshape(x.shape[:-1] + (d,))
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    return packed, sc.astype(np.uint8)


def dequant_fp4(codes, scales):
    """E2M1 codes [..., d/2] and E4M3 scales [..., d/16] -> float64 rows [..., d] (exact)."""
    codes = np.asarray(codes, dtype=np.uint8)
    lo = codes & 0xF
    hi = codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (codes.shape[-1] * 2,)).astype(np.int64)
    mag = E2M1_GRID[c & 7]
    val = np.where((c >> 3) & 1, -mag, mag)
    s = e4m3_decode(scales)
    return val * np.repeat(s, GROUP, axis=-1)


# --------------------------------------------------------------------------
# Indexer [CSA2]
# --------------------------------------------------------------------------
def indexer_scores(q_bytes, w, k_bytes):
    """s_t = sum_h w_h * relu(q_h . k_t) for every key row t.

    [CSA2] says a Full layer projects indexer K from its main KV and
    selects Top-512, and a Reindex layer rescores that K with its own
    indexer Q; the pages give no formula. The reading taken: one E4M3 key
    per position shared by all indexer heads, E4M3 per-head queries q_h,
    fp32 head weights w_h, no 1/sqrt(d) factor.
    q_bytes [H_I, d_I] uint8, w [H_I] float, k_bytes [m, d_I] uint8 -> [m] float64.
    """
    Q = e4m3_decode(q_bytes)
    K = e4m3_decode(k_bytes)
    dots = K @ Q.T                                  # [m, H_I], exact products, fp64 sums
    return np.maximum(dots, 0.0) @ np.asarray(w, dtype=np.float64)


def block_means(k_bytes, n, block=8):
    """Mean indexer key of each aligned block of 8 positions, stored as E4M3.

    [CSA2] pools candidates in blocks of 8 positions; the block's own
    score is not defined on the pages. The reading taken: the block is
    scored by the indexer on the mean of its present keys (the last block
    may be partial), rounded to E4M3 so the same scan scores it.
    k_bytes [>=n, d_I] -> [ceil(n/8), d_I] uint8.
    """
    n = int(n)
    nb = (n + block - 1) // block
    K = e4m3_decode(np.asarray(k_bytes)[:n])
    out = np.zeros((nb, K.shape[1]), dtype=np.uint8)
    for j in range(nb):
        rows = K[j * block:min((j + 1) * block, n)]
        out[j] = e4m3_encode(rows.sum(axis=0) / rows.shape[0])
    return out


# --------------------------------------------------------------------------
# Top-K [CSA2]
# --------------------------------------------------------------------------
def topk_select(scores, positions, k):
    """The k best candidates by (score descending, position ascending).

    Candidates with position < 0 are absent. Returns int32 [k]: the chosen
    positions sorted ascending, padded with -1 when fewer than k exist.
    """
    scores = np.asarray(scores, dtype=np.float64)
    positions = np.asarray(positions, dtype=np.int64)
    keep = positions >= 0
    s, p = scores[keep], positions[keep]
    order = np.lexsort((p, -s))                     # last key is the primary one
    chosen = np.sort(p[order[:k]])
    out = np.full(k, -1, dtype=np.int32)
    out[:chosen.size] = chosen
    return out


def full_topk(q_bytes, w, k_bytes, n, k=512):
    """Full mode [CSA2]: score every visible position t < n, select Top-k.

    Returns (idx int32 [k], scores float64 [n]).
    """
    s = indexer_scores(q_bytes, w, np.asarray(k_bytes)[:int(n)])
    return topk_select(s, np.arange(int(n)), k), s


def form_pool(q_bytes, w, kbar_bytes, P=2048):
    """Hierarchical candidate pool [CSA2]: the Full layer keeps up to P blocks.

    Block j is scored with the pool-forming (Full layer's) indexer query on
    its mean key; the best min(P, #blocks) blocks by (score desc, block id
    asc) form the pool. Returns (block ids int32 [P] ascending, -1 padded;
    block scores float64).
    """
    nb = np.asarray(kbar_bytes).shape[0]
    s = indexer_scores(q_bytes, w, kbar_bytes)
    return topk_select(s, np.arange(nb), P), s


def form_pool_block_max(scores, n, P=2048, block=8):
    """Pool variant with guaranteed recall (a reading beyond the pages).

    [CSA2] lets the Full layer form a pool of up to P blocks of 8 positions
    but does not say how a block is scored. This variant scores block j by
    the largest Full-layer score of its positions 8j .. 8j+7 below n, and keeps
    the best min(P, #blocks) blocks by (score desc, block id asc). Any block
    holding one of the Full Top-k positions then scores at least the k-th
    score, so for P >= k the pool holds all of them.
    scores [>= n] float -> (block ids int32 [P] ascending, -1 padded;
    block scores float64 [ceil(n/8)]).
    """
    n = int(n)
    s = np.asarray(scores, dtype=np.float64)[:n]
    nb = (n + block - 1) // block
    bmax = np.array([s[j * block:min((j + 1) * block, n)].max() for j in range(nb)], dtype=np.float64)
    return topk_select(bmax, np.arange(nb), P), bmax


def pool_positions(pool_blocks, n, block=8):
    """Positions covered by the pool's blocks that are < n, ascending."""
    pb = np.asarray(pool_blocks, dtype=np.int64)
    pb = pb[pb >= 0]
    pos = (pb[:, None] * block + np.arange(block)[None, :]).reshape(-1)
    return np.sort(pos[pos < int(n)])


def reindex_topk(q_bytes, w, k_bytes, pool_blocks, n, k=512):
    """Reindex mode [CSA2]: rescore only the pool's positions with this layer's
    own indexer query, then Top-k. Returns (idx int32 [k], scores, positions)."""
    pos = pool_positions(pool_blocks, n)
    s = indexer_scores(q_bytes, w, np.asarray(k_bytes)[pos])
    return topk_select(s, pos, k), s, pos


# --------------------------------------------------------------------------
# Sparse attention + SWA [CSA2], [CED], [FP4]
# --------------------------------------------------------------------------
def sparse_attention(q_bits, codes, scales, idx, swa_bits, swa_len, scale=None):
    """softmax(q X^T * scale) X over the gathered main-KV rows and the SWA rows.

    q_bits [H, d] bf16 bits; codes/scales: the FP4 cache of this sequence;
    idx [k] int (-1 = absent); swa_bits [W, d] bf16 bits, of which the first
    swa_len slots hold keys. Main K = V (one shared vector per position);
    SWA K = V likewise; SWA keys are distinct from the sparse ones.
    Returns float64 [H, d]; zeros when there is no key at all.
    """
    q = bf16_bits_to_f64(q_bits)
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    idx = np.asarray(idx, dtype=np.int64)
    idx = idx[idx >= 0]
    X_sparse = dequant_fp4(np.asarray(codes)[idx], np.asarray(scales)[idx])
    X_swa = bf16_bits_to_f64(np.asarray(swa_bits)[:int(swa_len)])
    X = np.concatenate([X_sparse.reshape(-1, d), X_swa.reshape(-1, d)], axis=0)
    if X.shape[0] == 0:
        return np.zeros_like(q)
    logits = (q @ X.T) * scale                      # [H, keys]
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    return (p @ X) / p.sum(axis=1, keepdims=True)


def layer_group(mode, q_layers, swa_layers, swa_len, codes, scales, n,
                kI=None, qI=None, w=None, pool_blocks=None, k=512):
    """One CSA2 layer group: a Full or Reindex layer followed by Reuse layers.

    [CSA2]: Full selects new Top-512 over all positions; Reindex rescores
    the pool with its own indexer query; Reuse takes the group's last Top-K
    unchanged and skips the indexer ([TG]: sharing Top-K removes re-scoring
    the whole history). Every layer has its own main Q and SWA KV.
    q_layers [L, H, d], swa_layers [L, W, d]. Returns (idx [k], out [L, H, d]).
    """
    if mode == "full":
        idx, _ = full_topk(qI, w, kI, n, k)
    elif mode == "reindex":
        idx, _, _ = reindex_topk(qI, w, kI, pool_blocks, n, k)
    else:
        raise ValueError(mode)
    outs = np.stack([sparse_attention(q_layers[l], codes, scales, idx, swa_layers[l], swa_len)
                     for l in range(len(q_layers))])
    return idx, outs


def swa_ring_after(rows, n, W=128):
    """The ring a layer holds after n tokens were appended one by one [CED].

    [CED] keeps a 128-token sliding window in every layer; how it is stored is
    the build's choice: a ring with token t at slot t mod W, rewritten by each
    new token. rows [n][d] in token order -> ring [W][d] (slots of tokens not
    yet seen are zero)."""
    rows = np.asarray(rows)
    ring = np.zeros((W,) + rows.shape[1:], dtype=rows.dtype)
    for t in range(int(n)):
        ring[t % W] = rows[t]
    return ring


# --------------------------------------------------------------------------
# Prefill causal rule [CSA2] (encoder: compression ratio 2), [CED]
# --------------------------------------------------------------------------
def prefill_visible(p, ratio=2):
    """Compressed entries visible to the query at token position p.

    Entry j summarises tokens ratio*j .. ratio*j + ratio - 1 (how the tokens
    are merged is not on the pages; entries are inputs here). The entry is
    visible once its last token is <= p, so the count is floor((p+1)/ratio).
    """
    return (np.asarray(p, dtype=np.int64) + 1) // ratio


def prefill_swa_rows(p, W=128):
    """Token positions in the query's sliding window: max(0, p-W+1) .. p."""
    return np.arange(max(0, int(p) - W + 1), int(p) + 1)
