"""GPU parity of multi-token decode: R new tokens of each sequence decoded in
one step (rows_per_seq = R). Each token is its own query row: it sees the
cache up to itself, has its own indexer query, Top-K, pool and layer
queries, and attends over its own 128-token window. The oracle runs each
token as a single-token step."""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp4_kv_cache_06_b300 import csa2
from tests._parity import bits16, check_attn, check_topk, u8, vmax_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("R", [4, 2, 8])
def test_multi_token_decode_full_and_reindex_groups(R):
    S, W, H, L, P, k = 3, 128, 64, 2, 256, 512
    n_prev = [5000, 300, 90]                         # tokens cached before the step, per sequence
    n_cap = 5200
    B = S * R
    seed = 600 + R
    kv = synth.normal_bf16((S, n_cap, 512), seed=seed, stream="kv")
    codes = torch.empty((S, n_cap, 256), dtype=torch.uint8, device=DEV)
    scales = torch.empty((S, n_cap, 32), dtype=torch.uint8, device=DEV)
    csa2.csa2_quantize_kv_fp4(kv.to(DEV), codes, scales)
    kI = synth.indexer_keys_e4m3((S, n_cap, 128), seed=seed, bias_prob=0.05)
    kI_d = kI.to(DEV)
    # token i of sequence s sits at position n_prev[s] + i and sees positions up to itself
    n_row = np.array([n_prev[r // R] + r % R + 1 for r in range(B)], dtype=np.int64)
    n_t = torch.from_numpy(n_row).to(DEV)
    kbar = torch.zeros((S, (n_cap + 7) // 8, 128), dtype=torch.uint8, device=DEV)
    n_seq = torch.tensor([n_prev[s] + R for s in range(S)], dtype=torch.int64, device=DEV)
    csa2.csa2_block_means(kI_d, n_seq, kbar, n_max=n_cap)
    qI1 = synth.normal_e4m3((B, 8, 128), seed=seed, stream="qI", sub=0)
    w1 = synth.uniform_f32((B, 8), seed=seed, stream="w", sub=0)
    qI2 = synth.normal_e4m3((B, 8, 128), seed=seed, stream="qI", sub=1)
    w2 = synth.uniform_f32((B, 8), seed=seed, stream="w", sub=1)
    qs = [synth.normal_bf16((B, H, 512), seed=seed, stream="q", sub=l) for l in range(2 * L)]
    swas = [synth.normal_bf16((S, W + R - 1, 512), seed=seed, stream="swa", sub=l) for l in range(2 * L)]
    swa_len = np.minimum(n_row, W).astype(np.int32)  # tokens 0 .. p of the sequence, at most W
    swa_len_d = torch.from_numpy(swa_len).to(DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_LAYER_GROUP, B, n_cap, k, P, H))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pool = torch.full((B, P), -1, dtype=torch.int32, device=DEV)
    idx1 = torch.empty((B, k), dtype=torch.int32, device=DEV)
    idx2 = torch.empty((B, k), dtype=torch.int32, device=DEV)
    outs = [torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV) for _ in range(2 * L)]
    n_max = int(n_row.max())
    csa2.csa2_layer_group(csa2.MODE_FULL, n_t, n_max, codes, scales, kI_d, qI1.to(DEV), w1.to(DEV), idx1,
                          [q.to(DEV) for q in qs[:L]], [x.to(DEV) for x in swas[:L]], swa_len_d, outs[:L], ws,
                          kbar=kbar, pool=pool, form_pool=csa2.POOL_MEAN_KEY, P=P, d_status=st, rows_per_seq=R)
    csa2.csa2_layer_group(csa2.MODE_REINDEX, n_t, n_max, codes, scales, kI_d, qI2.to(DEV), w2.to(DEV), idx2,
                          [q.to(DEV) for q in qs[L:]], [x.to(DEV) for x in swas[L:]], swa_len_d, outs[L:], ws,
                          kbar=kbar, pool=pool, form_pool=False, P=P, d_status=st, rows_per_seq=R)
    torch.cuda.synchronize()
    assert st.item() == 0
    g1, g2, gp = idx1.cpu().numpy(), idx2.cpu().numpy(), pool.cpu().numpy()
    quant = [oracle.quantize_fp4(bits16(kv)[s]) for s in range(S)]
    compared = 0

    def attend(l, r, ref_idx):
        s, i = r // R, r % R
        c, sc = quant[s]
        rows = bits16(swas[l])[s][i + W - swa_len[r]: i + W]        # the window's present rows
        ref = oracle.sparse_attention(bits16(qs[l])[r], c, sc, ref_idx, rows, int(swa_len[r]))
        sel = ref_idx[ref_idx >= 0]
        few = len(sel) + int(swa_len[r]) < 300
        vm = vmax_of(np.concatenate([oracle.dequant_fp4(c[sel], sc[sel]), oracle.bf16_bits_to_f64(rows)])) if few else None
        check_attn(outs[l][r:r + 1], ref[None], vmax=vm)

    for r in range(B):
        s, n = r // R, int(n_row[r])
        kb = u8(kI)[s]
        ref_idx, ref_s = oracle.full_topk(u8(qI1)[r], w1.numpy()[r], kb, n, k)
        check_topk(g1[r], ref_idx, ref_s, np.arange(n), k)
        # the block means are the sequence's, after all R tokens were appended;
        # each token scores the blocks that hold its visible positions
        kbar_seq = oracle.block_means(kb, n_prev[s] + R)
        ref_pool, ref_bs = oracle.form_pool(u8(qI1)[r], w1.numpy()[r], kbar_seq[:(n + 7) // 8], P)
        check_topk(gp[r], ref_pool, ref_bs, np.arange(ref_bs.size), P)
        if np.array_equal(g1[r], ref_idx):
            for l in range(L):
                attend(l, r, ref_idx)
                compared += 1
        if not np.array_equal(gp[r], ref_pool):
            continue
        ref_idx2, ref_s2, ref_pos2 = oracle.reindex_topk(u8(qI2)[r], w2.numpy()[r], kb, ref_pool, n, k)
        check_topk(g2[r], ref_idx2, ref_s2, ref_pos2, k)
        if np.array_equal(g2[r], ref_idx2):
            for l in range(L, 2 * L):
                attend(l, r, ref_idx2)
                compared += 1
    assert compared >= 3 * B


def test_rows_per_seq_must_divide_the_rows():
    B, R = 6, 4
    with pytest.raises(ValueError):
        csa2.csa2_layer_group(csa2.MODE_FULL, torch.ones(B, dtype=torch.int64, device=DEV), 1,
                              torch.zeros((2, 8, 256), dtype=torch.uint8, device=DEV),
                              torch.zeros((2, 8, 32), dtype=torch.uint8, device=DEV),
                              torch.zeros((2, 8, 128), dtype=torch.uint8, device=DEV),
                              torch.zeros((B, 8, 128), dtype=torch.uint8, device=DEV),
                              torch.zeros((B, 8), dtype=torch.float32, device=DEV),
                              torch.zeros((B, 512), dtype=torch.int32, device=DEV),
                              [torch.zeros((B, 64, 512), dtype=torch.bfloat16, device=DEV)],
                              [torch.zeros((2, 128 + R - 1, 512), dtype=torch.bfloat16, device=DEV)],
                              torch.ones(B, dtype=torch.int32, device=DEV),
                              [torch.empty((B, 64, 512), dtype=torch.bfloat16, device=DEV)],
                              csa2.alloc_workspace(1 << 20), rows_per_seq=R)
