"""GPU parity at the benchmark workloads' full sizes, on sampled outputs.

Each test builds a workload with the shapes of one timed configuration and
runs it through the same calls, and so the same launch configuration (grid,
key splits, Top-K mode), that the bench times. The oracle then recomputes
sampled sequences (or prefill queries) one by one:
- the Full scan's Top-512 over every position;
- the pool of 2048 blocks;
- the Reindex Top-512;
- every sampled layer's attention output.

Inputs come from `synth` on the host. Indexer keys are random per position.
Main-KV position t holds bf16 row t mod R of a per-sequence block of R rows,
quantised by the kernel in place, so the oracle can quantise any gathered row
itself without regenerating gigabytes of rows.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp4_kv_cache_06_b300 import csa2
from tests._parity import attn_with_oracle_idx, bits16, check_attn, check_topk, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"
R = 4096                 # distinct main-KV rows per sequence
SEED = 4321


def _periodic_cache(B, n_cap):
    base = synth.normal_bf16((B, R, 512), seed=SEED, stream="kv")
    cb = torch.empty((B, R, 256), dtype=torch.uint8, device=DEV)
    sb = torch.empty((B, R, 32), dtype=torch.uint8, device=DEV)
    csa2.csa2_quantize_kv_fp4(base.to(DEV), cb, sb)
    rows = torch.arange(n_cap, device=DEV) % R
    return base, cb[:, rows].contiguous(), sb[:, rows].contiguous()


def _keys(B, n, bias):
    kI = torch.empty((B, n, 128), dtype=torch.uint8, device=DEV)
    for b in range(B):
        kI[b] = synth.indexer_keys_e4m3((n, 128), seed=SEED, bias_prob=bias, sub=b).to(DEV)
    return kI


def _keys_host(b, n, bias):
    return u8(synth.indexer_keys_e4m3((n, 128), seed=SEED, bias_prob=bias, sub=b))


def _layer_inputs(B, H, L, sub0=0):
    qs = [synth.normal_bf16((B, H, 512), seed=SEED, stream="q", sub=sub0 + l) for l in range(L)]
    swas = [synth.normal_bf16((B, 128, 512), seed=SEED, stream="swa", sub=sub0 + l) for l in range(L)]
    return qs, swas


def _oracle_rows(base_b):
    return oracle.quantize_fp4(bits16(base_b))


_compared = {"group": 0, "oracle_idx": 0}


def _reset():
    _compared["group"] = 0
    _compared["oracle_idx"] = 0


def _check_attention(out_b, q_b, swa_b, c, s, idx):
    """out_b [1][H][512] from the kernel; the oracle attends over rows idx mod R."""
    idx = np.asarray(idx)
    rows = np.where(idx >= 0, idx % R, -1)
    ref = oracle.sparse_attention(bits16(q_b), c, s, rows, bits16(swa_b), 128)
    check_attn(out_b, ref[None])


def _check_layers(b, gpu_idx, ref_idx, outs, qs, swas, codes, scales, c, s, layers):
    """Attention parity of sequence b's layers. Where the kernel's selection
    equals the oracle's, the group's own outputs are compared; where it
    differs inside the tie band, the row is attended again on the GPU over
    the oracle's entries and that output is compared."""
    same = np.array_equal(gpu_idx, ref_idx)
    for l in layers:
        if same:
            got = outs[l][b:b + 1]
            _compared["group"] += 1
        else:
            got = attn_with_oracle_idx(qs[l][b], codes[b], scales[b], ref_idx, swas[l][b])
            _compared["oracle_idx"] += 1
        _check_attention(got, qs[l][b], swas[l][b], c, s, ref_idx)


def _reindex_with_pool(qI_b, w_b, kI_b, n, pool_row, k=512):
    """The Reindex scan and Top-K of one sequence on the GPU over a given pool
    (the oracle's, where the kernel's pool differs inside the tie band)."""
    idx = torch.empty((1, k), dtype=torch.int32, device=DEV)
    P = len(pool_row)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_INDEX_REINDEX, 1, n, k, P, 64))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa2.csa2_index_reindex(qI_b[None].to(DEV), w_b[None].to(DEV), kI_b[None], torch.tensor([n], device=DEV),
                            torch.from_numpy(np.asarray(pool_row, dtype=np.int32)[None].copy()).to(DEV), k, idx, ws,
                            d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return idx.cpu().numpy()[0]


def _group(mode, n_t, n_max, codes, scales, kI, qI, w, qs, swas, kbar, pool, form_pool, qP=None, wP=None,
           k=512, P=2048):
    B, H = qs[0].shape[:2]
    idx = torch.empty((B, k), dtype=torch.int32, device=DEV)
    outs = [torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV) for _ in qs]
    swa_len = torch.full((B,), 128, dtype=torch.int32, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_LAYER_GROUP, B, codes.shape[1], k, P, H))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa2.csa2_layer_group(mode, n_t, n_max, codes, scales, kI, qI, w, idx, [q.to(DEV) for q in qs],
                          [x.to(DEV) for x in swas], swa_len, outs, ws, kbar=kbar, pool=pool,
                          form_pool=form_pool, qI_pool=qP, w_pool=wP, P=P, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return idx.cpu().numpy(), outs


def _full_state(B, n, bias):
    base, codes, scales = _periodic_cache(B, n)
    kI = _keys(B, n, bias)
    kbar = torch.zeros((B, (n + 7) // 8, 128), dtype=torch.uint8, device=DEV)
    n_t = torch.full((B,), n, dtype=torch.int64, device=DEV)
    csa2.csa2_block_means(kI, n_t, kbar, n_max=n)
    pool = torch.full((B, 2048), -1, dtype=torch.int32, device=DEV)
    return base, codes, scales, kI, kbar, n_t, pool


def test_decoder_group_full_b32_ctx131072_sampled():
    """Full + 3 Reuse, batch 32, 131,072 positions, 5 % biased keys: eight
    sampled sequences, every layer of each compared."""
    _reset()
    cfg = synth.get_config(2)
    B, n, H, L = cfg.B, cfg.n, cfg.H, 4
    base, codes, scales, kI, kbar, n_t, pool = _full_state(B, n, cfg.bias_prob)
    qI = synth.normal_e4m3((B, 8, 128), seed=SEED, stream="qI")
    w = synth.uniform_f32((B, 8), seed=SEED, stream="w")
    qs, swas = _layer_inputs(B, H, L)
    gi, outs = _group(csa2.MODE_FULL, n_t, n, codes, scales, kI, qI.to(DEV), w.to(DEV), qs, swas, kbar, pool,
                      False)
    sample = (0, 4, 9, 13, 18, 22, 27, 31)
    for b in sample:
        ref_idx, ref_s = oracle.full_topk(u8(qI)[b], w.numpy()[b], _keys_host(b, n, cfg.bias_prob), n)
        check_topk(gi[b], ref_idx, ref_s, np.arange(n), 512)
        c, s = _oracle_rows(base[b])
        _check_layers(b, gi[b], ref_idx, outs, qs, swas, codes, scales, c, s, range(L))
    assert _compared["group"] + _compared["oracle_idx"] == len(sample) * L
    assert _compared["group"] >= len(sample) * L // 2, _compared


def test_decoder_group_pool_reindex_b8_ctx1m_sampled():
    """Pool formation + Reindex + 3 Reuse, batch 8, 1,048,576 positions."""
    _reset()
    cfg = synth.get_config(3)
    B, n, H, L, P = cfg.B, cfg.n, cfg.H, 4, cfg.P
    base, codes, scales, kI, kbar, n_t, pool = _full_state(B, n, 0.0)
    qI = synth.normal_e4m3((B, 8, 128), seed=SEED, stream="qI")
    w = synth.uniform_f32((B, 8), seed=SEED, stream="w")
    qP = synth.normal_e4m3((B, 8, 128), seed=SEED, stream="qI_pool")
    wP = synth.uniform_f32((B, 8), seed=SEED, stream="w_pool")
    qs, swas = _layer_inputs(B, H, L)
    gi, outs = _group(csa2.MODE_REINDEX, n_t, n, codes, scales, kI, qI.to(DEV), w.to(DEV), qs, swas, kbar, pool,
                      True, qP=qP.to(DEV), wP=wP.to(DEV), P=P)
    gp = pool.cpu().numpy()
    sample = (0, 7)
    for b in sample:
        kb = _keys_host(b, n, 0.0)
        kbar_ref = oracle.block_means(kb, n)
        ref_pool, ref_bs = oracle.form_pool(u8(qP)[b], wP.numpy()[b], kbar_ref, P)
        check_topk(gp[b], ref_pool, ref_bs, np.arange(kbar_ref.shape[0]), P)
        ref_idx, ref_s, ref_pos = oracle.reindex_topk(u8(qI)[b], w.numpy()[b], kb, ref_pool, n)
        # the Reindex selection: the group's where its pool is the oracle's,
        # else the GPU Reindex run again over the oracle's pool
        g_idx = gi[b] if np.array_equal(gp[b], ref_pool) else _reindex_with_pool(qI[b], w[b], kI[b], n, ref_pool)
        check_topk(g_idx, ref_idx, ref_s, ref_pos, 512)
        c, s = _oracle_rows(base[b])
        _check_layers(b, gi[b], ref_idx, outs, qs, swas, codes, scales, c, s, range(L))
    assert _compared["group"] + _compared["oracle_idx"] == len(sample) * L


def test_decoder_stack_b4_ctx1m_sampled():
    """The 20-layer stack's groups at 1,048,576 positions, batch 4: Full + 3
    Reuse forming the pool with the Full layer's indexer query, then four
    Reindex + 3 Reuse groups over that pool."""
    _reset()
    cfg = synth.get_config(5)
    B, n, H = cfg.B, cfg.n, cfg.H
    base, codes, scales, kI, kbar, n_t, pool = _full_state(B, n, 0.0)
    G = len(cfg.groups)
    qIs = [synth.normal_e4m3((B, 8, 128), seed=SEED, stream="qI", sub=g) for g in range(G)]
    ws_ = [synth.uniform_f32((B, 8), seed=SEED, stream="w", sub=g) for g in range(G)]
    results = []
    l0 = 0
    for g, (mode, n_reuse, form_pool) in enumerate(cfg.groups):
        L = 1 + n_reuse
        qs, swas = _layer_inputs(B, H, L, sub0=l0)
        m = csa2.MODE_FULL if mode == "full" else csa2.MODE_REINDEX
        gi, outs = _group(m, n_t, n, codes, scales, kI, qIs[g].to(DEV), ws_[g].to(DEV), qs, swas, kbar, pool,
                          form_pool)
        results.append((mode, gi, outs, qs, swas))
        l0 += L
    gp = pool.cpu().numpy()
    sample = (0, 3)
    for b in sample:
        kb = _keys_host(b, n, 0.0)
        c, s = _oracle_rows(base[b])
        # group 0: Full Top-512 and the pool formed with the same indexer query
        ref_idx, ref_s = oracle.full_topk(u8(qIs[0])[b], ws_[0].numpy()[b], kb, n)
        check_topk(results[0][1][b], ref_idx, ref_s, np.arange(n), 512)
        kbar_ref = oracle.block_means(kb, n)
        ref_pool, ref_bs = oracle.form_pool(u8(qIs[0])[b], ws_[0].numpy()[b], kbar_ref, cfg.P)
        check_topk(gp[b], ref_pool, ref_bs, np.arange(kbar_ref.shape[0]), cfg.P)
        _, gi, outs, qs, swas = results[0]
        _check_layers(b, gi[b], ref_idx, outs, qs, swas, codes, scales, c, s, (0, len(outs) - 1))
        same_pool = np.array_equal(gp[b], ref_pool)
        for g in range(1, G):
            ref_idx, ref_s, ref_pos = oracle.reindex_topk(u8(qIs[g])[b], ws_[g].numpy()[b], kb, ref_pool, n)
            _, gi, outs, qs, swas = results[g]
            g_idx = gi[b] if same_pool else _reindex_with_pool(qIs[g][b], ws_[g][b], kI[b], n, ref_pool)
            check_topk(g_idx, ref_idx, ref_s, ref_pos, 512)
            _check_layers(b, gi[b], ref_idx, outs, qs, swas, codes, scales, c, s, (len(outs) - 1,))
    assert _compared["group"] + _compared["oracle_idx"] == len(sample) * (2 + (G - 1))


def test_encoder_prefill_chunk4096_ctx262144_sampled():
    """4096 queries at tokens 258,048 .. 262,143 over 131,072 compressed
    entries (ratio 2), Full + 5 Reuse, causal visibility and sliding windows."""
    cfg = synth.get_config(4)
    Q, n, H, W, k = cfg.prefill_queries, cfg.n, cfg.H, cfg.W, cfg.k
    L = 1 + cfg.groups[0][1]
    p0 = n * cfg.ratio - Q
    base, codes, scales = _periodic_cache(1, n)
    kI_h = synth.indexer_keys_e4m3((n, 128), seed=SEED)
    qI = synth.normal_e4m3((Q, 8, 128), seed=SEED, stream="qI")
    w = synth.uniform_f32((Q, 8), seed=SEED, stream="w")
    qs = [synth.normal_bf16((Q, H, 512), seed=SEED, stream="q", sub=l) for l in range(L)]
    swas = [synth.normal_bf16((Q + W - 1, 512), seed=SEED, stream="swa", sub=l) for l in range(L)]
    pos = np.arange(p0, p0 + Q)
    n_vis = np.minimum(oracle.prefill_visible(pos, cfg.ratio), n)
    swa_len = np.minimum(pos + 1, W).astype(np.int32)
    outs = [torch.empty((Q, H, 512), dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    idx = torch.empty((Q, k), dtype=torch.int32, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_PREFILL_GROUP, Q, n, k, 0, H))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa2.csa2_prefill_group(torch.from_numpy(n_vis).to(DEV), codes[0], scales[0], kI_h.to(DEV), qI.to(DEV),
                            w.to(DEV), idx, [x.to(DEV) for x in qs], [x.to(DEV) for x in swas],
                            torch.from_numpy(swa_len).to(DEV), outs, ws, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    gi = idx.cpu().numpy()
    c, s = _oracle_rows(base[0])
    kb = u8(kI_h)
    compared = 0
    for qi in (0, 1, 2047, Q - 2, Q - 1):
        ref_idx, ref_s = oracle.full_topk(u8(qI)[qi], w.numpy()[qi], kb, int(n_vis[qi]), k)
        check_topk(gi[qi], ref_idx, ref_s, np.arange(int(n_vis[qi])), k)
        same = np.array_equal(gi[qi], ref_idx)
        rows = oracle.prefill_swa_rows(pos[qi], W) - (p0 - W + 1)
        sel = np.where(ref_idx >= 0, ref_idx % R, -1)
        for l in (0, L - 1):
            ref = oracle.sparse_attention(bits16(qs[l])[qi], c, s, sel, bits16(swas[l])[rows], len(rows))
            if same:
                got = outs[l][qi:qi + 1]
            else:                         # tie-band difference: attend over the oracle's entries
                got = attn_with_oracle_idx(qs[l][qi], codes[0], scales[0], ref_idx, swas[l][rows], W)
            check_attn(got, ref[None])
            compared += int(same)
    assert compared >= 6, "too few sampled queries kept the group's own selection"
