"""The twenty-layer decode stack over 256 appended steps at full shape.

Batch 4, 1,048,320 cached positions before the first step and 1,048,576
after the last; one Full + 3 Reuse group that forms the pool, then four
Reindex + 3 Reuse groups. The steps run through the benchmark's own
workload object, so every call, grid and Top-K mode is the one that is
timed. At steps 0, 1, 63, 127, 191, 254 and 255 two sequences are checked
against the oracle:
- the rows the step appended: FP4 codes and scales, indexer key, the block
  mean of the block being filled, the SWA ring slot of two layers
  (bit-exact), and the whole SWA ring of each checked layer;
- the Full layer's Top-512, the pool of 2048 blocks and every Reindex
  group's Top-512 (equal sets outside the tie band);
- the attention output of the first layer of every group.

The oracle's per-position scores and block means of the 1,048,320 initial
positions are computed once and extended by the appended positions at each
checked step. Both are defined per position (block means per aligned block
of eight, and 1,048,320 is a multiple of eight), so the extension equals a
recomputation over all positions.

Inputs are drawn on the device by `synth`, as the workload draws them, and
copied to the host; the initial rows are drawn again rather than read back
from caches the kernels have written to.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
import synth
from fp4_kv_cache_06_b300 import csa2
from tests._parity import attn_with_oracle_idx, bits16, check_attn, check_topk, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"
SEED = 1234                       # the workload's default seed
CHECK_STEPS = (0, 1, 63, 127, 191, 254, 255)
SAMPLE = (0, 3)
CHUNK = 1 << 17                   # rows per drawn block of the initial main KV


def _initial_rows(b, positions, n_pre):
    """bf16 bits of initial main-KV rows of sequence b at the given positions
    (< n_pre), drawn again in the workload's chunks."""
    positions = np.asarray(positions, dtype=np.int64)
    out = np.empty((len(positions), 512), dtype=np.uint16)
    for c in np.unique(positions // CHUNK):
        sel = np.nonzero(positions // CHUNK == c)[0]
        c0 = int(c) * CHUNK
        # the same shape as the workload's draw (a device draw of another
        # shape does not reproduce its values)
        x = synth.normal_bf16((1, min(CHUNK, n_pre - c0), 512), SEED, "kv", DEV, sub=b * 4096 + int(c))
        out[sel] = bits16(x[0, torch.from_numpy(positions[sel] - c0).to(DEV)])
    return out


def _rows_of(b, positions, n_pre, kv_new_bits):
    """bf16 bits of main-KV rows at `positions` after the appends (positions
    >= n_pre hold the appended token's row)."""
    positions = np.asarray(positions, dtype=np.int64)
    out = np.empty((len(positions), 512), dtype=np.uint16)
    old = positions < n_pre
    if old.any():
        out[old] = _initial_rows(b, positions[old], n_pre)
    out[~old] = kv_new_bits[b]
    return out


def test_stack_256_appended_steps_at_checked_steps():
    cfg = synth.get_config(5)
    wl = bench.DecodeWorkload(cfg, torch.device(DEV), seed=SEED)
    n_pre = wl.n_first - 1
    assert n_pre % 8 == 0 and n_pre + cfg.steps == cfg.n
    W, P, k, G = cfg.W, cfg.P, cfg.k, len(cfg.groups)
    first_layer = np.cumsum([0] + [1 + g[1] for g in cfg.groups])[:G]
    ring_layers = (0, wl.layers - 1)

    # inputs (generator output, never written by a kernel)
    qI = [u8(t) for t in wl.qI]
    w = [t.cpu().numpy() for t in wl.w]
    q_bits = [bits16(wl.q[l]) for l in first_layer]
    kv_new = bits16(wl.kv_new)
    kI_new = u8(wl.kI_new)
    swa_new = [bits16(t) for t in wl.swa_new]
    ring0 = [synth.normal_bf16((wl.B, W, 512), SEED, "swa", DEV, sub=l) for l in range(wl.layers)]
    ring0 = [bits16(t) for t in ring0]
    c_new, s_new = oracle.quantize_fp4(kv_new)

    # oracle state of the initial positions, once per sampled sequence
    keys0, s0, kbar0 = {}, {}, {}
    for b in SAMPLE:
        keys0[b] = u8(synth.indexer_keys_e4m3((n_pre, cfg.d_I), SEED, DEV, bias_prob=cfg.bias_prob, sub=b))
        s0[b] = oracle.indexer_scores(qI[0][b], w[0][b], keys0[b])
        kbar0[b] = oracle.block_means(keys0[b], n_pre)

    checked = {"steps": 0, "attn_group": 0, "attn_oracle_idx": 0}

    def check(step):
        pos = n_pre + step
        n = pos + 1
        codes, scales = wl.codes, wl.scales
        for b in SAMPLE:
            # appended rows
            assert np.array_equal(u8(codes[b, pos]), c_new[b])
            assert np.array_equal(u8(scales[b, pos]), s_new[b])
            assert np.array_equal(u8(wl.kI[b, pos]), kI_new[b])
            keys_app = np.repeat(kI_new[b][None], step + 1, axis=0)
            kb_tail = oracle.block_means(keys_app, step + 1)
            nb0 = n_pre // 8
            assert np.array_equal(u8(wl.kbar[b, nb0:nb0 + len(kb_tail)]), kb_tail)
            ring = {}
            for l in ring_layers + tuple(int(x) for x in first_layer):
                r = ring0[l][b].copy()
                for t in range(n_pre, n):
                    r[t % W] = swa_new[l][b]
                ring[l] = r
            for l in ring_layers:
                assert np.array_equal(bits16(wl.swa[l][b, pos % W]), swa_new[l][b])
                assert np.array_equal(bits16(wl.swa[l][b]), ring[l])
            # Full Top-512 and the pool (formed with the Full layer's query)
            s_full = np.concatenate([s0[b], oracle.indexer_scores(qI[0][b], w[0][b], keys_app)])
            ref_idx = [oracle.topk_select(s_full, np.arange(n), k)]
            gidx = [u8(wl.idx[g][b]) for g in range(G)]
            check_topk(gidx[0], ref_idx[0], s_full, np.arange(n), k)
            kbar_all = np.concatenate([kbar0[b], kb_tail])
            ref_pool, ref_bs = oracle.form_pool(qI[0][b], w[0][b], kbar_all, P)
            gpool = u8(wl.pool[b])
            check_topk(gpool, ref_pool, ref_bs, np.arange(kbar_all.shape[0]), P)
            same_pool = np.array_equal(gpool, ref_pool)
            keys_all = np.concatenate([keys0[b], keys_app])
            for g in range(1, G):
                ri, rs, rp = oracle.reindex_topk(qI[g][b], w[g][b], keys_all, ref_pool, n, k)
                ref_idx.append(ri)
                if same_pool:
                    got = gidx[g]
                else:                       # tie-band pool difference: Reindex over the oracle's pool
                    got = _reindex_with_pool(wl.qI[g][b], wl.w[g][b], wl.kI[b], n, ref_pool, k)
                check_topk(got, ri, rs, rp, k)
            # attention of each group's first layer
            need = np.unique(np.concatenate([r[r >= 0] for r in ref_idx]))
            rows = _rows_of(b, need, n_pre, kv_new)
            c_sel, s_sel = oracle.quantize_fp4(rows)
            where = {int(p): i for i, p in enumerate(need)}
            for g in range(G):
                l = int(first_layer[g])
                local = np.array([where[int(p)] if p >= 0 else -1 for p in ref_idx[g]], dtype=np.int64)
                ref = oracle.sparse_attention(q_bits[g][b], c_sel, s_sel, local, ring[l], W)
                if np.array_equal(gidx[g], ref_idx[g]):
                    out = wl.out[l][b:b + 1]
                    checked["attn_group"] += 1
                else:                           # tie-band selection difference
                    out = attn_with_oracle_idx(wl.q[l][b], codes[b], scales[b], ref_idx[g], wl.swa[l][b], W)
                    checked["attn_oracle_idx"] += 1
                try:
                    check_attn(out, ref[None])
                except AssertionError as e:
                    raise AssertionError(f"step {step}, sequence {b}, group {g}: {e}") from None
        checked["steps"] += 1

    for step in range(cfg.steps):
        wl.step()
        if step in CHECK_STEPS:
            torch.cuda.synchronize()
            check(step)
    assert checked["steps"] == len(CHECK_STEPS)
    assert checked["attn_group"] + checked["attn_oracle_idx"] == len(CHECK_STEPS) * len(SAMPLE) * G
    assert checked["attn_group"] >= len(CHECK_STEPS) * len(SAMPLE) * G // 2, checked


def _reindex_with_pool(qI_b, w_b, kI_b, n, pool_row, k):
    """The GPU Reindex of one sequence over a given pool (the oracle's)."""
    idx = torch.empty((1, k), dtype=torch.int32, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_INDEX_REINDEX, 1, kI_b.shape[0], k, len(pool_row), 64))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa2.csa2_index_reindex(qI_b[None], w_b[None], kI_b[None], torch.tensor([n], device=DEV),
                            torch.from_numpy(np.asarray(pool_row, dtype=np.int32)[None].copy()).to(DEV), k, idx, ws,
                            d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return idx.cpu().numpy()[0]
