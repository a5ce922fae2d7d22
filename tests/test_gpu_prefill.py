"""GPU parity of the prefill path: the tcgen05 FP8 indexer GEMM and the
encoder group (Full + Reuse) over a chunk of queries with the causal rule,
against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp4_kv_cache_06_b300 import csa2
from tests._parity import attn_with_oracle_idx, bits16, check_attn, check_topk, u8, vmax_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("Q,n", [(32, 128), (100, 1000), (64, 4097), (7, 300)])
def test_prefill_index_scores_match_oracle(Q, n):
    qI = synth.normal_e4m3((Q, 8, 128), seed=Q, stream="qI")
    w = synth.uniform_f32((Q, 8), seed=Q, stream="w")
    kI = synth.indexer_keys_e4m3((n, 128), seed=n, bias_prob=0.05)
    stride = n + 3
    scores = torch.full((Q, stride), -5.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa2.csa2_prefill_index_scores(qI.to(DEV), w.to(DEV), kI.to(DEV), scores, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    s = scores.cpu().numpy()
    for q in range(Q):
        ref = oracle.indexer_scores(u8(qI)[q], w.numpy()[q], u8(kI))
        np.testing.assert_allclose(s[q, :n], ref, rtol=2e-6, atol=1e-6)
    assert np.all(s[:, n:] == -5.0)


@pytest.mark.parametrize("p0,Q,n_keys", [(2000, 48, 1024), (60, 40, 64)])
def test_prefill_group_causal(p0, Q, n_keys):
    """Queries at tokens p0..p0+Q-1, ratio 2: query p sees floor((p+1)/2) entries
    and the SWA rows of tokens max(0, p-127)..p. Full + 1 Reuse layer."""
    H, W, k, L = 64, 128, 512, 2
    kv = synth.normal_bf16((n_keys, 512), seed=p0, stream="kv").to(DEV)
    codes = torch.empty((n_keys, 256), dtype=torch.uint8, device=DEV)
    scales = torch.empty((n_keys, 32), dtype=torch.uint8, device=DEV)
    csa2.csa2_quantize_kv_fp4(kv[None], codes[None], scales[None])
    kI = synth.indexer_keys_e4m3((n_keys, 128), seed=p0).to(DEV)
    qI = synth.normal_e4m3((Q, 8, 128), seed=p0, stream="qI").to(DEV)
    w = synth.uniform_f32((Q, 8), seed=p0, stream="w").to(DEV)
    pos = np.arange(p0, p0 + Q)
    n_vis = np.minimum(oracle.prefill_visible(pos, 2), n_keys)
    swa_len = np.minimum(pos + 1, W).astype(np.int32)
    qs = [synth.normal_bf16((Q, H, 512), seed=p0, stream="q", sub=l).to(DEV) for l in range(L)]
    swas = [synth.normal_bf16((Q + W - 1, 512), seed=p0, stream="swa", sub=l).to(DEV) for l in range(L)]
    outs = [torch.empty((Q, H, 512), dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    idx = torch.empty((Q, k), dtype=torch.int32, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_PREFILL_GROUP, Q, n_keys, k, 0, H))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa2.csa2_prefill_group(torch.from_numpy(n_vis).to(DEV), codes, scales, kI, qI, w, idx, qs, swas,
                            torch.from_numpy(swa_len).to(DEV), outs, ws, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    c, s = oracle.quantize_fp4(bits16(kv))
    gi = idx.cpu().numpy()
    compared = {"group": 0, "oracle_idx": 0}
    for q in range(Q):
        ref_idx, ref_s = oracle.full_topk(u8(qI)[q], w.cpu().numpy()[q], u8(kI), int(n_vis[q]), k)
        check_topk(gi[q], ref_idx, ref_s, np.arange(int(n_vis[q])), k)
        toks = oracle.prefill_swa_rows(pos[q], W)
        rows = toks - (p0 - W + 1)
        for l in range(L):
            sw = bits16(swas[l])[rows]
            ref = oracle.sparse_attention(bits16(qs[l])[q], c, s, ref_idx, sw, len(rows))
            sel = ref_idx[ref_idx >= 0]
            few = len(sel) + len(rows) < 300
            vm = vmax_of(np.concatenate([oracle.dequant_fp4(c[sel], s[sel]), oracle.bf16_bits_to_f64(sw)])) if few else None
            if np.array_equal(gi[q], ref_idx):
                check_attn(outs[l][q:q + 1], ref[None], vmax=vm)
                compared["group"] += 1
            else:
                # a tie-band difference in the selection: the same row's
                # attention over the oracle's entries
                got = attn_with_oracle_idx(qs[l][q], codes, scales, ref_idx, swas[l][torch.from_numpy(rows).to(DEV)], W)
                check_attn(got, ref[None], vmax=vm)
                compared["oracle_idx"] += 1
    # every query and layer was compared, and most through the group's own output
    assert compared["group"] + compared["oracle_idx"] == Q * L
    assert compared["group"] >= Q * L // 2, compared
