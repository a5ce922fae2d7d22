"""GPU checks of decoding at compression ratio 2 (the encoder's cadence):
every token appends each layer's SWA row, but a compressed main-KV entry is
appended only when its second token arrives, at entry (t + 1) / 2 - 1, and
the token sees (t + 1) / 2 entries. The step writes those counts itself, so
the layer group that follows runs on them."""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp4_kv_cache_06_b300 import csa2
from tests._parity import bits16, check_attn, check_topk, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_ratio2_cadence_and_group_on_device_counts():
    B, n_cap, W, H, L, ratio = 2, 3000, 128, 64, 2, 2
    t0 = np.array([3997, 4002], dtype=np.int64)          # token positions of the first step
    n0 = (t0 + 1) // ratio                                # entries already cached
    seed = 77
    kv = synth.normal_bf16((B, n_cap, 512), seed=seed, stream="kv")
    codes = torch.zeros((B, n_cap, 256), dtype=torch.uint8, device=DEV)
    scales = torch.zeros((B, n_cap, 32), dtype=torch.uint8, device=DEV)
    for b in range(B):
        csa2.csa2_quantize_kv_fp4(kv[b:b + 1, :n0[b]].to(DEV), codes[b:b + 1], scales[b:b + 1])
    kI = synth.indexer_keys_e4m3((B, n_cap, 128), seed=seed, bias_prob=0.05)
    kI_d = torch.zeros((B, n_cap, 128), dtype=torch.uint8, device=DEV)
    for b in range(B):
        kI_d[b, :n0[b]] = kI[b, :n0[b]].to(DEV)
    kbar = torch.zeros((B, (n_cap + 7) // 8, 128), dtype=torch.uint8, device=DEV)
    csa2.csa2_block_means(kI_d, torch.from_numpy(n0).to(DEV), kbar, n_max=n_cap)
    swa = [torch.zeros((B, W, 512), dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    swa_host = [np.zeros((B, W, 512), dtype=np.uint16) for _ in range(L)]
    pos = torch.from_numpy(t0.copy()).to(DEV)
    n_vis = torch.zeros(B, dtype=torch.int64, device=DEV)
    swa_len = torch.zeros(B, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    steps = 6
    for i in range(steps):
        t = t0 + i
        e = (t + 1) // ratio - 1                          # entry that completes at t (if (t+1) % 2 == 0)
        kv_new = kv[np.arange(B), np.minimum(e, n_cap - 1)].contiguous()
        kI_new = kI[np.arange(B), np.minimum(e, n_cap - 1)].contiguous()
        swa_new = [synth.normal_bf16((B, 512), seed=seed, stream="swa_new", sub=100 * i + l) for l in range(L)]
        before = codes.clone()
        csa2.csa2_append_step_ratio(kv_new.to(DEV), kI_new.to(DEV), [x.to(DEV) for x in swa_new], swa, pos, ratio,
                                    codes, scales, kI_d, kbar, n_vis_out=n_vis, swa_len_out=swa_len, d_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        np.testing.assert_array_equal(n_vis.cpu().numpy(), (t + 1) // ratio)
        np.testing.assert_array_equal(swa_len.cpu().numpy(), np.minimum(t + 1, W))
        for b in range(B):
            changed = np.nonzero((codes[b] != before[b]).any(dim=1).cpu().numpy())[0]
            if (t[b] + 1) % ratio == 0:
                c, s = oracle.quantize_fp4(bits16(kv_new)[b:b + 1])
                np.testing.assert_array_equal(u8(codes)[b, e[b]], c[0])
                np.testing.assert_array_equal(u8(scales)[b, e[b]], s[0])
                assert set(changed.tolist()) <= {int(e[b])}
            else:
                assert changed.size == 0
            for l in range(L):
                swa_host[l][b, t[b] % W] = bits16(swa_new[l])[b]
        pos += 1
    # the group of the last token runs on the counts the step wrote
    t_last = t0 + steps - 1
    nv = (t_last + 1) // ratio
    qI = synth.normal_e4m3((B, 8, 128), seed=seed, stream="qI")
    w = synth.uniform_f32((B, 8), seed=seed, stream="w")
    qs = [synth.normal_bf16((B, H, 512), seed=seed, stream="q", sub=l) for l in range(L)]
    outs = [torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    idx = torch.empty((B, 512), dtype=torch.int32, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_LAYER_GROUP, B, n_cap, 512, 2048, H))
    csa2.csa2_layer_group(csa2.MODE_FULL, n_vis, int(nv.max()), codes, scales, kI_d, qI.to(DEV), w.to(DEV), idx,
                          [q.to(DEV) for q in qs], swa, swa_len, outs, ws, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    gi = idx.cpu().numpy()
    compared = 0
    for b in range(B):
        kb = u8(kI)[b]
        ref_idx, ref_s = oracle.full_topk(u8(qI)[b], w.numpy()[b], kb, int(nv[b]), 512)
        check_topk(gi[b], ref_idx, ref_s, np.arange(int(nv[b])), 512)
        if not np.array_equal(gi[b], ref_idx):
            continue
        c, s = oracle.quantize_fp4(bits16(kv)[b])
        for l in range(L):
            ref = oracle.sparse_attention(bits16(qs[l])[b], c, s, ref_idx, swa_host[l][b], W)
            check_attn(outs[l][b:b + 1], ref[None])
            compared += 1
    assert compared >= L
