"""GPU parity of the cache writers (FP4 quantise/append, indexer-K append with
block means, SWA ring append) against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp4_kv_cache_06_b300 import csa2
from tests._parity import bits16, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _quant_gpu(x_bits_np, n_cap=None, pos=None):
    x = torch.from_numpy(x_bits_np.view(np.int16)).view(torch.bfloat16).to(DEV)
    B, rows, _ = x.shape
    n_cap = rows if n_cap is None else n_cap
    codes = torch.full((B, n_cap, 256), 0xAB, dtype=torch.uint8, device=DEV)
    scales = torch.full((B, n_cap, 32), 0xAB, dtype=torch.uint8, device=DEV)
    p = None if pos is None else torch.tensor(pos, dtype=torch.int64, device=DEV)
    csa2.csa2_quantize_kv_fp4(x, codes, scales, pos=p)
    torch.cuda.synchronize()
    return u8(codes), u8(scales)


def test_quantize_every_bf16_value_bit_exact():
    """Every finite bf16 pattern as a group member beside a fixed group amax."""
    all_bits = np.arange(65536, dtype=np.uint16)
    vals = oracle.bf16_bits_to_f64(all_bits)
    for amax_bits in (0x3F80, 0x4040, 0x3E2A, 0x4380, 0x3B80, 0x4500, 0x3C00, 0x3A00, 0x7F7F, 0x0080):
        amax = oracle.bf16_bits_to_f64(np.array([amax_bits], dtype=np.uint16))[0]
        members = all_bits[np.isfinite(vals) & (np.abs(vals) <= amax)]
        m = members.size
        rows = (m + 31) // 32
        g = np.zeros((rows * 32, 16), dtype=np.uint16)
        g[:, 0] = amax_bits
        g[:m, 1] = members
        g[:m, 2] = members[::-1]
        x = g.reshape(1, rows, 512)
        c_gpu, s_gpu = _quant_gpu(x)
        c_ref, s_ref = oracle.quantize_fp4(x)
        np.testing.assert_array_equal(s_gpu, s_ref)
        np.testing.assert_array_equal(c_gpu, c_ref)


def test_quantize_golden_groups_and_edge_rows():
    from tests._golden import rows as golden_rows
    groups = []
    for _, xs, _, _ in golden_rows("fp4_quant_examples.txt"):
        groups.append(np.array([float(v) for v in xs.split()], dtype=np.float32))
    g = np.zeros((32, 16), dtype=np.float32)
    g[:len(groups)] = np.stack(groups)
    g[10] = -0.0                     # all negative zeros
    g[11] = 1e-30                    # deep underflow
    g[12] = np.float32(3.0e38)       # saturating scale
    g[13, ::2] = -448.0
    bits = (g.view(np.uint32) >> 16).astype(np.uint16).reshape(1, 1, 512)
    c_gpu, s_gpu = _quant_gpu(bits)
    c_ref, s_ref = oracle.quantize_fp4(bits)
    np.testing.assert_array_equal(s_gpu, s_ref)
    np.testing.assert_array_equal(c_gpu, c_ref)


def test_quantize_random_rows_at_positions_and_bounds():
    B, rows, n_cap = 3, 777, 2000
    x = synth.normal_bf16((B, rows, 512), seed=5, stream="kv")
    xb = bits16(x)
    pos = [0, 1000, 1223]            # the last sequence runs past n_cap for 0 rows (1223+777 = 2000)
    c_gpu, s_gpu = _quant_gpu(xb, n_cap=n_cap, pos=pos)
    for b in range(B):
        c_ref, s_ref = oracle.quantize_fp4(xb[b])
        np.testing.assert_array_equal(c_gpu[b, pos[b]:pos[b] + rows], c_ref)
        np.testing.assert_array_equal(s_gpu[b, pos[b]:pos[b] + rows], s_ref)
        untouched = np.ones(n_cap, bool)
        untouched[pos[b]:pos[b] + rows] = False
        assert np.all(c_gpu[b, untouched] == 0xAB)
    # rows beyond the capacity are skipped and reported, never written
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    xx = x[:1, :10].contiguous().to(DEV)
    codes = torch.full((1, 16, 256), 0xAB, dtype=torch.uint8, device=DEV)
    scales = torch.full((1, 16, 32), 0xAB, dtype=torch.uint8, device=DEV)
    csa2.csa2_quantize_kv_fp4(xx, codes, scales, pos=torch.tensor([10], dtype=torch.int64, device=DEV), d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 6
    c_ref, _ = oracle.quantize_fp4(bits16(xx)[0])
    np.testing.assert_array_equal(u8(codes)[0, 10:16], c_ref[:6])
    assert np.all(u8(codes)[0, :10] == 0xAB)


@pytest.mark.parametrize("d_I", [64, 128])
def test_indexer_append_and_block_means(d_I):
    B, n_cap = 2, 300
    k_all = synth.indexer_keys_e4m3((B, n_cap, d_I), seed=3, bias_prob=0.1)
    kI = torch.zeros((B, n_cap, d_I), dtype=torch.uint8, device=DEV)
    kbar = torch.zeros((B, (n_cap + 7) // 8, d_I), dtype=torch.uint8, device=DEV)
    # bulk append of 100 rows, then single-row appends, then a 37-row append
    steps = [(0, 100), (100, 1), (101, 1), (102, 5), (107, 37), (144, 1)]
    for p, r in steps:
        csa2.csa2_append_indexer_k(k_all[:, p:p + r].contiguous().to(DEV), kI, kbar,
                                   pos=torch.full((B,), p, dtype=torch.int64, device=DEV))
        torch.cuda.synchronize()
        n_now = p + r
        kb = u8(kbar)
        for b in range(B):
            ref = oracle.block_means(u8(k_all)[b], n_now)
            np.testing.assert_array_equal(kb[b, :ref.shape[0]], ref)
    np.testing.assert_array_equal(u8(kI)[:, :145], u8(k_all)[:, :145])
    # bulk recompute from an in-place cache matches too
    kbar2 = torch.zeros_like(kbar)
    n = torch.tensor([145, 77], dtype=torch.int64, device=DEV)
    csa2.csa2_block_means(kI, n, kbar2, n_max=145)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(u8(kbar2)[0, :19], oracle.block_means(u8(k_all)[0], 145))
    np.testing.assert_array_equal(u8(kbar2)[1, :10], oracle.block_means(u8(k_all)[1], 77))


def test_swa_append_ring_slot():
    B, W = 3, 128
    swa = torch.zeros((B, W, 512), dtype=torch.bfloat16, device=DEV)
    x = synth.normal_bf16((B, 512), seed=1, stream="swa_new").to(DEV)
    pos = torch.tensor([0, 127, 1000003], dtype=torch.int64, device=DEV)
    csa2.csa2_append_swa(x, pos, swa)
    torch.cuda.synchronize()
    for b, p in enumerate([0, 127, 1000003]):
        assert torch.equal(swa[b, p % W], x[b])
        assert int((swa[b].abs().sum(-1) > 0).sum()) == 1


@pytest.mark.parametrize("d_I,L", [(128, 4), (64, 1), (128, 20)])
def test_append_step_matches_individual_appends(d_I, L):
    """The fused one-launch append equals the three separate appends, bit for bit."""
    B, n_cap, W = 5, 64, 128
    pos_list = [0, 7, 8, 13, 63]
    pos = torch.tensor(pos_list, dtype=torch.int64, device=DEV)
    base_kI = synth.indexer_keys_e4m3((B, n_cap, d_I), seed=8).to(DEV)
    kv_new = synth.normal_bf16((B, 512), seed=8, stream="kv_new").to(DEV)
    kI_new = synth.indexer_keys_e4m3((B, 1, d_I), seed=9).to(DEV)[:, 0].contiguous()
    swa_new = [synth.normal_bf16((B, 512), seed=8, stream="swa_new", sub=l).to(DEV) for l in range(L)]

    def caches():
        kI = base_kI.clone()
        kbar = torch.zeros((B, n_cap // 8, d_I), dtype=torch.uint8, device=DEV)
        codes = torch.zeros((B, n_cap, 256), dtype=torch.uint8, device=DEV)
        scales = torch.zeros((B, n_cap, 32), dtype=torch.uint8, device=DEV)
        swa = [torch.zeros((B, W, 512), dtype=torch.bfloat16, device=DEV) for _ in range(L)]
        return kI, kbar, codes, scales, swa

    a = caches()
    csa2.csa2_append_step(kv_new, kI_new, swa_new, a[4], pos, a[2], a[3], a[0], a[1])
    b = caches()
    csa2.csa2_quantize_kv_fp4(kv_new[:, None].contiguous(), b[2], b[3], pos=pos)
    csa2.csa2_append_indexer_k(kI_new[:, None].contiguous(), b[0], b[1], pos=pos)
    for l in range(L):
        csa2.csa2_append_swa(swa_new[l], pos, b[4][l])
    torch.cuda.synchronize()
    for x, y in zip(a[:4], b[:4]):
        assert torch.equal(x, y)
    for x, y in zip(a[4], b[4]):
        assert torch.equal(x, y)
    # and the block means equal the oracle's over the appended cache
    kI_np = u8(a[0])
    for i, p in enumerate(pos_list):
        ref = oracle.block_means(kI_np[i], p + 1)
        np.testing.assert_array_equal(u8(a[1])[i, p // 8], ref[p // 8])


def test_swa_ring_export_and_restore():
    """Rings filled by per-token appends: the export is the window in token
    order (oracle), and restoring it into empty rings gives back the same
    rings and window lengths."""
    B, W, L = 3, 128, 2
    n = np.array([300, 50, 128], dtype=np.int64)
    rows = [synth.normal_bf16((B, int(n.max()), 512), seed=5, stream="swa", sub=l) for l in range(L)]
    rings = [torch.zeros((B, W, 512), dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    for t in range(int(n.max())):
        live = torch.from_numpy((t < n).astype(np.int64)).to(DEV)
        pos = torch.where(live > 0, torch.full_like(live, t), torch.full_like(live, -1))
        for l in range(L):
            for b in range(B):
                if t < n[b]:
                    csa2.csa2_append_swa(rows[l][b:b + 1, t].to(DEV), pos[b:b + 1], rings[l][b:b + 1])
    n_d = torch.from_numpy(n).to(DEV)
    out = [torch.full((B, W, 512), 7.0, dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    csa2.csa2_swa_export(rings, n_d, out)
    back = [torch.zeros((B, W, 512), dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    swa_len = torch.zeros(B, dtype=torch.int32, device=DEV)
    csa2.csa2_swa_restore(out, n_d, back, swa_len_out=swa_len)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(swa_len.cpu().numpy(), np.minimum(n, W))
    for l in range(L):
        ob, bb = bits16(out[l]), bits16(back[l])
        for b in range(B):
            c = min(int(n[b]), W)
            window = bits16(rows[l])[b, int(n[b]) - c:int(n[b])]
            np.testing.assert_array_equal(ob[b, :c], window)
            assert (ob[b, c:] == 0).all()
            np.testing.assert_array_equal(bb[b], oracle.swa_ring_after(bits16(rows[l])[b], int(n[b]), W))
            np.testing.assert_array_equal(bits16(rings[l])[b], bb[b])
