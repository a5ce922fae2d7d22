"""Bounded device waits: a kernel whose signal never comes reports
CSA2_ERR_TIMEOUT through d_status, releases what it holds and returns, and
the next normal call on the same stream is correct.

The failure is made on purpose but without faulting the GPU: the test hook
csa2_debug_set_fault makes the named kernel's producers withhold the signal
of their last tile, and shortens every device wait to a few milliseconds, so
the consumers' waits run out. Nothing traps, faults or hangs."""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp4_kv_cache_06_b300 import csa2
from tests._parity import bits16, check_attn

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT = 5                                   # CSA2_ERR_TIMEOUT
SHORT_WAIT_NS = 20_000_000                    # 20 ms


class _fault:
    def __init__(self, what):
        self.what = what

    def __enter__(self):
        csa2.debug_set_fault(self.what, SHORT_WAIT_NS)

    def __exit__(self, *exc):
        csa2.debug_set_fault(csa2.FAULT_NONE, 0)


def _attn_case(B, H=64, k=512, n=3000, W=128, seed=31):
    kv = synth.normal_bf16((B, n, 512), seed=seed, stream="kv").to(DEV)
    codes = torch.empty((B, n, 256), dtype=torch.uint8, device=DEV)
    scales = torch.empty((B, n, 32), dtype=torch.uint8, device=DEV)
    csa2.csa2_quantize_kv_fp4(kv, codes, scales)
    rng = np.random.default_rng(seed)
    idx = np.stack([np.sort(rng.permutation(n)[:k]) for _ in range(B)]).astype(np.int32)
    q = synth.normal_bf16((B, H, 512), seed=seed, stream="q").to(DEV)
    swa = synth.normal_bf16((B, W, 512), seed=seed, stream="swa").to(DEV)
    swa_len = torch.full((B,), W, dtype=torch.int32, device=DEV)
    return kv, codes, scales, torch.from_numpy(idx).to(DEV), q, swa, swa_len


@pytest.mark.parametrize("B", [2, 80])
def test_attention_wait_runs_out_and_next_call_is_correct(B):
    """B = 2 runs split-K (one key tile per CTA, plus the merge kernel);
    B = 80 runs unsplit CTAs of ten key tiles each."""
    H, k, W = 64, 512, 128
    kv, codes, scales, idx, q, swa, swa_len = _attn_case(B)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_SPARSE_ATTN, B, 0, k, 2048, H))
    ref_out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV)
    csa2.csa2_sparse_attn(q, codes, scales, idx, swa, swa_len, ref_out, ws)
    torch.cuda.synchronize()

    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((B, H, 512), 3.0, dtype=torch.bfloat16, device=DEV)
    with _fault(csa2.FAULT_ATTN):
        csa2.csa2_sparse_attn(q, codes, scales, idx, swa, swa_len, out, ws, d_status=st)
        torch.cuda.synchronize()
    assert st.item() == TIMEOUT

    # the context is healthy: the same call again gives the same (correct) result
    st.zero_()
    again = torch.empty_like(ref_out)
    csa2.csa2_sparse_attn(q, codes, scales, idx, swa, swa_len, again, ws, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(again, ref_out)
    b = B - 1
    c, s = oracle.quantize_fp4(bits16(kv)[b])
    ref = oracle.sparse_attention(bits16(q)[b], c, s, idx.cpu().numpy()[b], bits16(swa)[b], W)
    check_attn(again[b:b + 1], ref[None])


def test_layer_group_attention_wait_runs_out_then_recovers():
    """The fault inside a whole Full + 3 Reuse group call (indexer, Top-K and
    the four layers' attention in one launch): the group reports the timeout
    and the next group call on the stream is correct."""
    B, n, H, H_I, d_I, k, W = 4, 4096, 64, 8, 128, 512, 128
    seed = 41
    kv = synth.normal_bf16((B, n, 512), seed, "kv").to(DEV)
    kI = synth.indexer_keys_e4m3((B, n, d_I), seed).to(DEV)
    qI = synth.normal_e4m3((B, H_I, d_I), seed, "qI").to(DEV)
    w = synth.uniform_f32((B, H_I), seed, "w").to(DEV)
    qs = [synth.normal_bf16((B, H, 512), seed, "q", sub=l).to(DEV) for l in range(4)]
    swas = [synth.normal_bf16((B, W, 512), seed, "swa", sub=l).to(DEV) for l in range(4)]
    codes = torch.empty((B, n, 256), dtype=torch.uint8, device=DEV)
    scales = torch.empty((B, n, 32), dtype=torch.uint8, device=DEV)
    csa2.csa2_quantize_kv_fp4(kv, codes, scales)
    nt = torch.full((B,), n, dtype=torch.int64, device=DEV)
    swa_len = torch.full((B,), W, dtype=torch.int32, device=DEV)
    idx = torch.empty((B, k), dtype=torch.int32, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_LAYER_GROUP, B, n, k, 2048, H))

    def run(outs, st=None):
        csa2.csa2_layer_group(csa2.MODE_FULL, nt, n, codes, scales, kI, qI, w, idx, qs, swas, swa_len, outs, ws,
                              d_status=st)

    ref_outs = [torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    run(ref_outs)
    torch.cuda.synchronize()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = [torch.empty_like(o) for o in ref_outs]
    with _fault(csa2.FAULT_ATTN):
        run(outs, st)
        torch.cuda.synchronize()
    assert st.item() == TIMEOUT
    st.zero_()
    run(outs, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for a, r in zip(outs, ref_outs):
        assert torch.equal(a, r)


def test_full_scan_wait_runs_out_and_next_call_is_correct():
    """The TMA-fed Full indexer scan: its producer withholds the second key
    tile of every CTA, the MMA warps' wait on it runs out, and the next scan
    on the stream reproduces the scores of a normal call."""
    B, n, H_I, d_I = 4, 32768, 8, 128
    seed = 51
    kI = synth.indexer_keys_e4m3((B, n, d_I), seed).to(DEV)
    qI = synth.normal_e4m3((B, H_I, d_I), seed, "qI").to(DEV)
    w = synth.uniform_f32((B, H_I), seed, "w").to(DEV)
    nt = torch.full((B,), n, dtype=torch.int64, device=DEV)
    ref = torch.empty((B, n), dtype=torch.float32, device=DEV)
    csa2.csa2_index_scores(qI, w, kI, nt, n, ref)
    torch.cuda.synchronize()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = torch.zeros_like(ref)
    with _fault(csa2.FAULT_SCAN):
        csa2.csa2_index_scores(qI, w, kI, nt, n, got, d_status=st)
        torch.cuda.synchronize()
    assert st.item() == TIMEOUT
    st.zero_()
    csa2.csa2_index_scores(qI, w, kI, nt, n, got, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(got, ref)
    b = 2
    o = oracle.indexer_scores(qI.cpu().numpy()[b], w.cpu().numpy()[b], kI.cpu().numpy()[b, :2048])
    np.testing.assert_allclose(got.cpu().numpy()[b, :2048], o, rtol=2e-6, atol=1e-6)


def test_prefill_gemm_wait_runs_out_and_next_call_is_correct():
    """The tcgen05 FP8 prefill indexer GEMM: its TMA producer withholds the
    second entry tile of every CTA, the MMA issuer's wait runs out, the CTA
    releases its tensor memory, and the next call is correct."""
    Q, n_keys = 1024, 8192
    seed = 52
    kI = synth.indexer_keys_e4m3((n_keys, 128), seed).to(DEV)
    qI = synth.normal_e4m3((Q, 8, 128), seed, "qI").to(DEV)
    w = synth.uniform_f32((Q, 8), seed, "w").to(DEV)
    ref = torch.empty((Q, n_keys), dtype=torch.float32, device=DEV)
    csa2.csa2_prefill_index_scores(qI, w, kI, ref)
    torch.cuda.synchronize()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = torch.zeros_like(ref)
    with _fault(csa2.FAULT_PREFILL):
        csa2.csa2_prefill_index_scores(qI, w, kI, got, d_status=st)
        torch.cuda.synchronize()
    assert st.item() == TIMEOUT
    st.zero_()
    csa2.csa2_prefill_index_scores(qI, w, kI, got, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(got, ref)
    qq = 700
    o = oracle.indexer_scores(qI.cpu().numpy()[qq], w.cpu().numpy()[qq], kI.cpu().numpy())
    np.testing.assert_allclose(got.cpu().numpy()[qq], o, rtol=2e-6, atol=1e-6)


def test_fault_hook_rejects_bad_arguments():
    with pytest.raises(csa2.Csa2Error, match="INVALID_ARG"):
        csa2.debug_set_fault(99, 0)
    with pytest.raises(csa2.Csa2Error, match="INVALID_ARG"):
        csa2.debug_set_fault(csa2.FAULT_ATTN, -1)
    csa2.debug_set_fault(csa2.FAULT_NONE, 0)
