"""csa2_topk_noalloc against csa2_topk and the oracle, through the C ABI.

The no-workspace entry point exists for callers that cannot allocate
device memory (plugin hooks where allocation is forbidden, allocation-free
serving loops, C callers without an allocator). It must select exactly
what the workspace version selects, and a second call must not be
disturbed by what the first one left in the shared device scratch.
This file is collected last so that a failure here does not hide others.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_06_b300 import csa2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _with_workspace(scores, n, n_max, k, cand_pos=None):
    B = scores.shape[0]
    idx = torch.empty((B, k), dtype=torch.int32, device=DEV)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_TOPK, B, n_max, k))
    csa2.csa2_topk(scores, n, n_max, k, idx, ws, cand_pos=cand_pos)
    return idx


def _without_workspace(scores, n, n_max, k, cand_pos=None):
    B = scores.shape[0]
    idx = torch.full((B, k), 12345, dtype=torch.int32, device=DEV)
    csa2.csa2_topk_noalloc(scores, n, n_max, k, idx, cand_pos=cand_pos)
    return idx


def test_noalloc_matches_workspace_version_on_two_calls():
    g = torch.Generator(device="cpu").manual_seed(5)
    # call 1: 40 rows of 70,000 scores with exact ties, ragged lengths
    s1 = torch.randint(0, 40, (40, 70000), generator=g).to(torch.float32).to(DEV)
    n1 = torch.randint(1, 70000, (40,), generator=g).to(torch.int64).to(DEV)
    n1[0] = 70000
    n1[1] = 100                       # fewer than k candidates
    a1 = _without_workspace(s1, n1, 70000, 512)
    b1 = _with_workspace(s1, n1, 70000, 512)
    # call 2: different shape and data, candidate positions with absent entries
    s2 = torch.randn((7, 16384), generator=g).to(DEV)
    cp = torch.randperm(10 ** 6, generator=g)[:7 * 16384].reshape(7, 16384).to(torch.int32)
    cp[torch.rand((7, 16384), generator=g) < 0.25] = -1
    cp = cp.to(DEV)
    a2 = _without_workspace(s2, None, 16384, 2048, cand_pos=cp)
    b2 = _with_workspace(s2, None, 16384, 2048, cand_pos=cp)
    torch.cuda.synchronize()
    assert torch.equal(a1, b1)
    assert torch.equal(a2, b2)
    for b, ref in _oracle_rows(s1, n1, 512, [0, 1, 17, 39]).items():
        np.testing.assert_array_equal(a1[b].cpu().numpy(), ref)
    for b, ref in _oracle_rows(s2, None, 2048, [0, 6], cand_pos=cp).items():
        np.testing.assert_array_equal(a2[b].cpu().numpy(), ref)
    # sanity: the selection is a sorted, -1 padded index list
    r = a1.cpu().numpy()[1]
    assert np.all(r[:100] == np.arange(100)) and np.all(r[100:] == -1)


def _oracle_rows(scores, n, k, rows, cand_pos=None):
    """The oracle's selection for a few rows (fp32 scores are exact in float64)."""
    s = scores.cpu().double().numpy()
    n_h = None if n is None else n.cpu().numpy()
    cp = None if cand_pos is None else cand_pos.cpu().numpy()
    out = {}
    for b in rows:
        m = s.shape[1] if n_h is None else int(n_h[b])
        pos = np.arange(m) if cp is None else cp[b, :m]
        out[b] = oracle.topk_select(s[b, :m], pos, k)
    return out


def test_noalloc_full_scratch_after_other_shapes():
    """Two more calls after differently shaped ones, at the row limit where the
    scratch is exactly full: long ragged rows (the chunk-table path, whose
    tables now start at offsets set by the new row count) and caller-given
    candidate positions with absent entries. Each is compared with csa2_topk
    and, on sampled rows, with the oracle."""
    g = torch.Generator(device="cpu").manual_seed(11)
    B, n_max, k = csa2.TOPK_NOALLOC_MAX_ROWS, 40000, 512
    # small call first, so the scratch holds another shape's leftovers
    s0 = torch.rand((3, 5000), generator=g).to(DEV)
    _without_workspace(s0, None, 5000, 64)
    s3 = torch.randint(0, 3000, (B, n_max), generator=g).to(torch.float32).to(DEV) / 7.0
    n3 = torch.randint(20000, n_max + 1, (B,), generator=g).to(torch.int64)
    n3[5] = 300                                        # fewer than k candidates
    n3[9] = n_max
    n3 = n3.to(DEV)
    a3 = _without_workspace(s3, n3, n_max, k)
    b3 = _with_workspace(s3, n3, n_max, k)
    cp = torch.randperm(10 ** 7, generator=g)[:B * n_max].reshape(B, n_max).to(torch.int32)
    cp[torch.rand((B, n_max), generator=g) < 0.3] = -1
    cp = cp.to(DEV)
    a4 = _without_workspace(s3, n3, n_max, k, cand_pos=cp)
    b4 = _with_workspace(s3, n3, n_max, k, cand_pos=cp)
    torch.cuda.synchronize()
    assert torch.equal(a3, b3)
    assert torch.equal(a4, b4)
    rows = [0, 5, 9, 33, B - 1]
    for b, ref in _oracle_rows(s3, n3, k, rows).items():
        np.testing.assert_array_equal(a3[b].cpu().numpy(), ref)
    for b, ref in _oracle_rows(s3, n3, k, rows, cand_pos=cp).items():
        np.testing.assert_array_equal(a4[b].cpu().numpy(), ref)


def test_noalloc_rejects_rows_beyond_its_scratch():
    s = torch.zeros((65, 10), dtype=torch.float32, device=DEV)
    idx = torch.empty((65, 4), dtype=torch.int32, device=DEV)
    with pytest.raises(csa2.Csa2Error, match="UNSUPPORTED_SHAPE"):
        csa2.csa2_topk_noalloc(s, None, 10, 4, idx)
