"""csa2_topk_noalloc against csa2_topk, through the C ABI.

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
    # sanity: the selection is a sorted, -1 padded index list
    r = a1.cpu().numpy()[1]
    assert np.all(r[:100] == np.arange(100)) and np.all(r[100:] == -1)


def test_noalloc_rejects_rows_beyond_its_scratch():
    s = torch.zeros((65, 10), dtype=torch.float32, device=DEV)
    idx = torch.empty((65, 4), dtype=torch.int32, device=DEV)
    with pytest.raises(csa2.Csa2Error, match="UNSUPPORTED_SHAPE"):
        csa2.csa2_topk_noalloc(s, None, 10, 4, idx)
