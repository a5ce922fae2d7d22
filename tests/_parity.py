"""Shared helpers of the GPU parity tests (conversions and comparison rules)."""
import numpy as np
import torch

TOPK_BAND = 1e-5          # relative tie band around the oracle's k-th score
ATTN_MAX_ABS = 2e-3       # bf16 attention output vs float64 oracle
ATTN_MEAN_ABS = 2e-4


def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (numpy, CPU)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def check_topk(gpu_idx, oracle_idx, oracle_scores, oracle_pos, k, band=TOPK_BAND):
    """Top-K parity: sorted ascending, -1 padded, equal sizes, equal sets except
    for positions whose oracle score lies within `band` (relative) of the
    oracle's k-th score."""
    g = np.asarray(gpu_idx, dtype=np.int64)
    o = np.asarray(oracle_idx, dtype=np.int64)
    gv, ov = g[g >= 0], o[o >= 0]
    assert np.all(g[len(gv):] == -1), "GPU index list is not -1 padded at the end"
    assert np.all(np.diff(gv) > 0), "GPU index list is not strictly ascending"
    assert len(gv) == len(ov), (len(gv), len(ov))
    diff = set(gv.tolist()) ^ set(ov.tolist())
    if not diff:
        return 0
    s_of = dict(zip(np.asarray(oracle_pos).tolist(), np.asarray(oracle_scores).tolist()))
    sk = np.sort(np.asarray([s_of[p] for p in ov.tolist()]))[0] if len(ov) >= k else None
    assert sk is not None, f"sets differ with fewer than k candidates: {sorted(diff)[:10]}"
    for p in diff:
        assert p in s_of, f"GPU picked a position that is not a candidate: {p}"
        assert abs(s_of[p] - sk) <= band * abs(sk), (p, s_of[p], sk)
    return len(diff)


# bf16 carries an 8-bit significand, so rounding to bf16 moves a value by
# up to 2^-8 of its magnitude (half an ulp just above a power of two).
# With few keys the weights p_j are large: rounding each p_j moves the
# output by up to 2^-8 * max_j |v_jd| per dim d, and rounding the output
# itself adds 2^-8 * |o_d|. The absolute bounds above assume hundreds of
# keys, where these errors average out; tests with few keys pass vmax
# (per-dim max |v| over the keys) to add these terms.
BF16_REL = 2.0 ** -8


def vmax_of(keys):
    """Per-dim max |v| over a [keys, d] float64 array (zeros if empty)."""
    keys = np.asarray(keys, dtype=np.float64).reshape(-1, np.shape(keys)[-1])
    return np.abs(keys).max(axis=0) if keys.shape[0] else np.zeros(keys.shape[1])


def check_attn(gpu_out, oracle_out, max_abs=ATTN_MAX_ABS, mean_abs=ATTN_MEAN_ABS, vmax=None):
    """max-abs / mean-abs parity of bf16 outputs against float64. The max-abs
    bound applies on top of the output format's own rounding: a correctly
    rounded bf16 output may sit half an ulp (up to 2^-8 |ref|) from the exact
    value, which alone reaches 2e-3 at |ref| ~ 0.5."""
    g = bf16_to_f64(gpu_out)
    r = np.asarray(oracle_out)
    d = np.abs(g - r)
    assert np.all(np.isfinite(g))
    extra = 0.0 if vmax is None else BF16_REL * np.asarray(vmax)
    bound = max_abs + BF16_REL * np.abs(r) + extra
    worst = np.argmax(d - np.broadcast_to(bound, d.shape))
    assert np.all(d <= bound), (f"abs err {d.flat[worst]:.3e} > bound {np.broadcast_to(bound, d.shape).flat[worst]:.3e} "
                                f"at |ref| {abs(r.flat[worst]):.4f} (gpu {g.flat[worst]:.6f}, max err {d.max():.3e}, "
                                f"mean err {d.mean():.3e}, max |ref| {np.abs(r).max():.3f})")
    # the mean is taken against the oracle rounded to bf16, so that the
    # output format's own rounding (2^-9 |ref| on average, which outgrows the
    # bound once |ref| is near 1, as with windows of repeated rows) is not
    # counted as error
    rb = torch.from_numpy(np.ascontiguousarray(r, dtype=np.float64)).to(torch.bfloat16).to(torch.float64).numpy()
    dm = np.abs(g - np.broadcast_to(rb, g.shape))
    mbound = mean_abs + (0.0 if vmax is None else float(np.mean(extra)))
    assert dm.mean() <= mbound, f"mean abs err {dm.mean():.3e} > {mbound:.3e} (vs unrounded {d.mean():.3e})"
    return float(d.max()), float(dm.mean())


def attn_with_oracle_idx(q_row, codes_seq, scales_seq, oracle_idx, swa_rows, W=128):
    """Sparse attention for one row on the GPU with the oracle's Top-K as its
    index list (an input that comes from the oracle, never the reverse).

    Used where the kernel's own selection legitimately differs from the
    oracle's inside the tie band: the attention of that row is then still
    compared, over the entries the oracle chose. q_row [H][512] bf16;
    codes_seq [n][256], scales_seq [n][32] u8 (device); oracle_idx [k] ints
    (-1 padded); swa_rows [s][512] bf16 with s <= W. Returns [1][H][512]."""
    from fp4_kv_cache_06_b300 import csa2
    dev = codes_seq.device
    H = q_row.shape[0]
    k = len(oracle_idx)
    s = swa_rows.shape[0]
    swa = torch.zeros((1, W, 512), dtype=torch.bfloat16, device=dev)
    swa[0, :s] = swa_rows.to(dev)
    idx = torch.from_numpy(np.asarray(oracle_idx, dtype=np.int32)[None].copy()).to(dev)
    out = torch.empty((1, H, 512), dtype=torch.bfloat16, device=dev)
    ws = csa2.alloc_workspace(csa2.workspace_size(csa2.OP_SPARSE_ATTN, 1, 0, k, 2048, H), dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    csa2.csa2_sparse_attn(q_row[None].to(dev), codes_seq[None], scales_seq[None], idx, swa,
                          torch.tensor([s], dtype=torch.int32, device=dev), out, ws, d_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out
