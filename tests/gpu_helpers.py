"""Helpers shared by the GPU parity tests: host <-> device copies of the seeded inputs and
the acceptance rules the comparisons use."""
import numpy as np
import torch

DEV = "cuda"

# Attention output tolerance (max abs error): bf16 K/V with fp32 accumulation, and fp32.
ATOL_ATTN_BF16 = 2e-3
ATOL_ATTN_F32 = 1e-5
# Relative half-width of the top-k boundary band: a block whose oracle score lies within
# REL_TIE * |s_k| of the k-th best oracle score s_k may fall on either side.
REL_TIE = 1e-5


def to_dev(a: np.ndarray):
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(a).to(DEV)


def to_host(t) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def score_tolerance(q: np.ndarray, pooled: np.ndarray, n_rows: int, scale: float,
                    chain: int | None = None) -> np.ndarray:
    """Per-row bound on |fp32 score - fp64 score| for a length-n dot product accumulated in
    fp32 with at most ``chain`` roundings on any path: |err| <= chain * u * scale *
    sum|q_i z_i| with u = 2^-24, doubled for margin.  The decode kernel's longest path is
    n/128 fused multiply-adds per partial sum plus a 7-level add tree (chain = n/128 + 8);
    the tiled multi-query kernel accumulates serially (chain = n)."""
    n = q.shape[-1]
    if chain is None:
        chain = n / 128 + 8
    u = 2.0 ** -24
    absdot = np.abs(pooled[:n_rows].astype(np.float64)) @ np.abs(q.astype(np.float64)).reshape(-1)
    return 2.0 * chain * u * scale * absdot + 1e-30


def check_topk(gpu_blocks: np.ndarray, gpu_count: int, oracle_scores: np.ndarray, n_full: int,
               k_blk: int, band_abs=None):
    """GPU selection vs oracle scores: same count; every oracle-selected block outside the
    boundary band is selected, and no unselected block outside the band is.  Returns the
    number of blocks inside the band (0 means the sets must be identical).
    band_abs (optional, [n_full]): how far each block's GPU score may sit from the oracle's
    for a reason other than summation order (a bf16 cache value rounded the other way);
    it widens the band by the block's own amount plus the k-th block's."""
    k = min(k_blk, n_full)
    assert gpu_count == k
    sel = np.sort(gpu_blocks[:gpu_count].astype(np.int64))
    assert np.all(np.diff(sel) > 0), "blocks must be ascending and distinct"
    assert k == 0 or (sel[0] >= 0 and sel[-1] < n_full)
    if k == 0:
        return 0
    s = np.nan_to_num(oracle_scores[:n_full], nan=-np.inf)
    order = np.lexsort((np.arange(n_full), -s))
    s_k = s[order[k - 1]]
    if np.isfinite(s_k):
        extra = 0.0 if band_abs is None else band_abs[:n_full] + band_abs[order[k - 1]]
        band = np.abs(s - s_k) <= REL_TIE * abs(s_k) + extra
    else:
        band = s == s_k
    want = np.zeros(n_full, bool)
    want[order[:k]] = True
    got = np.zeros(n_full, bool)
    got[sel] = True
    bad = (want != got) & ~band
    assert not bad.any(), f"blocks differ outside the tie band: {np.flatnonzero(bad)[:10]}"
    return int(band.sum())
