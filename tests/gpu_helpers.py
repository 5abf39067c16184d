"""Helpers shared by the GPU parity tests: host <-> device copies of the seeded inputs and
the acceptance rules the comparisons use."""
import numpy as np
import torch

import qsa_synth
from oracle import oracle

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


# ------------------------------------------------------------------ bf16 pooled storage
# The kernel's fp32 pooled value: pooling, an RMS norm over d values, a weight and a
# rotation, each a few roundings of 2^-24; 2^-17 of the pair's magnitude bounds them.
BF16_FLIP_REL = 2.0 ** -17


def pooled_f64(inp, shape, n_ctx, rows):
    """The oracle's exact (fp64, unrounded) pooled rows."""
    H, d = shape.H_idx, shape.d_idx
    return np.stack([oracle.pool_row_f64(inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps,
                                         shape.rope_base, b) for b in rows])


def bf16_delta(z, d):
    """Per element: the bound on the kernel's fp32 error, BF16_FLIP_REL of the magnitude of
    the rotation pair (dims i and i + d/2 of a head) the element belongs to."""
    zz = z.reshape(z.shape[0], -1, 2, d // 2)
    pair = np.hypot(zz[:, :, 0, :], zz[:, :, 1, :])
    return BF16_FLIP_REL * np.concatenate([pair, pair], axis=-1).reshape(z.shape)


def _bf16_mag(bits):
    return qsa_synth.bf16_bits_to_f32((bits & 0x7FFF).astype(np.uint16)).astype(np.float64)


def check_bf16_rows(got_bits, want_bits, z, d):
    """Each stored bf16 value must be the rounding of some value within delta of the exact
    one: |z| inside the value's rounding interval widened by delta (the sign may differ
    only within delta of zero).  Returns how many values differ from the oracle's."""
    delta = bf16_delta(z, d)
    mag = got_bits & 0x7FFF
    g = _bf16_mag(got_bits)
    lo = np.where(mag > 0, 0.5 * (_bf16_mag(np.maximum(mag, 1) - 1) + g), 0.0)
    hi = 0.5 * (g + _bf16_mag(mag + 1))
    a = np.abs(z)
    sign_ok = ((got_bits >> 15) == (z < 0)) | (mag == 0)
    ok = np.where(sign_ok, (a >= lo - delta) & (a <= hi + delta), g + a <= delta)
    assert ok.all(), f"{int((~ok).sum())} stored values are not a rounding of the exact value"
    return int((got_bits != want_bits).sum())


def flip_band(q, z, d, scale):
    """Per row: how far the kernel's stored values can move a score from the oracle's (both
    roundings of values within delta of the exact one): one bf16 step plus 2 delta at an
    element whose exact value is within delta of a rounding midpoint or of zero."""
    delta = bf16_delta(z, d)
    a = np.abs(z)
    ulp = np.exp2(np.floor(np.log2(np.where(a > 0, a, 1.0))) - 7)
    mid = (np.floor(a / ulp) + 0.5) * ulp
    risky = (np.abs(a - mid) <= delta) | (a <= 2 * delta)
    return scale * ((risky * (ulp + 2 * delta)) @ np.abs(q.astype(np.float64)).reshape(-1))
