"""The benchmark-only input generators do what their docstrings state (CPU, no GPU).

These draws shape timing workloads only; parity tests use the plain generators.  The
checks pin the stated structure: counts, order, the shared fraction of the overlap lists,
and the clear-winners lean's separation of about three standard deviations.
"""
import math

import numpy as np
import pytest
import torch

import qsa_synth


def test_clear_winners_shapes_and_rows():
    n_rows, width = 20000, 2048
    cw = qsa_synth.clear_winners_torch(n_rows, width, 5, seed=3, device="cpu")
    rows = cw["rows"].numpy()
    assert cw["q_idx"].shape == (5, width) and cw["add"].shape == (width,)
    assert rows.shape[0] == 200                      # 1% of the rows
    assert np.all(np.diff(rows) > 0) and rows[0] >= 0 and rows[-1] < n_rows
    # the lean is a multiple of the queries' common direction: the queries' mean over many
    # draws points the same way
    many = qsa_synth.clear_winners_torch(n_rows, width, 4000, seed=3, device="cpu")
    cos = torch.nn.functional.cosine_similarity(many["q_idx"].mean(0), many["add"], dim=0)
    assert float(cos) > 0.99
    assert math.isclose(float(many["add"].norm() / many["q_idx"].mean(0).norm()),
                        3.0 * math.sqrt(2.0 / width), rel_tol=0.05)


def test_clear_winners_separation_is_three_sd():
    """Unit-variance rows: the leaning rows' dot products with the queries sit ~3 standard
    deviations (of the other rows' dot products) above them."""
    n_rows, width = 4000, 2048
    cw = qsa_synth.clear_winners_torch(n_rows, width, 8, seed=11, device="cpu", frac=0.05)
    g = torch.Generator().manual_seed(5)
    rows = torch.randn(n_rows, width, generator=g, dtype=torch.float64)
    rows[cw["rows"]] += cw["add"].double()
    dots = rows @ cw["q_idx"].double().T            # [n_rows][8]
    lean = torch.zeros(n_rows, dtype=torch.bool)
    lean[cw["rows"]] = True
    other = dots[~lean]
    gap = (dots[lean].mean(0) - other.mean(0)) / other.std(0)
    assert torch.all((gap > 2.6) & (gap < 3.4)), gap


@pytest.mark.parametrize("share", [0.0, 0.5, 0.9, 1.0])
def test_overlap_lists_share(share):
    n_cand = np.full(32, 3000)
    lists = qsa_synth.overlap_block_lists(n_cand, 256, 16, share, seed=9)
    assert len(lists) == 32
    for i, b in enumerate(lists):
        assert b.shape[0] == 256 and np.all(np.diff(b) > 0) and b[0] >= 0 and b[-1] < 3000
    # within a group, the blocks every member holds number at least the stated share
    for g0 in (0, 16):
        common = set(lists[g0].tolist())
        for b in lists[g0 + 1:g0 + 16]:
            common &= set(b.tolist())
        if share == 1.0:
            assert len(common) == 256
        pair = len(set(lists[g0].tolist()) & set(lists[g0 + 1].tolist()))
        assert pair >= round(share * 256) * round(share * 256) / 256 - 40
