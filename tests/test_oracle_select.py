"""Pins of the oracle's scoring, block-domain top-k and cell expansion."""
import json
import os

import numpy as np
import pytest

from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ score

def test_score_unit_query_picks_one_component():
    """q = e_(h,j) gives s_b = scale * z[b][h*d + j]: a transposed or shifted operand
    index would pick a different component."""
    rng = np.random.default_rng(20)
    H, d, n_rows = 3, 8, 11
    pooled = rng.standard_normal((n_rows, H * d)).astype(np.float32)
    for h, j in [(0, 0), (1, 5), (2, 7), (2, 4)]:
        q = np.zeros(H * d, np.float32)
        q[h * d + j] = 1.0
        s = oracle.scores(q, pooled, n_rows, H, d, 0.25)[0]
        np.testing.assert_array_equal(s, 0.25 * pooled[:, h * d + j].astype(np.float64))


def test_score_matches_library_matvec_per_query():
    rng = np.random.default_rng(21)
    H, d, n_rows = 4, 64, 50
    pooled = rng.standard_normal((n_rows, H * d)).astype(np.float32)
    q1 = rng.standard_normal(H * d).astype(np.float32)
    q2 = rng.standard_normal(H * d).astype(np.float32)
    scale = 1 / 8
    s1 = oracle.scores(q1, pooled, n_rows, H, d, scale)[0]
    s2 = oracle.scores(q2, pooled, n_rows, H, d, scale)[0]
    np.testing.assert_allclose(s1, scale * (pooled.astype(np.float64) @ q1.astype(np.float64)),
                               rtol=1e-12, atol=1e-12)
    # each query row is scored on its own (no cross-row mixing)
    qs = np.stack([q1, q2])
    s12 = oracle.scores(qs, pooled, n_rows, H, d, scale)
    np.testing.assert_array_equal(s12[0], s1)
    np.testing.assert_array_equal(s12[1], s2)


def test_score_causal_visibility_of_blocks():
    """Row b is visible to a query at position p only when 4b + 3 <= p."""
    H, d, n_rows = 1, 4, 6
    pooled = np.ones((n_rows, H * d), np.float32)
    q = np.ones((3, H * d), np.float32)
    q_pos = np.array([10, 11, 3], np.int32)
    s = oracle.scores(q, pooled, n_rows, H, d, 1.0, q_pos=q_pos)
    assert np.all(np.isfinite(s[0, :2])) and np.all(np.isneginf(s[0, 2:]))   # 4*2+3 = 11 > 10
    assert np.all(np.isfinite(s[1, :3])) and np.all(np.isneginf(s[1, 3:]))
    assert np.isfinite(s[2, 0]) and np.all(np.isneginf(s[2, 1:]))


def test_bf16_round_to_nearest_even():
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0                  # tie -> even
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6  # tie -> even (up)
    assert oracle.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -20) == 1.0 + 2.0 ** -7
    assert oracle.round_bf16(-3.0) == -3.0
    assert oracle.round_bf16(float("inf")) == float("inf")


def test_score_bf16_operand_mirror():
    H, d = 1, 2
    pooled = np.array([[1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]], np.float32)
    q = np.array([1.0, 1.0 + 2.0 ** -8], np.float32)
    s = oracle.scores(q, pooled, 1, H, d, 1.0, round_bf16_operands=True)[0, 0]
    assert s == 1.0 * 1.0 + (1.0 + 2.0 ** -6) * 1.0
    s32 = oracle.scores(q, pooled, 1, H, d, 1.0)[0, 0]
    assert s32 == pytest.approx((1 + 2.0 ** -8) + (1 + 3 * 2.0 ** -8) * (1 + 2.0 ** -8), rel=0,
                                abs=1e-15)


# ------------------------------------------------------------------ top-k

def _library_topk(s, n_full, k):
    order = np.lexsort((np.arange(n_full), -np.nan_to_num(s[:n_full], nan=-np.inf)))
    return np.sort(order[:min(k, n_full)]).astype(np.int32)


@pytest.mark.parametrize("n_full,k", [(512, 16), (15447, 512), (100, 100), (37, 64), (1, 1)])
def test_topk_equals_full_sort(n_full, k):
    rng = np.random.default_rng(n_full + k)
    s = rng.standard_normal(n_full + 1)  # the extra (open) row never competes
    s[-1] = 1e9
    got = oracle.topk(s, n_full, k)
    np.testing.assert_array_equal(got, _library_topk(s, n_full, k))


def test_topk_equals_pages_old_cell_level_path():
    """The pages' earlier path expanded each block score to its 4 cells (cell -> block
    map), took the top 2048 cells, and attended those; block-domain top-k must pick the
    same blocks when no tie straddles the boundary."""
    rng = np.random.default_rng(30)
    n_full, top_k_tokens = 3001, 2048
    s = rng.standard_normal(n_full)
    cell_blk = np.repeat(np.arange(n_full), 4)
    cell_score = s[cell_blk]
    order = np.argsort(-cell_score, kind="stable")[:top_k_tokens]
    old_blocks = np.unique(cell_blk[order])
    new_blocks = oracle.topk(s, n_full, top_k_tokens // 4)
    np.testing.assert_array_equal(new_blocks, old_blocks)


def test_expand_block_scores_matches_library_repeat_and_cell_topk():
    """The expansion step of the old path equals numpy's repeat; the oracle's top-k over the
    expanded cells (ties to the lower cell) then picks whole blocks, the block-domain set."""
    rng = np.random.default_rng(31)
    n_full = 777
    s = rng.standard_normal(n_full)
    cells = oracle.expand_block_scores(s, n_full)
    np.testing.assert_array_equal(cells, np.repeat(s, 4))
    assert oracle.expand_block_scores(s, 0).shape == (0,)
    top_cells = oracle.topk(cells, 4 * n_full, 512)
    np.testing.assert_array_equal(np.unique(top_cells // 4), oracle.topk(s, n_full, 128))
    assert np.all(np.bincount(top_cells // 4)[np.unique(top_cells // 4)] == 4)


def test_topk_ties_go_to_lower_index_and_nan_ranks_last():
    s = np.array([1.0, 2.0, 2.0, 2.0, np.nan, 2.0, -np.inf, 0.5])
    np.testing.assert_array_equal(oracle.topk(s, 8, 3), [1, 2, 3])
    np.testing.assert_array_equal(oracle.topk(s, 8, 6), [0, 1, 2, 3, 5, 7])
    # NaN ranks as -inf, and ties with -inf go to the lower index (4 before 6)
    np.testing.assert_array_equal(oracle.topk(s, 8, 7), [0, 1, 2, 3, 4, 5, 7])
    assert oracle.topk(s, 8, 0).shape == (0,)
    assert oracle.topk(s, 0, 5).shape == (0,)


def test_cells_expand_blocks_and_append_tail():
    blocks = np.array([0, 5, 9], np.int32)
    # p = 42: n_full = 43 // 4 = 10, tail = 40, 41, 42
    c = oracle.cells(blocks, 42)
    np.testing.assert_array_equal(c, [0, 1, 2, 3, 20, 21, 22, 23, 36, 37, 38, 39, 40, 41, 42])
    # p = 43 closes block 10: empty tail
    np.testing.assert_array_equal(oracle.cells(blocks, 43)[-1], 39)
    assert oracle.cells(blocks, 43).shape[0] == 12


def test_pages_cell_budget_2051():
    with open(os.path.join(GOLDEN, "pages_facts.json")) as f:
        g = json.load(f)
    k_blk = g["indexer_top_k_tokens"] // g["compression_ratio"]
    rng = np.random.default_rng(31)
    # 255,183 = 4 * 63,795 + 3: the largest tail; 255,181 (the pages' 256k input) has 1
    for n_ctx, want in [(255183, g["max_cells_with_open_block"]), (255182, 2050),
                        (255181, 2049), (255180, 2048)]:
        n_full = n_ctx // 4
        s = rng.standard_normal(n_full)
        blocks = oracle.topk(s, n_full, k_blk)
        c = oracle.cells(blocks, n_ctx - 1)
        assert c.shape[0] == want == 4 * min(k_blk, n_full) + n_ctx % 4
        assert np.all(np.diff(c) > 0) and c[-1] <= n_ctx - 1


def test_get_rows_is_plain_row_indexing():
    rng = np.random.default_rng(32)
    src = rng.standard_normal((40, 3, 8)).astype(np.float32)
    cl = np.array([3, 0, 39, 7], np.int32)
    got = oracle.get_rows(src, 24, 24, cl)
    np.testing.assert_array_equal(got, src.reshape(40, 24)[cl])
