"""The prefill selection fed by the score contraction (qsa_index_score_maxima,
qsa_topk_blocks_maxima).

The score kernel's epilogue also writes each query's largest score of every 32 consecutive
pooled rows; the top-k takes its threshold from those maxima and reads only the groups that
can hold a winner.  The scores must be bit-identical to qsa_index_score's tensor-core path,
the maxima exactly the group maxima of those scores, and the selection exactly the oracle's
top-k (the same integer result qsa_topk_blocks gives) on every row shape: rows long enough
for the maxima form (at least 32 * k candidates), rows that fall back to the sampled or
general forms, ties at the boundary, NaN, -inf, few distinct levels, heavy tails and narrow
bands."""
import math

import numpy as np
import pytest
import torch

import gather_qsa_pool_gb300 as qsa
import qsa_synth
from gpu_helpers import to_dev, to_host
from oracle import oracle

pytestmark = pytest.mark.gpu


def _ws(n_q):
    return torch.empty(qsa.topk_blocks_maxima_workspace_size(n_q), dtype=torch.uint8,
                       device="cuda")


def _group_maxima(s, n_groups):
    """Largest score of each group of 32 columns ([n_q][n_groups]; NaN left out, a group of
    NaN only gives NaN, which ranks as -inf)."""
    n = s.shape[-1]
    pad = np.full(s.shape[:-1] + (n_groups * 32 - n,), -np.inf, np.float32)
    full = np.concatenate([s, pad], axis=-1).reshape(s.shape[:-1] + (n_groups, 32))
    return np.fmax.reduce(full, axis=-1).astype(np.float32)


@pytest.mark.parametrize("H,d,depth,n_q,pooled", [(4, 64, 3001, 130, "f32"),
                                                  (16, 128, 10000, 300, "bf16"),
                                                  (16, 128, 4090, 257, "f32")])
def test_score_maxima_are_the_scores_group_maxima(H, d, depth, n_q, pooled):
    """Scores bit-identical to qsa_index_score (QSA_PREC_BF16_TC); maxima[i][g] the largest
    of scores[i][32g .. 32g+31] (rows the query cannot see are -inf), nothing written past
    the last group; partial query tiles, a partial last row tile and group, a maxima stride
    that breaks the 16-byte alignment of rows; an fp32 and a bf16 cache."""
    shape = qsa_synth.PrefillShape("tcm", depth, n_q, H, d, 8, 2, 128, 256, dtype="bf16")
    inp = qsa_synth.prefill_inputs(shape, seed=41 + n_q)
    n_rows = shape.n_rows
    o_pooled = oracle.pool_rows(inp["raw_k"], shape.n_ctx, H, d, inp["norm_w"], shape.eps,
                                shape.rope_base, 0, n_rows)
    src = to_dev(o_pooled)
    if pooled == "bf16":
        src = src.to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    ws = torch.zeros(qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC,
                                                    qsa.QSA_BF16 if pooled == "bf16"
                                                    else qsa.QSA_F32),
                     dtype=torch.uint8, device="cuda")
    q, q_pos = to_dev(inp["q_idx"]), to_dev(inp["q_pos"])
    ref = torch.empty(n_q, n_rows, device="cuda")
    qsa.index_score(q, src, n_rows, H, d, scale, ref, q_pos=q_pos,
                    precision=qsa.QSA_PREC_BF16_TC, workspace=ws)
    n_groups = (n_rows + 31) // 32
    scores = torch.full((n_q, n_rows + 3), 7.0, device="cuda")
    maxima = torch.full((n_q, n_groups + (3 if pooled == "bf16" else 8)), 9.0, device="cuda")
    qsa.index_score_maxima(q, src, n_rows, H, d, scale, scores, maxima, q_pos=q_pos,
                           workspace=ws)
    g_s, g_m, w_s = to_host(scores), to_host(maxima), to_host(ref)
    np.testing.assert_array_equal(g_s[:, :n_rows], w_s)
    assert np.all(g_s[:, n_rows:] == 7.0)
    np.testing.assert_array_equal(g_m[:, :n_groups], _group_maxima(w_s, n_groups))
    assert np.all(g_m[:, n_groups:] == 9.0)


def _rows(case, n_q, n_full, rng):
    if case == "normal":
        s = rng.standard_normal((n_q, n_full)).astype(np.float32)
    elif case == "equal":
        s = np.full((n_q, n_full), 0.25, np.float32)
    elif case == "few_levels":
        s = rng.integers(0, 40, size=(n_q, n_full)).astype(np.float32) * 0.5
    elif case == "heavy_tail":
        s = rng.standard_cauchy((n_q, n_full)).astype(np.float32)
    elif case == "narrow":
        s = (1.0 + 1e-6 * rng.standard_normal((n_q, n_full))).astype(np.float32)
    else:  # "specials": ties at the boundary, NaN, -inf, +-0 and a hot region
        s = rng.standard_normal((n_q, n_full)).astype(np.float32)
        for i in range(n_q):
            dup = rng.choice(n_full, size=n_full // 10, replace=False)
            s[i, dup] = s[i, rng.choice(n_full, size=dup.shape[0])]
            s[i, rng.choice(n_full, 40, replace=False)] = np.nan
            s[i, rng.choice(n_full, 40, replace=False)] = -np.inf
            s[i, rng.choice(n_full, 5, replace=False)] = -0.0
            s[i, 5000:5400] += 3.0  # many winners in a few groups
    return s


@pytest.mark.parametrize("case", ["normal", "equal", "few_levels", "heavy_tail", "narrow",
                                  "specials"])
def test_topk_with_maxima_exact(case):
    """Exact against the oracle and identical to qsa_topk_blocks; queries seeing 70,000 /
    20,000 / 16,384 / 16,383 / 50,001 / 16,416 full blocks (the maxima form needs k = 512
    groups of 32 candidates: the 16,383-block row takes the other forms)."""
    rng = np.random.default_rng(len(case) * 11)
    n_full, k = 70000, 512
    n_each = np.array([70000, 20000, 16384, 16383, 50001, 16416], np.int64)
    n_q = n_each.shape[0]
    s = _rows(case, n_q, n_full, rng)
    if case == "specials":
        for i in range(n_q):  # a tie exactly at the boundary of each row
            row = np.nan_to_num(s[i, :n_each[i]], nan=-np.inf)
            order = np.lexsort((np.arange(n_each[i]), -row))
            s[i, order[k]] = s[i, order[k - 1]]
    n_groups = (n_full + 31) // 32
    maxima = _group_maxima(s, n_groups)
    q_pos = (4 * n_each - 1).astype(np.int32)  # query i sees exactly n_each[i] full blocks
    blocks = torch.full((n_q, k), -3, dtype=torch.int32, device="cuda")
    counts = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    qsa.topk_blocks_maxima(to_dev(s), to_dev(maxima), n_full, k, blocks, counts, _ws(n_q),
                           q_pos=to_dev(q_pos))
    ref_b = torch.full((n_q, k), -3, dtype=torch.int32, device="cuda")
    ref_c = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(to_dev(s), n_full, k, ref_b, ref_c, q_pos=to_dev(q_pos))
    g_b, g_c = to_host(blocks), to_host(counts)
    np.testing.assert_array_equal(g_b, to_host(ref_b))
    np.testing.assert_array_equal(g_c, to_host(ref_c))
    for i in range(n_q):
        want = oracle.topk(s[i].astype(np.float64), int(n_each[i]), k)
        assert g_c[i] == want.shape[0]
        np.testing.assert_array_equal(g_b[i, :g_c[i]], want)


def test_topk_with_maxima_unaligned_rows_and_strides():
    """Rows 40,001 scores apart (row i starts 4i bytes past a 16-byte boundary, mod 16) and a
    padded maxima stride, all queries at the end of the context."""
    rng = np.random.default_rng(78)
    n_q, n_full, k = 6, 40001, 512
    s = (4 * rng.standard_normal((n_q, n_full))).astype(np.float32)
    n_groups = (n_full + 31) // 32
    maxima = np.full((n_q, n_groups + 7), np.nan, np.float32)
    maxima[:, :n_groups] = _group_maxima(s, n_groups)
    blocks = torch.full((n_q, k), -3, dtype=torch.int32, device="cuda")
    counts = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    qsa.topk_blocks_maxima(to_dev(s), to_dev(maxima), n_full, k, blocks, counts, _ws(n_q))
    g_b, g_c = to_host(blocks), to_host(counts)
    for i in range(n_q):
        want = oracle.topk(s[i].astype(np.float64), n_full, k)
        assert g_c[i] == k
        np.testing.assert_array_equal(g_b[i], want)


def test_topk_with_maxima_short_rows_and_small_k():
    """Rows with fewer candidates than k (every candidate selected), k = 1 and k = 3000 on
    100,000 blocks (3000 groups needed: the maxima form still applies)."""
    rng = np.random.default_rng(79)
    for n_full, k in [(300, 512), (100000, 1), (100000, 3000), (16384, 512)]:
        s = rng.standard_normal((2, n_full)).astype(np.float32)
        n_groups = (n_full + 31) // 32
        maxima = _group_maxima(s, n_groups)
        blocks = torch.full((2, k), -3, dtype=torch.int32, device="cuda")
        counts = torch.zeros(2, dtype=torch.int32, device="cuda")
        qsa.topk_blocks_maxima(to_dev(s), to_dev(maxima), n_full, k, blocks, counts, _ws(2))
        g_b, g_c = to_host(blocks), to_host(counts)
        for i in range(2):
            want = oracle.topk(s[i].astype(np.float64), n_full, k)
            assert g_c[i] == want.shape[0]
            np.testing.assert_array_equal(g_b[i, :g_c[i]], want)
            assert np.all(g_b[i, g_c[i]:] == -3)


def test_topk_with_maxima_many_queries_handed_back():
    """300 queries, most of them rows of equal scores (every block a candidate: each is
    handed back to the general kernel, whose persistent grid then takes two queries per CTA)
    and a few Gaussian rows: identical to qsa_topk_blocks, sampled rows against the oracle."""
    rng = np.random.default_rng(80)
    n_q, n_full, k = 300, 20000, 512
    s = np.full((n_q, n_full), 0.5, np.float32)
    s[::7] = rng.standard_normal((len(range(0, n_q, 7)), n_full)).astype(np.float32)
    maxima = _group_maxima(s, (n_full + 31) // 32)
    blocks = torch.full((n_q, k), -3, dtype=torch.int32, device="cuda")
    counts = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    qsa.topk_blocks_maxima(to_dev(s), to_dev(maxima), n_full, k, blocks, counts, _ws(n_q))
    ref_b = torch.full((n_q, k), -3, dtype=torch.int32, device="cuda")
    ref_c = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(to_dev(s), n_full, k, ref_b, ref_c)
    np.testing.assert_array_equal(to_host(blocks), to_host(ref_b))
    np.testing.assert_array_equal(to_host(counts), to_host(ref_c))
    g_b = to_host(blocks)
    for i in (0, 1, 7, 299):
        np.testing.assert_array_equal(g_b[i], oracle.topk(s[i].astype(np.float64), n_full, k))


@pytest.mark.parametrize("n_q,depth", [(130, 3001), (300, 10000), (600, 6003), (1000, 5002),
                                       (512, 17), (1, 900), (257, 1000)])
def test_aligned_row_scores_against_oracle(n_q, depth):
    """Score rows 16 bytes apart (the epilogue's whole-line transposed stores): every score
    of partial query and row tiles against the oracle's bf16-operand scores (one query; a
    second pair of 256 queries holding one live row; a context shorter than one row tile),
    columns past n_rows untouched (n_rows % 4 == 3 and 1 among them), and the same scores
    through a stride
    that breaks the alignment (the per-lane stores)."""
    from gpu_helpers import score_tolerance
    H, d = 16, 128
    shape = qsa_synth.PrefillShape("tma", depth, n_q, H, d, 8, 2, 128, 256, dtype="bf16")
    inp = qsa_synth.prefill_inputs(shape, seed=55 + n_q)
    n_rows = shape.n_rows
    o_pooled = oracle.pool_rows(inp["raw_k"], shape.n_ctx, H, d, inp["norm_w"], shape.eps,
                                shape.rope_base, 0, n_rows)
    scale = 1.0 / math.sqrt(d)
    ws = torch.zeros(qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC),
                     dtype=torch.uint8, device="cuda")
    q, q_pos, pooled = to_dev(inp["q_idx"]), to_dev(inp["q_pos"]), to_dev(o_pooled)
    ld = (n_rows + 3) // 4 * 4 + 8
    scores = torch.full((n_q, ld), 7.0, device="cuda")
    maxima = torch.empty(n_q, (n_rows + 31) // 32, device="cuda")
    qsa.index_score_maxima(q, pooled, n_rows, H, d, scale, scores, maxima, q_pos=q_pos,
                           workspace=ws)
    odd = torch.full((n_q, n_rows + 1), 7.0, device="cuda")
    qsa.index_score(q, pooled, n_rows, H, d, scale, odd, q_pos=q_pos,
                    precision=qsa.QSA_PREC_BF16_TC, workspace=ws)
    got = to_host(scores)
    assert np.all(got[:, n_rows:] == 7.0)
    np.testing.assert_array_equal(got[:, :n_rows], to_host(odd)[:, :n_rows])
    want = oracle.scores(inp["q_idx"], o_pooled, n_rows, H, d, scale, q_pos=inp["q_pos"],
                         round_bf16_operands=True)
    qb = np.array([oracle.round_bf16(float(x)) for x in inp["q_idx"].reshape(-1)],
                  np.float32).reshape(n_q, -1)
    for i in range(n_q):
        vis = np.isfinite(want[i])
        assert np.array_equal(np.isneginf(got[i, :n_rows]), ~vis)
        tol = score_tolerance(qb[i], o_pooled, n_rows, scale, chain=H * d)[vis]
        assert np.all(np.abs(got[i, :n_rows][vis] - want[i][vis]) <= tol)


@pytest.mark.parametrize("pad,shift", [(1, 0), (3, 1)])
def test_tensor_core_scores_with_strided_queries(pad, shift):
    """Query rows whose starts are not all on a 16-byte boundary (a row stride of H*d + 1,
    or rows of H*d + 4 starting one float in) are rounded to bf16 element by element: the
    tensor-core scores equal those of the contiguous queries bit for bit."""
    H, d, n_q, n_rows = 16, 128, 130, 700
    rng = np.random.default_rng(70 + pad)
    qh = rng.standard_normal((n_q, H * d)).astype(np.float32)
    pooled = to_dev(rng.standard_normal((n_rows, H * d)).astype(np.float32))
    ws = torch.zeros(qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC),
                     dtype=torch.uint8, device="cuda")
    q = to_dev(qh)
    big = torch.zeros(n_q, H * d + pad + shift, device="cuda")
    big[:, shift:shift + H * d] = q
    qs = big[:, shift:shift + H * d]
    want = torch.empty(n_q, n_rows, device="cuda")
    got = torch.empty(n_q, n_rows, device="cuda")
    qsa.index_score(q, pooled, n_rows, H, d, 0.125, want, precision=qsa.QSA_PREC_BF16_TC,
                    workspace=ws)
    qsa.index_score(qs, pooled, n_rows, H, d, 0.125, got, precision=qsa.QSA_PREC_BF16_TC,
                    workspace=ws)
    np.testing.assert_array_equal(to_host(got), to_host(want))
