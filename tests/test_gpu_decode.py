"""GPU parity of the decode path (pool update, index score, block top-k, gather, sparse
attention) against the fp64 oracle on the same seeded inputs.  Every input and every
expected value comes from qsa_synth or the oracle, never from the CUDA path."""
import math

import numpy as np
import pytest
import torch

import gather_qsa_pool_gb300 as qsa
import qsa_synth
from oracle import oracle
from gpu_helpers import (ATOL_ATTN_BF16, ATOL_ATTN_F32, check_topk, score_tolerance, to_dev,
                         to_host)

pytestmark = pytest.mark.gpu

TINY = qsa_synth.CONFIGS["tiny_f32_decode"]
SMALL_BF16 = qsa_synth.shrink(qsa_synth.CONFIGS["decode_64k"], name="small_bf16", n_ctx=9_003,
                              top_k_tokens=512)


def _atol(shape):
    return ATOL_ATTN_BF16 if shape.dtype == "bf16" else ATOL_ATTN_F32


def _pool_tol(z):
    # fp32 pooling + RMS norm + rotation: a few ulps of each component's magnitude
    return dict(rtol=2e-5, atol=2e-6 * max(1.0, float(np.abs(z).max())))


# ------------------------------------------------------------------ a1 pool update

@pytest.mark.parametrize("shape", [TINY, SMALL_BF16], ids=lambda s: s.name)
def test_pool_update_full_rebuild(shape):
    inp = qsa_synth.decode_inputs(shape, seed=1)
    n_ctx, H, d = shape.n_ctx, shape.H_idx, shape.d_idx
    want = oracle.pool_rows(inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps, shape.rope_base,
                            0, shape.n_rows)
    pooled = torch.zeros(shape.n_rows + 5, H * d, device="cuda")
    qsa.pool_update(to_dev(inp["raw_k"]), n_ctx, H, d, to_dev(inp["norm_w"]), shape.eps,
                    shape.rope_base, pooled, 0)
    got = to_host(pooled)
    np.testing.assert_allclose(got[:shape.n_rows], want, **_pool_tol(want))
    assert np.all(got[shape.n_rows:] == 0)


@pytest.mark.parametrize("n_ctx", [1, 2, 3, 4, 5, 6, 7, 8, 37, 2050])
def test_pool_update_every_tail_length(n_ctx):
    shape = TINY
    inp = qsa_synth.decode_inputs(shape, seed=2)
    H, d = shape.H_idx, shape.d_idx
    n_rows = (n_ctx + 3) // 4
    want = oracle.pool_rows(inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps,
                            shape.rope_base, 0, n_rows)
    pooled = torch.zeros(n_rows, H * d, device="cuda")
    qsa.pool_update(to_dev(inp["raw_k"]), n_ctx, H, d, to_dev(inp["norm_w"]), shape.eps,
                    shape.rope_base, pooled, 0)
    np.testing.assert_allclose(to_host(pooled), want, **_pool_tol(want))


def test_pool_update_incremental_equals_rebuild_and_respects_valid_rows():
    """Appending tokens one by one and recomputing only rows >= n_valid_full gives the
    same cache, bit for bit, as rebuilding every row; valid rows are never written."""
    shape = qsa_synth.shrink(SMALL_BF16, n_ctx=4001)
    inp = qsa_synth.decode_inputs(shape, seed=3, extra_tokens=40)
    H, d = shape.H_idx, shape.d_idx
    raw, w = to_dev(inp["raw_k"]), to_dev(inp["norm_w"])
    n_end = shape.n_ctx + 40
    cap = (n_end + 3) // 4
    inc = torch.zeros(cap, H * d, device="cuda")
    qsa.pool_update(raw, shape.n_ctx, H, d, w, shape.eps, shape.rope_base, inc, 0)
    n_ctx = shape.n_ctx
    sentinel_row = 17
    inc[sentinel_row] = 12345.0  # a valid row: must survive every incremental update
    while n_ctx < n_end:
        n_valid = n_ctx // 4
        n_ctx += 1
        qsa.pool_update(raw, n_ctx, H, d, w, shape.eps, shape.rope_base, inc, n_valid)
    assert torch.all(inc[sentinel_row] == 12345.0)
    inc[sentinel_row] = 0.0
    full = torch.zeros_like(inc)
    qsa.pool_update(raw, n_end, H, d, w, shape.eps, shape.rope_base, full, 0)
    full[sentinel_row] = 0.0
    assert torch.equal(inc, full)
    # invalidation: passing a smaller n_valid_full recomputes from there on
    inc[100:] = -7.0
    qsa.pool_update(raw, n_end, H, d, w, shape.eps, shape.rope_base, inc, 100)
    full2 = torch.zeros_like(inc)
    qsa.pool_update(raw, n_end, H, d, w, shape.eps, shape.rope_base, full2, 0)
    assert torch.equal(inc[100:], full2[100:])


# ------------------------------------------------------------------ a2 index score

@pytest.mark.parametrize("shape", [TINY, SMALL_BF16], ids=lambda s: s.name)
def test_index_score(shape):
    inp = qsa_synth.decode_inputs(shape, seed=4)
    H, d = shape.H_idx, shape.d_idx
    pooled = oracle.pool_rows(inp["raw_k"], shape.n_ctx, H, d, inp["norm_w"], shape.eps,
                              shape.rope_base, 0, shape.n_rows)
    scale = 1.0 / math.sqrt(d)
    want = oracle.scores(inp["q_idx"][0], pooled, shape.n_rows, H, d, scale)[0]
    scores = torch.full((1, shape.n_rows + 3), 99.0, device="cuda")
    qsa.index_score(to_dev(inp["q_idx"][:1]), to_dev(pooled), shape.n_rows, H, d, scale, scores)
    got = to_host(scores)[0]
    tol = score_tolerance(inp["q_idx"][0], pooled, shape.n_rows, scale)
    assert np.all(np.abs(got[:shape.n_rows] - want) <= tol)
    assert np.all(got[shape.n_rows:] == 99.0)


def test_index_score_general_path_odd_dims_and_queries():
    """H*d not a multiple of 128 and several queries take the tiled kernel."""
    rng = np.random.default_rng(5)
    H, d, n_rows, n_q = 3, 40, 1000, 5
    pooled = rng.standard_normal((n_rows, H * d)).astype(np.float32)
    q = rng.standard_normal((n_q, H * d)).astype(np.float32)
    scale = 0.2
    want = oracle.scores(q, pooled, n_rows, H, d, scale)
    got = torch.zeros(n_q, n_rows, device="cuda")
    qsa.index_score(to_dev(q), to_dev(pooled), n_rows, H, d, scale, got)
    got = to_host(got)
    for i in range(n_q):
        tol = score_tolerance(q[i], pooled, n_rows, scale, chain=H * d + 1)
        assert np.all(np.abs(got[i] - want[i]) <= tol)


# ------------------------------------------------------------------ a3 top-k

def _oracle_topk_on_f32(s32, n_full, k):
    return oracle.topk(s32.astype(np.float64), n_full, k)


@pytest.mark.parametrize("n_full,k_blk", [(512, 16), (15447, 512), (63795, 512), (64051, 512),
                                          (300, 512), (512, 512), (513, 512), (9, 1), (1, 1),
                                          (0, 4), (100000, 3000), (8, 3), (17, 16)])
def test_topk_exact_on_identical_scores(n_full, k_blk):
    """Same fp32 scores on both sides: the selection is integer work and must be exact,
    including duplicated scores (ties go to the lower index), NaN, -inf and -0/+0."""
    rng = np.random.default_rng(n_full * 7 + k_blk)
    s = rng.standard_normal(n_full + 1).astype(np.float32)
    if n_full > 20:
        dup = rng.choice(n_full, size=n_full // 10, replace=False)
        s[dup] = s[rng.choice(n_full, size=dup.shape[0])]   # many exact ties
        s[rng.choice(n_full, 3, replace=False)] = np.nan
        s[rng.choice(n_full, 3, replace=False)] = -np.inf
        s[rng.choice(n_full, 2, replace=False)] = -0.0
        s[rng.choice(n_full, 2, replace=False)] = 0.0
        # force a tie exactly at the boundary
        order = np.lexsort((np.arange(n_full), -np.nan_to_num(s[:n_full], nan=-np.inf)))
        if k_blk < n_full:
            s[order[k_blk]] = s[order[k_blk - 1]]
    scores = to_dev(s.reshape(1, -1))
    blocks = torch.full((1, k_blk), -5, dtype=torch.int32, device="cuda")
    counts = torch.full((1,), -5, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(scores, n_full, k_blk, blocks, counts)
    want = _oracle_topk_on_f32(s, n_full, k_blk)
    c = int(to_host(counts)[0])
    assert c == want.shape[0]
    np.testing.assert_array_equal(to_host(blocks)[0, :c], want)
    assert np.all(to_host(blocks)[0, c:] == -5)


def test_topk_all_equal_scores():
    s = np.full(5000, 1.5, np.float32)
    blocks = torch.zeros((1, 100), dtype=torch.int32, device="cuda")
    counts = torch.zeros(1, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(to_dev(s[None]), 5000, 100, blocks, counts)
    np.testing.assert_array_equal(to_host(blocks)[0], np.arange(100))


@pytest.mark.parametrize("case", ["equal", "few_levels", "heavy_tail", "narrow"])
def test_topk_large_rows_many_queries(case):
    """Several queries of 20k-70k blocks (the sampled-threshold form of the general kernel):
    all-equal rows (too many candidates: the full form), a few distinct levels (ties across
    the threshold), a heavy tail and a narrow band of values.  Exact against the oracle."""
    rng = np.random.default_rng(len(case))
    n_q, n_full, k = 5, 70000, 512
    if case == "equal":
        s = np.full((n_q, n_full), 0.25, np.float32)
    elif case == "few_levels":
        s = rng.integers(0, 40, size=(n_q, n_full)).astype(np.float32) * 0.5
    elif case == "heavy_tail":
        s = rng.standard_cauchy((n_q, n_full)).astype(np.float32)
    else:
        s = (1.0 + 1e-6 * rng.standard_normal((n_q, n_full))).astype(np.float32)
    n_each = np.array([70000, 20000, 16384, 16383, 50001], np.int64)
    q_pos = (4 * n_each - 1).astype(np.int32)  # query i sees exactly n_each[i] full blocks
    blocks = torch.full((n_q, k), -3, dtype=torch.int32, device="cuda")
    counts = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(to_dev(s), n_full, k, blocks, counts, q_pos=to_dev(q_pos))
    g_blocks, g_counts = to_host(blocks), to_host(counts)
    for i in range(n_q):
        want = _oracle_topk_on_f32(s[i], int(n_each[i]), k)
        assert g_counts[i] == want.shape[0]
        np.testing.assert_array_equal(g_blocks[i, :g_counts[i]], want)


def test_topk_sampled_form_on_unaligned_rows():
    """Rows 40,001 scores apart (row i starts 4i bytes past a 16-byte boundary, mod 16):
    the sampled candidate pass takes its vector form on the aligned rows and its scalar
    form on the others.  Exact against the oracle; a ragged column count (n mod 4 = 1)."""
    rng = np.random.default_rng(77)
    n_q, n_full, k = 6, 40001, 512
    s = (4 * rng.standard_normal((n_q, n_full))).astype(np.float32)
    blocks = torch.full((n_q, k), -3, dtype=torch.int32, device="cuda")
    counts = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(to_dev(s), n_full, k, blocks, counts)
    g_blocks, g_counts = to_host(blocks), to_host(counts)
    for i in range(n_q):
        want = _oracle_topk_on_f32(s[i], n_full, k)
        assert g_counts[i] == k
        np.testing.assert_array_equal(g_blocks[i], want)


@pytest.mark.parametrize("case", ["normal", "equal", "few_levels", "heavy_tail", "narrow"])
def test_topk_many_queries(case):
    """A prefill-sized query count (more than two per SM: the general kernel's
    two-CTAs-per-SM form) over rows of up to 40k blocks, each query seeing its own number
    of complete blocks (sampled form, full form, fewer blocks than k).  Exact against the
    oracle for every query; nothing written past each query's count."""
    rng = np.random.default_rng(100 + len(case))
    n_q, n_full, k = 320, 40000, 512
    if case == "normal":
        s = (4 * rng.standard_normal((n_q, n_full))).astype(np.float32)
    elif case == "equal":
        s = np.full((n_q, n_full), -1.5, np.float32)
    elif case == "few_levels":
        s = rng.integers(0, 40, size=(n_q, n_full)).astype(np.float32) * 0.5
    elif case == "heavy_tail":
        s = rng.standard_cauchy((n_q, n_full)).astype(np.float32)
    else:
        s = (1.0 + 1e-6 * rng.standard_normal((n_q, n_full))).astype(np.float32)
    base = np.array([40000, 20000, 16384, 16383, 30001, 513, 512, 100, 0, 1], np.int64)
    n_each = np.where(np.arange(n_q) < base.shape[0], base[np.arange(n_q) % base.shape[0]],
                      rng.integers(16384, n_full + 1, size=n_q))
    q_pos = (4 * n_each - 1 + (np.arange(n_q) % 4)).astype(np.int32)  # tails of 0-3 tokens
    blocks = torch.full((n_q, k), -3, dtype=torch.int32, device="cuda")
    counts = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(to_dev(s), n_full, k, blocks, counts, q_pos=to_dev(q_pos))
    g_blocks, g_counts = to_host(blocks), to_host(counts)
    for i in range(n_q):
        want = _oracle_topk_on_f32(s[i], int(n_each[i]), k)
        assert g_counts[i] == want.shape[0], i
        np.testing.assert_array_equal(g_blocks[i, :g_counts[i]], want)
        assert np.all(g_blocks[i, g_counts[i]:] == -3)


def test_topk_per_query_positions():
    """With q_pos, query i ranks only blocks complete at its position."""
    rng = np.random.default_rng(6)
    n_q, n_full, k = 6, 3000, 64
    s = rng.standard_normal((n_q, n_full)).astype(np.float32)
    q_pos = np.array([11999, 100, 3, 255, 256, 7000], np.int32)
    blocks = torch.full((n_q, k), -1, dtype=torch.int32, device="cuda")
    counts = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(to_dev(s), n_full, k, blocks, counts, q_pos=to_dev(q_pos))
    b, c = to_host(blocks), to_host(counts)
    for i in range(n_q):
        nf = min(n_full, (int(q_pos[i]) + 1) // 4)
        want = _oracle_topk_on_f32(s[i], nf, k)
        assert c[i] == want.shape[0]
        np.testing.assert_array_equal(b[i, :c[i]], want)


# ------------------------------------------------------------------ a4 gather

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gather_positions_and_rows(dtype):
    rng = np.random.default_rng(7)
    n_ctx, H_kv, d, k_blk = 10_003, 4, 128, 64
    K = rng.standard_normal((n_ctx, H_kv, d)).astype(np.float32)
    V = rng.standard_normal((n_ctx, H_kv, d)).astype(np.float32)
    if dtype == "bf16":
        K, V = qsa_synth.to_bf16_bits(K), qsa_synth.to_bf16_bits(V)
    n_full = n_ctx // 4
    blocks = np.sort(rng.choice(n_full, k_blk, replace=False)).astype(np.int32)
    max_cells = 4 * k_blk + 3
    want_cells = oracle.cells(blocks, n_ctx - 1)
    Kd, Vd = to_dev(K), to_dev(V)
    pos = torch.full((1, max_cells), -9, dtype=torch.int32, device="cuda")
    n_cells = torch.zeros(1, dtype=torch.int32, device="cuda")
    K_out = torch.zeros((max_cells, H_kv, d), dtype=Kd.dtype, device="cuda")
    V_out = torch.zeros_like(K_out)
    qsa.gather_kv(to_dev(blocks[None]), to_dev(np.array([k_blk], np.int32)), k_blk, pos, n_cells,
                  max_cells, n_ctx=n_ctx, K=Kd, V=Vd, K_out=K_out, V_out=V_out, H_kv=H_kv, d_k=d,
                  d_v=d)
    nc = int(to_host(n_cells)[0])
    assert nc == want_cells.shape[0] == 4 * k_blk + n_ctx % 4
    np.testing.assert_array_equal(to_host(pos)[0, :nc], want_cells)
    assert np.all(to_host(pos)[0, nc:] == -9)
    np.testing.assert_array_equal(to_host(K_out)[:nc].reshape(nc, -1),
                                  oracle.get_rows(K, H_kv * d, H_kv * d, want_cells))
    np.testing.assert_array_equal(to_host(V_out)[:nc].reshape(nc, -1),
                                  oracle.get_rows(V, H_kv * d, H_kv * d, want_cells))


# ------------------------------------------------------------------ a5 attention

def _random_cells(rng, n_ctx, k_blk):
    n_full = n_ctx // 4
    k = min(k_blk, n_full)
    blocks = np.sort(rng.choice(n_full, k, replace=False)).astype(np.int32)
    return oracle.cells(blocks, n_ctx - 1)


@pytest.mark.parametrize("dtype,H_q,H_kv,n_ctx,k_blk", [
    ("f32", 8, 2, 2050, 16), ("bf16", 32, 4, 61789, 512), ("bf16", 32, 4, 255181, 512),
    ("f32", 4, 4, 1000, 37), ("bf16", 16, 8, 3001, 1), ("bf16", 32, 4, 6, 512),
    ("bf16", 32, 4, 1, 512)])
def test_sparse_attn_over_listed_cells(dtype, H_q, H_kv, n_ctx, k_blk):
    rng = np.random.default_rng(n_ctx + H_q)
    d = 128
    # The cell list has the length and layout of a context of n_ctx tokens (k_blk blocks
    # plus the tail); above 70k tokens the positions wrap into a 70k-row cache to keep the
    # host copy small -- the kernel's launch shape depends only on the list, not on n_ctx.
    n_tok = min(n_ctx, 70_000)
    cells = _random_cells(rng, n_ctx, k_blk)
    cells = cells % n_tok if n_ctx > n_tok else cells
    K = rng.standard_normal((n_tok, H_kv, d)).astype(np.float32)
    V = rng.standard_normal((n_tok, H_kv, d)).astype(np.float32)
    if dtype == "bf16":
        K, V = qsa_synth.to_bf16_bits(K), qsa_synth.to_bf16_bits(V)
    q = rng.standard_normal((1, H_q, d)).astype(np.float32)
    scale = 1.0 / math.sqrt(d)
    want, want_lse = oracle.attention(q[0], K, V, H_q, H_kv, d, d, H_kv * d, H_kv * d, cells, scale)
    max_cells = 4 * k_blk + 3
    pos = np.full((1, max_cells), -1, np.int32)
    pos[0, :cells.shape[0]] = cells
    out = torch.full((1, H_q, d), 7.0, device="cuda")
    lse = torch.zeros((1, H_q), device="cuda")
    ws = torch.empty(max(qsa.sparse_attn_workspace_size(1, H_q, H_kv, d, max_cells) // 4, 1),
                     device="cuda")
    qsa.sparse_attn(to_dev(q), to_dev(K), to_dev(V), to_dev(np.array([cells.shape[0]], np.int32)),
                    max_cells, out, H_kv, d, d, scale, pos=to_dev(pos), lse=lse, workspace=ws)
    atol = ATOL_ATTN_BF16 if dtype == "bf16" else ATOL_ATTN_F32
    np.testing.assert_allclose(to_host(out)[0], want, rtol=0, atol=atol)
    np.testing.assert_allclose(to_host(lse)[0], want_lse, rtol=1e-5, atol=1e-5)


def test_sparse_attn_compact_rows_and_overflow_and_empty():
    rng = np.random.default_rng(9)
    H_q, H_kv, d, max_cells = 8, 2, 128, 67
    Kc = rng.standard_normal((2, max_cells, H_kv, d)).astype(np.float32)   # two queries
    Vc = rng.standard_normal((2, max_cells, H_kv, d)).astype(np.float32)
    q = rng.standard_normal((2, H_q, d)).astype(np.float32)
    n = np.array([50, 0], np.int32)
    out = torch.zeros((2, H_q, d), device="cuda")
    lse = torch.zeros((2, H_q), device="cuda")
    ws = torch.empty(max(qsa.sparse_attn_workspace_size(2, H_q, H_kv, d, max_cells) // 4, 1),
                     device="cuda")
    Kd = to_dev(Kc.reshape(2 * max_cells, H_kv, d))
    Vd = to_dev(Vc.reshape(2 * max_cells, H_kv, d))
    qsa.sparse_attn(to_dev(q), Kd, Vd, to_dev(n), max_cells, out, H_kv, d, d, 0.1, lse=lse,
                    workspace=ws)
    want, want_lse = oracle.attention(q[0], Kc[0], Vc[0], H_q, H_kv, d, d, H_kv * d, H_kv * d,
                                      np.arange(50, dtype=np.int32), 0.1)
    np.testing.assert_allclose(to_host(out)[0], want, atol=ATOL_ATTN_F32, rtol=0)
    assert np.all(to_host(out)[1] == 0) and np.all(np.isneginf(to_host(lse)[1]))
    # a truncated list (count > capacity) must give NaN, never a silently wrong answer
    qsa.sparse_attn(to_dev(q), Kd, Vd, to_dev(np.array([68, 10], np.int32)), max_cells, out,
                    H_kv, d, d, 0.1, lse=lse, workspace=ws)
    assert np.all(np.isnan(to_host(out)[0])) and np.all(np.isnan(to_host(lse)[0]))
    assert np.all(np.isfinite(to_host(out)[1]))


# ------------------------------------------------------------------ whole decode step

@pytest.mark.parametrize("shape,steps", [(TINY, 6), (SMALL_BF16, 5)], ids=lambda x: getattr(x, "name", str(x)))
def test_decode_steps_end_to_end(shape, steps):
    """Several appending decode steps through DecodeLayer vs the oracle's step."""
    inp = qsa_synth.decode_inputs(shape, seed=11, extra_tokens=steps, n_steps=steps)
    H, d = shape.H_idx, shape.d_idx
    raw, w = to_dev(inp["raw_k"]), to_dev(inp["norm_w"])
    K, V = to_dev(inp["K"]), to_dev(inp["V"])
    layer = qsa.DecodeLayer(cap_tokens=shape.n_ctx + steps, H_idx=H, d_idx=d, H_q=shape.H_q,
                            H_kv=shape.H_kv, d=shape.d, top_k_tokens=shape.top_k_tokens,
                            eps=shape.eps, rope_base=shape.rope_base)
    n0 = shape.n_ctx - 1
    layer.rebuild(raw, w, n0)
    o_pooled = oracle.pool_rows(inp["raw_k"], n0, H, d, inp["norm_w"], shape.eps, shape.rope_base,
                                0, (n0 + 3) // 4, np.zeros(((shape.n_ctx + steps + 3) // 4, H * d),
                                                          np.float32))
    o_valid = n0 // 4
    for s in range(steps):
        n_ctx = n0 + 1 + s
        out = layer.step(raw, w, K, V, n_ctx, to_dev(inp["q_idx"][s]), to_dev(inp["q"][s]))
        blocks, cells, o_out, _, o_scores = oracle.decode_step(
            inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps, shape.rope_base, o_pooled,
            o_valid, inp["q_idx"][s], shape.top_k_tokens, inp["q"][s], inp["K"], inp["V"],
            shape.H_q, shape.H_kv, shape.d)
        o_valid = n_ctx // 4
        g_blocks = to_host(layer.blocks)[0]
        g_count = int(to_host(layer.counts)[0])
        n_band = check_topk(g_blocks, g_count, o_scores, n_ctx // 4, shape.k_blk)
        g_cells = to_host(layer.pos)[0, :int(to_host(layer.n_cells)[0])]
        if np.array_equal(np.sort(g_blocks[:g_count]), blocks):
            np.testing.assert_array_equal(g_cells, cells)
            np.testing.assert_allclose(to_host(out)[0], o_out, rtol=0, atol=_atol(shape))
        else:
            assert n_band > 0


def test_decode_step_composite_equals_separate_calls():
    """qsa_decode_step (cell list written by the top-k kernel) and the five separate calls
    (cell list from qsa_gather_kv) give bit-identical outputs."""
    shape = SMALL_BF16
    inp = qsa_synth.decode_inputs(shape, seed=12, extra_tokens=3, n_steps=3)
    raw, w = to_dev(inp["raw_k"]), to_dev(inp["norm_w"])
    K, V = to_dev(inp["K"]), to_dev(inp["V"])
    kw = dict(cap_tokens=shape.n_ctx + 3, H_idx=shape.H_idx, d_idx=shape.d_idx, H_q=shape.H_q,
              H_kv=shape.H_kv, d=shape.d, top_k_tokens=shape.top_k_tokens)
    a, b = qsa.DecodeLayer(**kw), qsa.DecodeLayer(**kw)
    a.rebuild(raw, w, shape.n_ctx - 1)
    b.rebuild(raw, w, shape.n_ctx - 1)
    for s in range(3):
        n_ctx = shape.n_ctx + s
        oa = a.step(raw, w, K, V, n_ctx, to_dev(inp["q_idx"][s]), to_dev(inp["q"][s])).clone()
        ob = b.step_separate_calls(raw, w, K, V, n_ctx, to_dev(inp["q_idx"][s]),
                                   to_dev(inp["q"][s])).clone()
        assert torch.equal(a.pooled, b.pooled)
        assert torch.equal(a.blocks, b.blocks) and torch.equal(a.n_cells, b.n_cells)
        nc = int(a.n_cells.item())
        assert torch.equal(a.pos[0, :nc], b.pos[0, :nc])
        assert torch.equal(oa, ob)


def test_decode_step_with_uninitialised_workspace():
    """A workspace holding garbage (never cleared) still gives the same results: the top-k
    kernel notices that the histogram's total disagrees with the block count and rebuilds
    it from the scores."""
    shape = SMALL_BF16
    inp = qsa_synth.decode_inputs(shape, seed=13, extra_tokens=2, n_steps=2)
    raw, w = to_dev(inp["raw_k"]), to_dev(inp["norm_w"])
    K, V = to_dev(inp["K"]), to_dev(inp["V"])
    kw = dict(cap_tokens=shape.n_ctx + 2, H_idx=shape.H_idx, d_idx=shape.d_idx, H_q=shape.H_q,
              H_kv=shape.H_kv, d=shape.d, top_k_tokens=shape.top_k_tokens)
    a, b = qsa.DecodeLayer(**kw), qsa.DecodeLayer(**kw)
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    a.workspace.view(torch.int32).random_(0, 1 << 20, generator=g)
    for lay in (a, b):
        lay.rebuild(raw, w, shape.n_ctx - 1)
    for s in range(2):
        n_ctx = shape.n_ctx + s
        oa = a.step(raw, w, K, V, n_ctx, to_dev(inp["q_idx"][s]), to_dev(inp["q"][s])).clone()
        ob = b.step_separate_calls(raw, w, K, V, n_ctx, to_dev(inp["q_idx"][s]),
                                   to_dev(inp["q"][s])).clone()
        assert torch.equal(a.blocks, b.blocks)
        assert torch.equal(oa, ob)
