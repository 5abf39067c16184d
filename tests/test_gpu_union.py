"""Grouped-union sparse attention (qsa_sparse_attn_union) against the oracle's attention over
each query's own cells, and against qsa_sparse_attn on the same lists.

The union kernel stages, for each group of 16 consecutive queries, the union of the blocks
the group selected, and masks every query to its own cells; its result must be the plain
per-query attention (max abs error 2e-3 for bf16 K/V with fp32 accumulation).  Cases cover
groups that share most, some or none of their blocks, a ragged last group, open-block tails
at every offset, an empty list, a truncated list (NaN) and cells outside the cache."""
import math

import numpy as np
import pytest
import torch

import gather_qsa_pool_gb300 as qsa
import qsa_synth
from gpu_helpers import ATOL_ATTN_BF16, to_dev, to_host
from oracle import oracle

pytestmark = pytest.mark.gpu


def _lists(n_q, p0, k_blk, share, seed, max_cells):
    """Cell lists of queries at positions p0 .. p0+n_q-1: block lists with the given share
    inside each group of 16, expanded to cells plus each query's open tail by the oracle."""
    pos_q = p0 + np.arange(n_q)
    n_cand = (pos_q + 1) // 4
    blocks = qsa_synth.overlap_block_lists(n_cand, k_blk, 16, share, seed)
    pos = np.full((n_q, max_cells), -1, np.int32)
    n = np.zeros(n_q, np.int32)
    cells = []
    for i in range(n_q):
        cl = oracle.cells(blocks[i], int(pos_q[i]))
        pos[i, :cl.shape[0]] = cl
        n[i] = cl.shape[0]
        cells.append(cl)
    return pos, n, cells


def _run_union(q, K, V, pos, n, max_cells, H_kv, d, scale, lse=True):
    n_q, H_q = q.shape[0], q.shape[1]
    out = torch.full((n_q, H_q, d), float("nan"), device="cuda")
    l = torch.full((n_q, H_q), float("nan"), device="cuda") if lse else None
    ws = torch.empty(qsa.sparse_attn_union_workspace_size(n_q, max_cells), dtype=torch.uint8,
                     device="cuda")
    qsa.sparse_attn_union(q, K, V, n, max_cells, out, H_kv, d, scale, pos, lse=l, workspace=ws)
    return out, l


@pytest.mark.parametrize("share,n_q,H_kv,p0,seed", [
    (0.9, 40, 2, 1501, 1),    # mostly shared; ragged last group (8 queries)
    (0.5, 32, 1, 2222, 2),    # half shared; one KV head
    (0.0, 17, 4, 3003, 3),    # independent selections; a group of one query
    (1.0, 16, 2, 1800, 4),    # identical selections (only the tails differ)
])
def test_union_matches_oracle_per_query(share, n_q, H_kv, p0, seed):
    d, k_blk = 128, 64
    max_cells = 4 * k_blk + 3
    n_kv = p0 + n_q + 5
    rng = np.random.default_rng(seed)
    H_q = 8 * H_kv
    K = qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, H_kv, d)).astype(np.float32))
    V = qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, H_kv, d)).astype(np.float32))
    q = rng.standard_normal((n_q, H_q, d)).astype(np.float32)
    pos, n, cells = _lists(n_q, p0, k_blk, share, seed, max_cells)
    scale = 1.0 / math.sqrt(d)
    Kd, Vd = to_dev(K), to_dev(V)
    out, lse = _run_union(to_dev(q), Kd, Vd, to_dev(pos), to_dev(n), max_cells, H_kv, d, scale)
    g_out, g_lse = to_host(out), to_host(lse)
    for i in range(n_q):
        want, want_lse = oracle.attention(q[i], K, V, H_q, H_kv, d, d, H_kv * d, H_kv * d,
                                          cells[i], scale)
        np.testing.assert_allclose(g_out[i], want, rtol=0, atol=ATOL_ATTN_BF16)
        np.testing.assert_allclose(g_lse[i], want_lse, rtol=0, atol=1e-4)
    # the same lists through qsa_sparse_attn
    ref = torch.empty(n_q, H_q, d, device="cuda")
    ws = torch.empty(max(qsa.sparse_attn_workspace_size(n_q, H_q, H_kv, d, max_cells) // 4, 1),
                     device="cuda")
    qsa.sparse_attn(to_dev(q), Kd, Vd, to_dev(n), max_cells, ref, H_kv, d, d, scale,
                    pos=to_dev(pos), workspace=ws)
    np.testing.assert_allclose(g_out, to_host(ref), rtol=0, atol=ATOL_ATTN_BF16)


def test_union_special_lists():
    """An empty list (output 0, lse -inf), a truncated list (NaN), a list with cells outside
    the cache (skipped) and a single cell (output = its V row), in one group with ordinary
    lists."""
    d, H_kv, k_blk = 128, 2, 32
    H_q, n_q, p0 = 16, 20, 900
    max_cells = 4 * k_blk + 3
    n_kv = p0 + n_q
    rng = np.random.default_rng(77)
    K = qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, H_kv, d)).astype(np.float32))
    V = qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, H_kv, d)).astype(np.float32))
    q = rng.standard_normal((n_q, H_q, d)).astype(np.float32)
    pos, n, cells = _lists(n_q, p0, k_blk, 0.6, 9, max_cells)
    n[3] = 0                                  # empty
    n[5] = max_cells + 1                      # truncated
    pos[7, 0], pos[7, 5] = -3, n_kv + 11      # outside the cache: skipped
    cells[7] = np.array([c for c in pos[7, :n[7]] if 0 <= c < n_kv], np.int32)
    pos[18, 0], n[18] = 123, 1                # a single cell
    cells[18] = np.array([123], np.int32)
    scale = 1.0 / math.sqrt(d)
    out, lse = _run_union(to_dev(q), to_dev(K), to_dev(V), to_dev(pos), to_dev(n), max_cells,
                          H_kv, d, scale)
    g_out, g_lse = to_host(out), to_host(lse)
    assert np.all(g_out[3] == 0) and np.all(np.isneginf(g_lse[3]))
    assert np.all(np.isnan(g_out[5])) and np.all(np.isnan(g_lse[5]))
    vrow = qsa_synth.bf16_bits_to_f32(V[123]).reshape(H_kv, d)
    np.testing.assert_allclose(g_out[18], np.repeat(vrow, 8, axis=0), rtol=0, atol=1e-6)
    for i in range(n_q):
        if i in (3, 5):
            continue
        want, want_lse = oracle.attention(q[i], K, V, H_q, H_kv, d, d, H_kv * d, H_kv * d,
                                          cells[i], scale)
        np.testing.assert_allclose(g_out[i], want, rtol=0, atol=ATOL_ATTN_BF16)
        np.testing.assert_allclose(g_lse[i], want_lse, rtol=0, atol=1e-4)


def test_union_prefill_chunk_255181_against_per_query_kernel():
    """The 1024-query chunk after 255,181 tokens, with lists whose groups share 90% of their
    blocks (512 per query), in the benchmark's launch configuration: every output against
    qsa_sparse_attn over the same lists, a sample against the oracle."""
    shape = qsa_synth.CONFIGS["prefill_256k"]
    n_q, n_ctx, d, H_kv, H_q = shape.n_q, shape.n_ctx, shape.d, shape.H_kv, shape.H_q
    g = torch.Generator(device="cuda")
    g.manual_seed(2561)
    K = torch.randn(n_ctx, H_kv, d, generator=g, device="cuda").to(torch.bfloat16)
    V = torch.randn(n_ctx, H_kv, d, generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn(n_q, H_q, d, generator=g, device="cuda")
    q_pos = shape.depth + np.arange(n_q)
    blocks = qsa_synth.overlap_block_lists((q_pos + 1) // 4, shape.k_blk, 16, 0.9, 2562)
    bl = np.zeros((n_q, shape.k_blk), np.int32)
    cnt = np.zeros(n_q, np.int32)
    for i, b in enumerate(blocks):
        bl[i, :b.shape[0]] = b
        cnt[i] = b.shape[0]
    pos = torch.empty(n_q, shape.max_cells, dtype=torch.int32, device="cuda")
    n = torch.empty(n_q, dtype=torch.int32, device="cuda")
    qsa.gather_kv(to_dev(bl), to_dev(cnt), shape.k_blk, pos, n, shape.max_cells,
                  q_pos=to_dev(q_pos.astype(np.int32)), n_kv=n_ctx)
    scale = 1.0 / math.sqrt(d)
    out, lse = _run_union(q, K, V, pos, n, shape.max_cells, H_kv, d, scale)
    ref = torch.empty(n_q, H_q, d, device="cuda")
    ref_lse = torch.empty(n_q, H_q, device="cuda")
    qsa.sparse_attn(q, K, V, n, shape.max_cells, ref, H_kv, d, d, scale, pos=pos, lse=ref_lse)
    g_out = to_host(out)
    np.testing.assert_allclose(g_out, to_host(ref), rtol=0, atol=ATOL_ATTN_BF16)
    np.testing.assert_allclose(to_host(lse), to_host(ref_lse), rtol=0, atol=1e-4)
    Kh, Vh, qh = to_host(K), to_host(V), to_host(q)
    g_pos, g_n = to_host(pos), to_host(n)
    for i in (0, 15, 16, 500, 1023):
        cl = g_pos[i, :g_n[i]]
        np.testing.assert_array_equal(cl, oracle.cells(blocks[i], int(q_pos[i])))
        want, _ = oracle.attention(qh[i], Kh, Vh, H_q, H_kv, d, d, H_kv * d, H_kv * d, cl, scale)
        np.testing.assert_allclose(g_out[i], want, rtol=0, atol=ATOL_ATTN_BF16)
