"""GPU parity of the mask-driven variant (mask -> position list, attention over the list)
and of the prefill-chunk path (per-query causal scores, per-query top-k, gathered
attention) against the fp64 oracle."""
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


# ------------------------------------------------------------------ a7 mask -> list

@pytest.mark.parametrize("n_kv,ld_pad", [(32768, 0), (100_000, 0), (1000, 0), (64, 0), (63, 0),
                                         (1, 0), (65_600, 0), (4096, 4)])
def test_mask_to_list(n_kv, ld_pad):
    """Rows of whole 64-key words on 16-byte boundaries (read 64 bytes a thread), ragged rows
    and rows whose stride breaks the alignment (ballots), one and two chunks of 65,536."""
    n_rows, max_list = 3, 2048
    m = qsa_synth.mask_rows(n_rows, n_kv, seed=n_kv)
    if n_kv >= 64:
        m[1, :] = 0            # empty row
    wide = np.zeros((n_rows, n_kv + ld_pad), np.uint8)
    wide[:, :n_kv] = m
    wide[:, n_kv:] = 1         # past the row: never listed
    pos = torch.full((n_rows, max_list), -3, dtype=torch.int32, device="cuda")
    counts = torch.zeros(n_rows, dtype=torch.int32, device="cuda")
    bits = torch.zeros((n_rows, (n_kv + 63) // 64), dtype=torch.int64, device="cuda")
    qsa.mask_to_list(to_dev(wide), max_list, pos, counts, bits, n_kv=n_kv)
    g_pos, g_cnt, g_bits = to_host(pos), to_host(counts), to_host(bits).view(np.uint64)
    for r in range(n_rows):
        w_pos, w_cnt, w_bits = oracle.mask_to_list(m[r], max_list)
        assert g_cnt[r] == w_cnt
        np.testing.assert_array_equal(g_pos[r, :min(w_cnt, max_list)], w_pos)
        assert np.all(g_pos[r, min(w_cnt, max_list):] == -3)
        np.testing.assert_array_equal(g_bits[r], w_bits)


def test_mask_to_list_overflow_keeps_true_count():
    m = np.ones((2, 5000), np.uint8)
    m[1, ::3] = 0
    pos = torch.zeros((2, 2048), dtype=torch.int32, device="cuda")
    counts = torch.zeros(2, dtype=torch.int32, device="cuda")
    qsa.mask_to_list(to_dev(m), 2048, pos, counts)
    for r in range(2):
        w_pos, w_cnt, _ = oracle.mask_to_list(m[r], 2048)
        assert int(to_host(counts)[r]) == w_cnt > 2048
        np.testing.assert_array_equal(to_host(pos)[r], w_pos)


# ------------------------------------------------------------------ a8 mask-mode attention

def test_mask_mode_attention_dkq576():
    """DKQ 576 / d_v 512, 16 query heads on one KV head, V = first 512 columns of each
    K row, bf16; list from the mask; one row overflowing its list gives NaN."""
    shape = qsa_synth.CONFIGS["mask_32k"]
    inp = qsa_synth.mask_attn_inputs(shape, seed=4)
    m = qsa_synth.mask_rows(shape.n_q, shape.n_kv, seed=5)
    m[3, :] = 0
    m[3, 100:100 + 3000] = 1   # 3000 set positions: more than the 2048-entry list
    assert qsa.mask_sparse_eligible(True, 0.0, 0.0, shape.n_kv, shape.max_list)
    KV = to_dev(inp["KV"])
    pos = torch.zeros((shape.n_q, shape.max_list), dtype=torch.int32, device="cuda")
    counts = torch.zeros(shape.n_q, dtype=torch.int32, device="cuda")
    qsa.mask_to_list(to_dev(m), shape.max_list, pos, counts)
    out = torch.zeros((shape.n_q, shape.H_q, shape.d_v), device="cuda")
    lse = torch.zeros((shape.n_q, shape.H_q), device="cuda")
    ws_n = qsa.sparse_attn_workspace_size(shape.n_q, shape.H_q, 1, shape.d_v, shape.max_list)
    ws = torch.empty(max(ws_n // 4, 1), device="cuda")
    scale = 1.0 / math.sqrt(shape.d_k)
    qsa.sparse_attn(to_dev(inp["q"]), KV, KV, counts, shape.max_list, out, 1, shape.d_k,
                    shape.d_v, scale, pos=pos, lse=lse, workspace=ws, ld_k=shape.d_k,
                    ld_v=shape.d_k)
    g_out, g_lse = to_host(out), to_host(lse)
    for r in range(shape.n_q):
        w_pos, w_cnt, _ = oracle.mask_to_list(m[r], shape.max_list)
        if w_cnt > shape.max_list:
            assert np.all(np.isnan(g_out[r])) and np.all(np.isnan(g_lse[r]))
            continue
        want, want_lse = oracle.attention(inp["q"][r], inp["KV"], inp["KV"], shape.H_q, 1,
                                          shape.d_k, shape.d_v, shape.d_k, shape.d_k, w_pos, scale)
        np.testing.assert_allclose(g_out[r], want, rtol=0, atol=ATOL_ATTN_BF16)
        np.testing.assert_allclose(g_lse[r], want_lse, rtol=1e-5, atol=1e-4)


# ------------------------------------------------------------------ a6 prefill chunk

def _prefill_case(dtype, depth, n_q, k_tokens, seed):
    shape = qsa_synth.PrefillShape("prefill_small", depth, n_q, 4, 64, 8, 2, 128, k_tokens,
                                   dtype=dtype)
    return shape, qsa_synth.prefill_inputs(shape, seed)


@pytest.mark.parametrize("H,d,depth,n_q", [(4, 64, 3001, 130), (16, 128, 10000, 600)])
def test_prefill_scores_on_tensor_cores(H, d, depth, n_q):
    """qsa_index_score with QSA_PREC_BF16_TC (tcgen05, bf16 operands, fp32 accumulation)
    against the oracle with both operands rounded to bf16; rows a query cannot see are
    -inf.  Shapes cover partial query and row tiles."""
    shape = qsa_synth.PrefillShape("tc", depth, n_q, H, d, 8, 2, 128, 256, dtype="bf16")
    inp = qsa_synth.prefill_inputs(shape, seed=31)
    n_rows = shape.n_rows
    o_pooled = oracle.pool_rows(inp["raw_k"], shape.n_ctx, H, d, inp["norm_w"], shape.eps,
                                shape.rope_base, 0, n_rows)
    scale = 1.0 / math.sqrt(d)
    ws = torch.zeros(qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC),
                     dtype=torch.uint8, device="cuda")
    scores = torch.full((n_q, n_rows + 5), 7.0, device="cuda")
    qsa.index_score(to_dev(inp["q_idx"]), to_dev(o_pooled), n_rows, H, d, scale, scores,
                    q_pos=to_dev(inp["q_pos"]), precision=qsa.QSA_PREC_BF16_TC, workspace=ws)
    got = to_host(scores)
    assert np.all(got[:, n_rows:] == 7.0)
    rows = np.arange(n_q) if n_q <= 130 else np.random.default_rng(3).choice(n_q, 48, replace=False)
    want = oracle.scores(inp["q_idx"][rows], o_pooled, n_rows, H, d, scale,
                         q_pos=inp["q_pos"][rows], round_bf16_operands=True)
    qb = np.array([oracle.round_bf16(float(x)) for x in inp["q_idx"][rows].reshape(-1)],
                  np.float32).reshape(len(rows), -1)
    for j, i in enumerate(rows):
        vis = np.isfinite(want[j])
        assert np.array_equal(np.isneginf(got[i, :n_rows]), ~vis)
        tol = score_tolerance(qb[j], o_pooled, n_rows, scale, chain=H * d)[vis]
        assert np.all(np.abs(got[i, :n_rows][vis] - want[j][vis]) <= tol)


@pytest.mark.parametrize("dtype,depth,n_q,k_tokens,prec", [("f32", 3001, 64, 256, "f32"),
                                                           ("bf16", 700, 130, 1024, "f32"),
                                                           ("bf16", 2900, 200, 512, "tc")])
def test_prefill_chunk(dtype, depth, n_q, k_tokens, prec):
    shape, inp = _prefill_case(dtype, depth, n_q, k_tokens, seed=21)
    tc = prec == "tc"
    H, d, n_ctx = shape.H_idx, shape.d_idx, shape.n_ctx
    n_rows, k_blk, max_cells = shape.n_rows, shape.k_blk, shape.max_cells
    scale_idx = 1.0 / math.sqrt(d)
    # oracle
    o_pooled = oracle.pool_rows(inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps,
                                shape.rope_base, 0, n_rows)
    o_scores = oracle.scores(inp["q_idx"], o_pooled, n_rows, H, d, scale_idx, q_pos=inp["q_pos"],
                             round_bf16_operands=tc)
    # GPU
    pooled = torch.zeros(n_rows, H * d, device="cuda")
    qsa.pool_update(to_dev(inp["raw_k"]), n_ctx, H, d, to_dev(inp["norm_w"]), shape.eps,
                    shape.rope_base, pooled, 0)
    q_pos = to_dev(inp["q_pos"])
    scores = torch.zeros(n_q, n_rows, device="cuda")
    if tc:
        ws = torch.zeros(qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC),
                         dtype=torch.uint8, device="cuda")
        qsa.index_score(to_dev(inp["q_idx"]), pooled, n_rows, H, d, scale_idx, scores,
                        q_pos=q_pos, precision=qsa.QSA_PREC_BF16_TC, workspace=ws)
    else:
        qsa.index_score(to_dev(inp["q_idx"]), pooled, n_rows, H, d, scale_idx, scores,
                        q_pos=q_pos)
    blocks = torch.zeros(n_q, k_blk, dtype=torch.int32, device="cuda")
    counts = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(scores, n_ctx // 4, k_blk, blocks, counts, q_pos=q_pos)
    pos = torch.zeros(n_q, max_cells, dtype=torch.int32, device="cuda")
    n_cells = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    K, V = to_dev(inp["K"]), to_dev(inp["V"])
    qsa.gather_kv(blocks, counts, k_blk, pos, n_cells, max_cells, q_pos=q_pos, n_kv=n_ctx)
    out = torch.zeros(n_q, shape.H_q, shape.d, device="cuda")
    ws = torch.empty(max(qsa.sparse_attn_workspace_size(n_q, shape.H_q, shape.H_kv, shape.d,
                                                        max_cells) // 4, 1), device="cuda")
    qsa.sparse_attn(to_dev(inp["q"]), K, V, n_cells, max_cells, out, shape.H_kv, shape.d,
                    shape.d, 1.0 / math.sqrt(shape.d), pos=pos, workspace=ws)
    g_scores, g_blocks, g_counts = to_host(scores), to_host(blocks), to_host(counts)
    g_out, g_pos, g_nc = to_host(out), to_host(pos), to_host(n_cells)
    atol = ATOL_ATTN_BF16 if dtype == "bf16" else ATOL_ATTN_F32
    checked = 0
    for i in range(n_q):
        p = int(inp["q_pos"][i])
        nf = (p + 1) // 4
        assert np.all(np.isneginf(g_scores[i, nf:n_rows]))
        n_band = check_topk(g_blocks[i], int(g_counts[i]), o_scores[i], nf, k_blk)
        w_blocks = oracle.topk(o_scores[i], nf, k_blk)
        if not np.array_equal(g_blocks[i, :g_counts[i]], w_blocks):
            assert n_band > 0
            continue
        cells = oracle.cells(w_blocks, p)
        np.testing.assert_array_equal(g_pos[i, :g_nc[i]], cells)
        want, _ = oracle.attention(inp["q"][i], inp["K"], inp["V"], shape.H_q, shape.H_kv,
                                   shape.d, shape.d, shape.H_kv * shape.d, shape.H_kv * shape.d,
                                   cells, 1.0 / math.sqrt(shape.d))
        np.testing.assert_allclose(g_out[i], want, rtol=0, atol=atol)
        checked += 1
    assert checked >= n_q - 2


@pytest.mark.parametrize("n_q,lens", [(1, [2048]), (4, [0, 1, 65, 2048]), (3, [63, 64, 129]),
                                      (160, None)])
def test_latent_attention_list_lengths(n_q, lens):
    """The latent-KV form (DKQ 576, d_v 512, 16 heads, V = first 512 columns of the K row)
    over position lists of many lengths: empty, one cell, stage edges, a full list; 160
    queries take the one-CTA-per-query path.  Every output against the oracle."""
    n_kv, d_k, d_v, H, max_list = 5000, 576, 512, 16, 2048
    rng = np.random.default_rng(n_q)
    KV = qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, d_k)).astype(np.float32))
    q = rng.standard_normal((n_q, H, d_k)).astype(np.float32)
    if lens is None:
        lens = list(rng.integers(0, 300, size=n_q))
    pos = np.full((n_q, max_list), -7, np.int32)
    for i, L in enumerate(lens):
        pos[i, :L] = np.sort(rng.choice(n_kv, size=L, replace=False))
    counts = np.array(lens, np.int32)
    out = torch.zeros((n_q, H, d_v), device="cuda")
    lse = torch.zeros((n_q, H), device="cuda")
    scale = 1.0 / math.sqrt(d_k)
    kv = to_dev(KV)
    ws_n = qsa.sparse_attn_workspace_size(n_q, H, 1, d_v, max_list)
    ws = torch.empty(max(ws_n // 4, 1), device="cuda")
    qsa.sparse_attn(to_dev(q), kv, kv, to_dev(counts), max_list, out, 1, d_k, d_v, scale,
                    pos=to_dev(pos), lse=lse, workspace=ws, ld_k=d_k, ld_v=d_k)
    g_out, g_lse = to_host(out), to_host(lse)
    for i, L in enumerate(lens):
        if L == 0:
            assert np.all(g_out[i] == 0.0) and np.all(np.isneginf(g_lse[i]))
            continue
        want, want_lse = oracle.attention(q[i], KV, KV, H, 1, d_k, d_v, d_k, d_k, pos[i, :L],
                                          scale)
        np.testing.assert_allclose(g_out[i], want, rtol=0, atol=ATOL_ATTN_BF16)
        np.testing.assert_allclose(g_lse[i], want_lse, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("case", ["32k", "ragged", "unaligned", "overflow", "max_kv", "many"])
def test_mask_sparse_attn_one_call(case):
    """qsa_mask_sparse_attn (each query's list built from its mask row inside the attention
    kernel) against the oracle's list and attention, and bit for bit against the two-call
    path (qsa_mask_to_list, then qsa_sparse_attn) on the same inputs: rows of whole aligned
    64-key words, a ragged key count, row strides off the 16-byte grid, a list overflow
    (NaN result, true count), an empty row, the longest rows (65,536 keys) and 160 queries
    (one CTA per query, no cluster)."""
    d_k, d_v, H, max_list = 576, 512, 16, 2048
    n_q, n_kv, pad, dens = {"32k": (4, 32768, 0, 0.06), "ragged": (3, 5000, 0, 0.1),
                            "unaligned": (4, 4096, 3, 0.2), "overflow": (2, 5000, 0, 0.6),
                            "max_kv": (2, 65536, 0, 0.03), "many": (160, 8192, 0, 0.02)}[case]
    rng = np.random.default_rng(len(case) * 31 + n_kv)
    KV = qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, d_k)).astype(np.float32))
    q = rng.standard_normal((n_q, H, d_k)).astype(np.float32)
    m = (rng.random((n_q, n_kv)) < dens).astype(np.uint8)
    if case == "ragged":
        m[1, :] = 0                                    # empty row
    wide = np.zeros((n_q, n_kv + pad), np.uint8)
    wide[:, :n_kv] = m * rng.integers(1, 256, size=m.shape).astype(np.uint8)  # any nonzero byte
    wide[:, n_kv:] = 1                                 # past the row: never listed
    kv, d_mask, d_q = to_dev(KV), to_dev(wide), to_dev(q)
    scale = 1.0 / math.sqrt(d_k)
    out = torch.full((n_q, H, d_v), -5.0, device="cuda")
    lse = torch.full((n_q, H), -5.0, device="cuda")
    cnt = torch.full((n_q,), -1, dtype=torch.int32, device="cuda")
    qsa.mask_sparse_attn(d_q, kv, d_mask, max_list, out, scale, counts_out=cnt, lse=lse,
                         n_kv=n_kv)
    # the two-call path
    pos = torch.zeros((n_q, max_list), dtype=torch.int32, device="cuda")
    cnt2 = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    qsa.mask_to_list(d_mask, max_list, pos, cnt2, n_kv=n_kv)
    out2 = torch.zeros((n_q, H, d_v), device="cuda")
    lse2 = torch.zeros((n_q, H), device="cuda")
    ws_n = qsa.sparse_attn_workspace_size(n_q, H, 1, d_v, max_list)
    ws = torch.empty(max(ws_n // 4, 1), device="cuda")
    qsa.sparse_attn(d_q, kv, kv, cnt2, max_list, out2, 1, d_k, d_v, scale, pos=pos, lse=lse2,
                    workspace=ws, ld_k=d_k, ld_v=d_k, n_kv=n_kv)
    g_out, g_lse, g_cnt = to_host(out), to_host(lse), to_host(cnt)
    np.testing.assert_array_equal(g_cnt, to_host(cnt2))
    np.testing.assert_array_equal(g_out.view(np.uint32), to_host(out2).view(np.uint32))
    np.testing.assert_array_equal(g_lse.view(np.uint32), to_host(lse2).view(np.uint32))
    for r in range(n_q) if n_q <= 8 else range(0, n_q, 23):
        w_pos, w_cnt, _ = oracle.mask_to_list(m[r], max_list)
        assert g_cnt[r] == w_cnt
        if w_cnt > max_list:
            assert np.all(np.isnan(g_out[r])) and np.all(np.isnan(g_lse[r]))
        elif w_cnt == 0:
            assert np.all(g_out[r] == 0.0) and np.all(np.isneginf(g_lse[r]))
        else:
            want, want_lse = oracle.attention(q[r], KV, KV, H, 1, d_k, d_v, d_k, d_k, w_pos,
                                              scale)
            np.testing.assert_allclose(g_out[r], want, rtol=0, atol=ATOL_ATTN_BF16)
            np.testing.assert_allclose(g_lse[r], want_lse, rtol=1e-5, atol=1e-4)
    if case == "overflow":
        assert np.all(g_cnt > max_list)


def test_dkq576_with_separate_values():
    """DKQ 576 / d_v 512 with a V tensor of its own (not the K row's first columns): the
    general attention kernel, against the oracle."""
    n_kv, d_k, d_v, H, max_list, n_q = 3000, 576, 512, 16, 512, 2
    rng = np.random.default_rng(99)
    K = qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, d_k)).astype(np.float32))
    V = qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, d_v)).astype(np.float32))
    q = rng.standard_normal((n_q, H, d_k)).astype(np.float32)
    lens = [300, 512]
    pos = np.zeros((n_q, max_list), np.int32)
    for i, L in enumerate(lens):
        pos[i, :L] = np.sort(rng.choice(n_kv, size=L, replace=False))
    out = torch.zeros((n_q, H, d_v), device="cuda")
    ws_n = qsa.sparse_attn_workspace_size(n_q, H, 1, d_v, max_list)
    ws = torch.empty(max(ws_n // 4, 1), device="cuda")
    scale = 1.0 / math.sqrt(d_k)
    qsa.sparse_attn(to_dev(q), to_dev(K), to_dev(V), to_dev(np.array(lens, np.int32)), max_list,
                    out, 1, d_k, d_v, scale, pos=to_dev(pos), workspace=ws, ld_k=d_k, ld_v=d_v)
    g_out = to_host(out)
    for i, L in enumerate(lens):
        want, _ = oracle.attention(q[i], K, V, H, 1, d_k, d_v, d_k, d_v, pos[i, :L], scale)
        np.testing.assert_allclose(g_out[i], want, rtol=0, atol=ATOL_ATTN_BF16)


def test_prefill_attention_all_heads_per_query():
    """Many queries with 4 KV heads x 8 query heads (bf16, 128 dims) and position lists: one
    CTA per query stages whole cell rows.  List lengths cover empty, one cell, the 32-cell
    stage edges, the three-stage ring and a full 2051-cell list; every output and log-sum-exp
    against the oracle."""
    n_q, H_kv, G, d, n_kv, max_cells = 48, 4, 8, 128, 9000, 2051
    H_q = H_kv * G
    rng = np.random.default_rng(2051)
    K = qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, H_kv * d)).astype(np.float32))
    V = qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, H_kv * d)).astype(np.float32))
    q = rng.standard_normal((n_q, H_q, d)).astype(np.float32)
    edge = [0, 1, 31, 32, 33, 63, 64, 65, 95, 96, 97, 129, 2051]
    lens = edge + list(rng.integers(1, max_cells + 1, size=n_q - len(edge)))
    pos = np.full((n_q, max_cells), -9, np.int32)
    for i, L in enumerate(lens):
        pos[i, :L] = np.sort(rng.choice(n_kv, size=L, replace=False))
    pos[5, 3] = -1  # a skipped entry inside a list
    out = torch.zeros((n_q, H_q, d), device="cuda")
    lse = torch.zeros((n_q, H_q), device="cuda")
    ws_n = qsa.sparse_attn_workspace_size(n_q, H_q, H_kv, d, max_cells)
    ws = torch.empty(max(ws_n // 4, 1), device="cuda")
    scale = 1.0 / math.sqrt(d)
    qsa.sparse_attn(to_dev(q), to_dev(K), to_dev(V), to_dev(np.array(lens, np.int32)), max_cells,
                    out, H_kv, d, d, scale, pos=to_dev(pos), lse=lse, workspace=ws)
    g_out, g_lse = to_host(out), to_host(lse)
    for i, L in enumerate(lens):
        if L == 0:
            assert np.all(g_out[i] == 0.0) and np.all(np.isneginf(g_lse[i]))
            continue
        cells = pos[i, :L]
        cells = cells[cells >= 0]
        want, want_lse = oracle.attention(q[i], K, V, H_q, H_kv, d, d, H_kv * d, H_kv * d, cells,
                                          scale)
        np.testing.assert_allclose(g_out[i], want, rtol=0, atol=ATOL_ATTN_BF16)
        np.testing.assert_allclose(g_lse[i], want_lse, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("ld_pad", [0, 64], ids=["contiguous", "strided"])
def test_prefill_attention_block_lists(ld_pad):
    """Lists made of whole 4-token blocks (the prefill selections) and a tail: groups of four
    consecutive rows are staged by one copy when the cache rows are contiguous (ld_pad 0) and
    row by row otherwise; lists whose groups are broken (a skipped entry, a two-cell shift, a
    gap) take the row-by-row form.  Every output and log-sum-exp against the oracle."""
    n_q, H_kv, G, d, n_kv, max_cells = 40, 4, 8, 128, 9000, 2051
    H_q, ld = H_kv * G, H_kv * d + ld_pad
    rng = np.random.default_rng(4096 + ld_pad)
    K = qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, ld)).astype(np.float32))
    V = qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, ld)).astype(np.float32))
    q = rng.standard_normal((n_q, H_q, d)).astype(np.float32)
    edge = [0, 1, 3, 4, 5, 31, 32, 33, 36, 64, 97, 2048, 2049, 2051]
    lens = edge + list(rng.integers(1, max_cells + 1, size=n_q - len(edge)))
    pos = np.full((n_q, max_cells), -9, np.int32)
    n_blk = n_kv // 4
    for i, L in enumerate(lens):
        nb, tail = L // 4, L % 4
        b = np.sort(rng.choice(n_blk - 1, size=nb, replace=False))
        cells = (4 * b[:, None] + np.arange(4)).reshape(-1)
        t0 = 4 * (n_blk - 1)
        pos[i, :L] = np.concatenate([cells, t0 + np.arange(tail)]).astype(np.int32)
    pos[20, 6] = -1                                   # a skipped entry inside a group
    pos[21, :lens[21]] = np.sort(np.concatenate([[3, 7], pos[21, 2:lens[21]] + 8]))[:lens[21]]
    pos[22, 5] += 1                                   # a gap: the group is not consecutive
    pos[22, 6:8] += 1
    out = torch.zeros((n_q, H_q, d), device="cuda")
    lse = torch.zeros((n_q, H_q), device="cuda")
    ws = torch.empty(max(qsa.sparse_attn_workspace_size(n_q, H_q, H_kv, d, max_cells) // 4, 1),
                     device="cuda")
    scale = 1.0 / math.sqrt(d)
    qsa.sparse_attn(to_dev(q), to_dev(K), to_dev(V), to_dev(np.array(lens, np.int32)), max_cells,
                    out, H_kv, d, d, scale, pos=to_dev(pos), lse=lse, workspace=ws)
    g_out, g_lse = to_host(out), to_host(lse)
    for i, L in enumerate(lens):
        cells = pos[i, :L]
        cells = cells[(cells >= 0) & (cells < n_kv)]
        if len(cells) == 0:
            assert np.all(g_out[i] == 0.0) and np.all(np.isneginf(g_lse[i]))
            continue
        want, want_lse = oracle.attention(q[i], K, V, H_q, H_kv, d, d, ld, ld, cells, scale)
        np.testing.assert_allclose(g_out[i], want, rtol=0, atol=ATOL_ATTN_BF16)
        np.testing.assert_allclose(g_lse[i], want_lse, rtol=1e-5, atol=1e-4)
