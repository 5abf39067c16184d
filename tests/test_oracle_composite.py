"""Pins of the oracle's composite decode steps (``oracle.decode_step`` and
``oracle.decode_step_multi``), which every end-to-end GPU comparison and the smoke check
rely on.  Each composite chains the pinned pieces (pool -> score -> top-k -> cells ->
attention) and chooses the two scales, the query positions, each query's candidate count
and the validity watermark; these tests check those choices against definitions written
out independently of the oracle:

  - scores: the pooled rows times the query, with the indexer scale 1/sqrt(64) = 1/8 of the
    tiny configuration's stated score formula (sum_h q_h . k_h / sqrt(64)), by numpy;
  - selection: a numpy lexsort of those scores (descending, lower block first on ties);
  - attention: torch's scaled_dot_product_attention in fp64 (its default scale is
    1/sqrt(head dim)) over all positions, over the causal prefix of each query, or with a
    boolean mask admitting only the selected cells; the log-sum-exp by torch.logsumexp.
When every block is selected (top-k at least the context), QSA is dense causal attention
(Qiita, ariera, llama.cpp series part 10, "QSA and the QSA indexer": the indexer only
narrows the cells attention runs over).
"""
import math

import numpy as np
import pytest
import torch

import qsa_synth
from oracle import oracle

TINY = qsa_synth.CONFIGS["tiny_f32_decode"]
SCALE_IDX_TINY = 1.0 / 8.0  # the tiny configuration's score formula divides by sqrt(64)


def _f64(a):
    """Stored values (fp32, or bf16 bit patterns) as fp64 torch tensors."""
    if a.dtype == np.uint16:
        a = qsa_synth.bf16_bits_to_f32(a)
    return torch.from_numpy(np.asarray(a, np.float64))


def _sdpa(q, K, V, n_tok, H_q, H_kv, d, visible):
    """fp64 SDPA of one query token q [H_q][d] over K/V rows [0, n_tok) with the boolean
    visibility vector ``visible`` [n_tok]; KV head h // (H_q / H_kv) serves query head h.
    Returns (out [H_q][d], lse [H_q])."""
    G = H_q // H_kv
    k = _f64(K[:n_tok]).reshape(n_tok, H_kv, d).permute(1, 0, 2).repeat_interleave(G, dim=0)
    v = _f64(V[:n_tok]).reshape(n_tok, H_kv, d).permute(1, 0, 2).repeat_interleave(G, dim=0)
    qq = torch.from_numpy(np.asarray(q, np.float64)).reshape(H_q, 1, d)
    m = torch.from_numpy(np.asarray(visible, bool)).reshape(1, 1, n_tok).expand(H_q, 1, n_tok)
    out = torch.nn.functional.scaled_dot_product_attention(qq, k, v, attn_mask=m)
    logits = (qq @ k.transpose(1, 2))[:, 0, :] / math.sqrt(d)
    lse = torch.logsumexp(logits.masked_fill(~m[:, 0, :], -math.inf), dim=-1)
    return out[:, 0, :].numpy(), lse.numpy()


def _np_topk(s, n_cand, k):
    order = np.lexsort((np.arange(n_cand), -s[:n_cand]))
    return np.sort(order[:min(k, n_cand)]).astype(np.int64)


def _fresh_pool(inp, shape, n_ctx, store=np.float32):
    return oracle.pool_rows(inp["raw_k"], n_ctx, shape.H_idx, shape.d_idx, inp["norm_w"],
                            shape.eps, shape.rope_base, 0, (n_ctx + 3) // 4,
                            np.zeros(((n_ctx + 3) // 4, shape.H_idx * shape.d_idx), store))


def test_decode_step_is_dense_attention_when_every_block_is_selected():
    inp = qsa_synth.decode_inputs(TINY, seed=0)
    n_ctx = TINY.n_ctx
    n_full = n_ctx // 4
    pooled = np.zeros(((n_ctx + 3) // 4, TINY.H_idx * TINY.d_idx), np.float32)
    blocks, cells, out, lse, s = oracle.decode_step(
        inp["raw_k"], n_ctx, TINY.H_idx, TINY.d_idx, inp["norm_w"], TINY.eps, TINY.rope_base,
        pooled, 0, inp["q_idx"][0], 4 * (n_full + 3), inp["q"][0], inp["K"], inp["V"],
        TINY.H_q, TINY.H_kv, TINY.d)
    np.testing.assert_array_equal(blocks, np.arange(n_full))
    np.testing.assert_array_equal(cells, np.arange(n_ctx))
    want, want_lse = _sdpa(inp["q"][0], inp["K"], inp["V"], n_ctx, TINY.H_q, TINY.H_kv, TINY.d,
                           np.ones(n_ctx, bool))
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-12)
    # the scores of every row, the open one included, with the stated scale
    ref = _fresh_pool(inp, TINY, n_ctx).astype(np.float64) @ inp["q_idx"][0].astype(np.float64)
    np.testing.assert_allclose(s, SCALE_IDX_TINY * ref, rtol=1e-12, atol=1e-12)
    assert s.shape == ((n_ctx + 3) // 4,)


def test_decode_step_attends_over_exactly_the_selected_cells():
    """The tiny configuration as stated: top-k 64 tokens (16 blocks) plus the open tail."""
    inp = qsa_synth.decode_inputs(TINY, seed=3)
    n_ctx = TINY.n_ctx
    n_full = n_ctx // 4
    pooled = np.zeros(((n_ctx + 3) // 4, TINY.H_idx * TINY.d_idx), np.float32)
    blocks, cells, out, lse, s = oracle.decode_step(
        inp["raw_k"], n_ctx, TINY.H_idx, TINY.d_idx, inp["norm_w"], TINY.eps, TINY.rope_base,
        pooled, 0, inp["q_idx"][0], TINY.top_k_tokens, inp["q"][0], inp["K"], inp["V"],
        TINY.H_q, TINY.H_kv, TINY.d)
    ref = SCALE_IDX_TINY * (_fresh_pool(inp, TINY, n_ctx).astype(np.float64)
                            @ inp["q_idx"][0].astype(np.float64))
    np.testing.assert_allclose(s, ref, rtol=1e-12, atol=1e-12)
    want_blocks = _np_topk(ref, n_full, TINY.top_k_tokens // 4)
    np.testing.assert_array_equal(blocks, want_blocks)
    want_cells = np.concatenate([(4 * want_blocks[:, None] + np.arange(4)).reshape(-1),
                                 np.arange(4 * n_full, n_ctx)])
    np.testing.assert_array_equal(cells, want_cells)
    assert cells.shape[0] == TINY.top_k_tokens + n_ctx % 4
    vis = np.zeros(n_ctx, bool)
    vis[want_cells] = True
    want, want_lse = _sdpa(inp["q"][0], inp["K"], inp["V"], n_ctx, TINY.H_q, TINY.H_kv, TINY.d,
                           vis)
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-12)


def test_decode_step_bf16_shapes_dense_and_incremental():
    """The bf16 decode shapes (indexer 16 x 128, attention 32 / 4 heads x 128) on a short
    context where top-k 2048 tokens covers every block: two appending steps, the second
    updating the cache incrementally from the first's watermark, against dense SDPA and
    against a cache pooled from scratch."""
    shape = qsa_synth.shrink(qsa_synth.CONFIGS["decode_64k"], n_ctx=1001)
    inp = qsa_synth.decode_inputs(shape, seed=5, extra_tokens=2, n_steps=2)
    H, d = shape.H_idx, shape.d_idx
    pooled = np.zeros(((shape.n_ctx + 2 + 3) // 4, H * d), np.float32)
    valid = 0
    for step in range(2):
        n_ctx = shape.n_ctx + 1 + step
        _, cells, out, lse, s = oracle.decode_step(
            inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps, shape.rope_base, pooled, valid,
            inp["q_idx"][step], shape.top_k_tokens, inp["q"][step], inp["K"], inp["V"],
            shape.H_q, shape.H_kv, shape.d)
        valid = n_ctx // 4
        n_rows = (n_ctx + 3) // 4
        fresh = _fresh_pool(inp, shape, n_ctx)
        np.testing.assert_array_equal(pooled[:n_rows], fresh)
        ref = fresh.astype(np.float64) @ inp["q_idx"][step].astype(np.float64) / math.sqrt(128)
        np.testing.assert_allclose(s, ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(cells, np.arange(n_ctx))
        want, want_lse = _sdpa(inp["q"][step], inp["K"], inp["V"], n_ctx, shape.H_q,
                               shape.H_kv, shape.d, np.ones(n_ctx, bool))
        np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("n_q", [2, 3, 4])
def test_decode_step_multi_is_causal_dense_when_every_block_is_selected(n_q):
    """Query i of the last n_q tokens sits at n_ctx - n_q + i and sees positions up to its
    own: with every block selected that is textbook causal attention."""
    inp = qsa_synth.decode_inputs(TINY, seed=40 + n_q, extra_tokens=n_q, n_steps=n_q)
    n_ctx = TINY.n_ctx + n_q - 1
    pooled = np.zeros(((n_ctx + 3) // 4, TINY.H_idx * TINY.d_idx), np.float32)
    res, s = oracle.decode_step_multi(
        inp["raw_k"], n_ctx, TINY.H_idx, TINY.d_idx, inp["norm_w"], TINY.eps, TINY.rope_base,
        pooled, 0, inp["q_idx"], 4 * (n_ctx // 4 + 3), inp["q"], inp["K"], inp["V"], TINY.H_q,
        TINY.H_kv, TINY.d)
    ref = SCALE_IDX_TINY * (_fresh_pool(inp, TINY, n_ctx).astype(np.float64)
                            @ inp["q_idx"].astype(np.float64).T).T
    np.testing.assert_allclose(s, ref, rtol=1e-12, atol=1e-12)
    for i in range(n_q):
        p = n_ctx - n_q + i
        blocks, cells, out, lse = res[i]
        np.testing.assert_array_equal(blocks, np.arange((p + 1) // 4))
        np.testing.assert_array_equal(cells, np.arange(p + 1))
        vis = np.arange(n_ctx) <= p
        want, want_lse = _sdpa(inp["q"][i], inp["K"], inp["V"], n_ctx, TINY.H_q, TINY.H_kv,
                               TINY.d, vis)
        np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-12)


def test_decode_step_multi_selects_among_blocks_complete_at_each_position():
    """Three queries with top-k 64 tokens on a context ending mid-block: each query's
    candidates stop at its own position, its tail ends at its own position, and it attends
    over exactly its cells."""
    n_q = 3
    inp = qsa_synth.decode_inputs(TINY, seed=77, extra_tokens=n_q, n_steps=n_q)
    n_ctx = 2053  # queries at 2050, 2051 (completes block 512) and 2052
    pooled = np.zeros(((n_ctx + 3) // 4, TINY.H_idx * TINY.d_idx), np.float32)
    res, s = oracle.decode_step_multi(
        inp["raw_k"], n_ctx, TINY.H_idx, TINY.d_idx, inp["norm_w"], TINY.eps, TINY.rope_base,
        pooled, 0, inp["q_idx"], TINY.top_k_tokens, inp["q"], inp["K"], inp["V"], TINY.H_q,
        TINY.H_kv, TINY.d)
    ref = SCALE_IDX_TINY * (_fresh_pool(inp, TINY, n_ctx).astype(np.float64)
                            @ inp["q_idx"].astype(np.float64).T).T
    np.testing.assert_allclose(s, ref, rtol=1e-12, atol=1e-12)
    k_blk = TINY.top_k_tokens // 4
    for i in range(n_q):
        p = n_ctx - n_q + i
        n_cand = (p + 1) // 4
        blocks, cells, out, lse = res[i]
        want_blocks = _np_topk(ref[i], n_cand, k_blk)
        np.testing.assert_array_equal(blocks, want_blocks)
        want_cells = np.concatenate([(4 * want_blocks[:, None] + np.arange(4)).reshape(-1),
                                     np.arange(4 * n_cand, p + 1)])
        np.testing.assert_array_equal(cells, want_cells)
        vis = np.zeros(n_ctx, bool)
        vis[want_cells] = True
        want, want_lse = _sdpa(inp["q"][i], inp["K"], inp["V"], n_ctx, TINY.H_q, TINY.H_kv,
                               TINY.d, vis)
        np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-12)
    # position 2051 completes block 512: the second query may select it, the first may not
    assert (n_ctx - n_q + 1 + 1) // 4 == 513 and (n_ctx - n_q + 1) // 4 == 512
