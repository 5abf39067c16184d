"""Full-size GPU parity in the launch configuration bench.py times (one decode step through
qsa_decode_step at the pages' context lengths; the 1024-query prefill chunk at 255,181
tokens), against the fp64 oracle on sampled outputs or in full where the oracle is fast
enough, and against properties that hold at any size.  Inputs come from qsa_synth only."""
import math

import numpy as np
import pytest
import torch

import gather_qsa_pool_gb300 as qsa
import qsa_synth
from oracle import oracle
from gpu_helpers import (ATOL_ATTN_BF16, check_bf16_rows, check_topk, flip_band, pooled_f64,
                         score_tolerance, to_dev, to_host)

pytestmark = pytest.mark.gpu


def _layer(shape, steps):
    return qsa.DecodeLayer(cap_tokens=shape.n_ctx + steps, H_idx=shape.H_idx, d_idx=shape.d_idx,
                           H_q=shape.H_q, H_kv=shape.H_kv, d=shape.d,
                           top_k_tokens=shape.top_k_tokens, eps=shape.eps,
                           rope_base=shape.rope_base)


def test_decode_61789_tokens_three_queries_bf16_pooled_full_oracle():
    """A step carrying three query tokens (a token and two drafts) over a bf16 pooled cache
    at 61,789 tokens, in the benchmark's launch configuration, against the oracle's
    multi-query step: every stored pooled value (bf16 rule), every score of every query, each
    query's selection (band widened by possible bf16 roundings), cell list and output."""
    shape = qsa_synth.CONFIGS["decode_64k"]
    n_q = 3
    inp = qsa_synth.decode_inputs(shape, seed=62, extra_tokens=n_q, n_steps=n_q)
    H, d = shape.H_idx, shape.d_idx
    raw, w, K, V = (to_dev(inp["raw_k"]), to_dev(inp["norm_w"]), to_dev(inp["K"]),
                    to_dev(inp["V"]))
    lay = qsa.DecodeLayer(cap_tokens=shape.n_ctx + n_q, H_idx=H, d_idx=d, H_q=shape.H_q,
                          H_kv=shape.H_kv, d=shape.d, top_k_tokens=shape.top_k_tokens,
                          eps=shape.eps, rope_base=shape.rope_base,
                          pooled_dtype=torch.bfloat16, max_queries=n_q)
    n0 = shape.n_ctx
    lay.rebuild(raw, w, n0)
    o_pooled = np.zeros((lay.cap_rows, H * d), np.uint16)
    oracle.pool_rows(inp["raw_k"], n0, H, d, inp["norm_w"], shape.eps, shape.rope_base, 0,
                     (n0 + 3) // 4, o_pooled)
    n_ctx = n0 + n_q
    out = to_host(lay.step(raw, w, K, V, n_ctx, to_dev(inp["q_idx"]), to_dev(inp["q"])))
    res, o_scores = oracle.decode_step_multi(
        inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps, shape.rope_base, o_pooled,
        n0 // 4, inp["q_idx"], shape.top_k_tokens, inp["q"], inp["K"], inp["V"], shape.H_q,
        shape.H_kv, shape.d)
    n_rows = (n_ctx + 3) // 4
    z = pooled_f64(inp, shape, n_ctx, range(n_rows))
    flips = check_bf16_rows(to_host(lay.pooled)[:n_rows], o_pooled[:n_rows], z, d)
    assert flips <= 1e-3 * n_rows * H * d
    g_scores = to_host(lay.scores_of(n_q, n_ctx))
    scale = 1.0 / math.sqrt(d)
    g_pooled_vals = qsa_synth.bf16_bits_to_f32(to_host(lay.pooled)[:n_rows])
    blocks, counts = to_host(lay.blocks), to_host(lay.counts)
    pos, n_cells = to_host(lay.pos), to_host(lay.n_cells)
    for i in range(n_q):
        # the GPU's scores of its own cache: the fp32 summation rule
        ref = g_pooled_vals.astype(np.float64) @ inp["q_idx"][i].astype(np.float64) * scale
        tol = score_tolerance(inp["q_idx"][i], g_pooled_vals, n_rows, scale)
        assert np.all(np.abs(g_scores[i] - ref) <= tol)
        p = n_ctx - n_q + i
        n_i = min(n_ctx // 4, (p + 1) // 4)
        check_topk(blocks[i], int(counts[i]), o_scores[i], n_i, shape.k_blk,
                   band_abs=flip_band(inp["q_idx"][i], z[:n_i], d, scale))
        o_blocks, o_cells, o_out, _ = res[i]
        if np.array_equal(blocks[i, :counts[i]], o_blocks):
            np.testing.assert_array_equal(pos[i, :n_cells[i]], o_cells)
            np.testing.assert_allclose(out[i], o_out, rtol=0, atol=ATOL_ATTN_BF16)


def test_decode_61789_tokens_full_oracle():
    """Every pooled row, every score, the selection and the attention output of two
    appending decode steps at 61,789 tokens against the oracle."""
    shape = qsa_synth.CONFIGS["decode_64k"]
    steps = 2
    inp = qsa_synth.decode_inputs(shape, seed=61, extra_tokens=steps, n_steps=steps)
    H, d = shape.H_idx, shape.d_idx
    raw, w, K, V = (to_dev(inp["raw_k"]), to_dev(inp["norm_w"]), to_dev(inp["K"]),
                    to_dev(inp["V"]))
    lay = _layer(shape, steps)
    n0 = shape.n_ctx - 1
    lay.rebuild(raw, w, n0)
    o_pooled = np.zeros((lay.cap_rows, H * d), np.float32)
    oracle.pool_rows(inp["raw_k"], n0, H, d, inp["norm_w"], shape.eps, shape.rope_base, 0,
                     (n0 + 3) // 4, o_pooled)
    o_valid = n0 // 4
    for s in range(steps):
        n_ctx = n0 + 1 + s
        out = lay.step(raw, w, K, V, n_ctx, to_dev(inp["q_idx"][s]), to_dev(inp["q"][s]))
        blocks, cells, o_out, _, o_scores = oracle.decode_step(
            inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps, shape.rope_base, o_pooled,
            o_valid, inp["q_idx"][s], shape.top_k_tokens, inp["q"][s], inp["K"], inp["V"],
            shape.H_q, shape.H_kv, shape.d)
        o_valid = n_ctx // 4
        n_rows = (n_ctx + 3) // 4
        g_pooled = to_host(lay.pooled)[:n_rows]
        np.testing.assert_allclose(g_pooled, o_pooled[:n_rows], rtol=2e-5,
                                   atol=2e-6 * float(np.abs(o_pooled[:n_rows]).max()))
        g_scores = to_host(lay.scores)[:n_rows]
        tol = score_tolerance(inp["q_idx"][s], o_pooled, n_rows, 1.0 / math.sqrt(d))
        assert np.all(np.abs(g_scores - o_scores) <= tol)
        g_count = int(to_host(lay.counts)[0])
        g_blocks = to_host(lay.blocks)[0]
        n_band = check_topk(g_blocks, g_count, o_scores, n_ctx // 4, shape.k_blk)
        if np.array_equal(g_blocks[:g_count], blocks):
            nc = int(to_host(lay.n_cells)[0])
            np.testing.assert_array_equal(to_host(lay.pos)[0, :nc], cells)
            np.testing.assert_allclose(to_host(out)[0], o_out, rtol=0, atol=ATOL_ATTN_BF16)
        else:
            assert n_band > 0


def test_decode_clear_winners_61789_full_oracle():
    """Scores with clear winners (the benchmark's clear-winners workload: 1% of the completed
    pooled rows leaning toward the queries' common direction, about three standard
    deviations up), over two appending steps at 61,789 tokens: the step takes the leaned
    cache as given (the same rows on both sides), and every score, the histogram-fed
    selection on these peaked rows (against the oracle's scores, tie band), the cell list
    and the attention output are compared with the oracle; most leaning rows must be
    selected (with scores of no preference a row is selected with probability k / n, 3%
    here), or the workload would not be peaked."""
    shape = qsa_synth.CONFIGS["decode_64k"]
    steps = 2
    inp = qsa_synth.decode_inputs(shape, seed=64, extra_tokens=steps, n_steps=steps)
    H, d = shape.H_idx, shape.d_idx
    raw, w, K, V = (to_dev(inp["raw_k"]), to_dev(inp["norm_w"]), to_dev(inp["K"]),
                    to_dev(inp["V"]))
    n0 = shape.n_ctx - 1
    o_valid = n0 // 4
    cw = qsa_synth.clear_winners_torch(o_valid, H * d, steps, seed=65, device="cpu")
    q_idx = cw["q_idx"].numpy()
    lean_rows = cw["rows"].numpy()
    lay = _layer(shape, steps)
    lay.rebuild(raw, w, n0)
    o_pooled = np.zeros((lay.cap_rows, H * d), np.float32)
    oracle.pool_rows(inp["raw_k"], n0, H, d, inp["norm_w"], shape.eps, shape.rope_base, 0,
                     (n0 + 3) // 4, o_pooled)
    o_pooled[lean_rows] += cw["add"].numpy()
    lay.pooled[:o_valid].copy_(torch.from_numpy(o_pooled[:o_valid]))
    for s in range(steps):
        n_ctx = n0 + 1 + s
        out = lay.step(raw, w, K, V, n_ctx, to_dev(q_idx[s]), to_dev(inp["q"][s]))
        blocks, cells, o_out, _, o_scores = oracle.decode_step(
            inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps, shape.rope_base, o_pooled,
            o_valid, q_idx[s], shape.top_k_tokens, inp["q"][s], inp["K"], inp["V"],
            shape.H_q, shape.H_kv, shape.d)
        o_valid = n_ctx // 4
        n_rows = (n_ctx + 3) // 4
        g_scores = to_host(lay.scores)[:n_rows]
        tol = score_tolerance(q_idx[s], o_pooled, n_rows, 1.0 / math.sqrt(d))
        assert np.all(np.abs(g_scores - o_scores) <= tol)
        g_count = int(to_host(lay.counts)[0])
        g_blocks = to_host(lay.blocks)[0]
        n_band = check_topk(g_blocks, g_count, o_scores, n_ctx // 4, shape.k_blk)
        assert np.isin(lean_rows, g_blocks[:g_count]).mean() > 0.6
        if np.array_equal(g_blocks[:g_count], blocks):
            nc = int(to_host(lay.n_cells)[0])
            np.testing.assert_array_equal(to_host(lay.pos)[0, :nc], cells)
            np.testing.assert_allclose(to_host(out)[0], o_out, rtol=0, atol=ATOL_ATTN_BF16)
        else:
            assert n_band > 0


@pytest.mark.parametrize("name", ["decode_128k", "decode_256k"])
def test_decode_appending_256_steps_full_oracle(name):
    """The decode sweep at 126,253 and 255,181 tokens: 256 consecutive steps, each appending
    one token (new raw indexer key, K and V rows) so that every step recomputes the open
    block and every fourth step completes one, in the benchmark's launch configuration.
    Step 0 runs at exactly the named context; there every pooled row is compared with the
    oracle's.  At every step: the rows the step recomputed, every score (fp32 summation
    bound), the selection against the oracle's own scores (tie band), the cell list and
    the attention output whenever the selected sets agree.  After the last step the whole
    incrementally maintained cache is compared with the oracle's cache rebuilt from scratch,
    and is bit-identical to the library's own full rebuild."""
    shape = qsa_synth.CONFIGS[name]
    steps = 256
    inp = qsa_synth.decode_inputs(shape, seed=shape.n_ctx, extra_tokens=steps, n_steps=steps)
    H, d = shape.H_idx, shape.d_idx
    scale = 1.0 / math.sqrt(d)
    raw, w, K, V = (to_dev(inp["raw_k"]), to_dev(inp["norm_w"]), to_dev(inp["K"]),
                    to_dev(inp["V"]))
    q_idx, q = to_dev(inp["q_idx"]), to_dev(inp["q"])
    lay = _layer(shape, steps)
    n0 = shape.n_ctx - 1
    lay.rebuild(raw, w, n0)
    o_pooled = np.zeros((lay.cap_rows, H * d), np.float32)
    oracle.pool_rows(inp["raw_k"], n0, H, d, inp["norm_w"], shape.eps, shape.rope_base, 0,
                     (n0 + 3) // 4, o_pooled)
    o_valid = n0 // 4
    agree = 0
    for s in range(steps):
        n_ctx = n0 + 1 + s
        n_rows = (n_ctx + 3) // 4
        lay.step(raw, w, K, V, n_ctx, q_idx[s], q[s])
        blocks, cells, o_out, _, o_scores = oracle.decode_step(
            inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps, shape.rope_base, o_pooled,
            o_valid, inp["q_idx"][s], shape.top_k_tokens, inp["q"][s], inp["K"], inp["V"],
            shape.H_q, shape.H_kv, shape.d)
        r0 = 0 if s == 0 else o_valid
        o_valid = n_ctx // 4
        g_rows = to_host(lay.pooled[r0:n_rows])
        np.testing.assert_allclose(g_rows, o_pooled[r0:n_rows], rtol=2e-5,
                                   atol=2e-6 * float(np.abs(o_pooled[r0:n_rows]).max()))
        g_scores = to_host(lay.scores)[:n_rows]
        tol = score_tolerance(inp["q_idx"][s], o_pooled, n_rows, scale)
        assert np.all(np.abs(g_scores - o_scores) <= tol), f"step {s}"
        g_count = int(to_host(lay.counts)[0])
        g_blocks = to_host(lay.blocks)[0]
        n_band = check_topk(g_blocks, g_count, o_scores, n_ctx // 4, shape.k_blk)
        if np.array_equal(g_blocks[:g_count], blocks):
            nc = int(to_host(lay.n_cells)[0])
            assert nc == 4 * shape.k_blk + n_ctx % 4
            np.testing.assert_array_equal(to_host(lay.pos)[0, :nc], cells)
            np.testing.assert_allclose(to_host(lay.out)[0], o_out, rtol=0, atol=ATOL_ATTN_BF16)
            agree += 1
        else:
            assert n_band > 0
    assert agree >= steps - 2
    # the incremental cache after 256 appends against rebuilds from scratch
    n_ctx = n0 + steps
    n_rows = (n_ctx + 3) // 4
    fresh = oracle.pool_rows(inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps,
                             shape.rope_base, 0, n_rows)
    np.testing.assert_array_equal(o_pooled[:n_rows], fresh)
    g_pooled = to_host(lay.pooled)[:n_rows]
    np.testing.assert_allclose(g_pooled, fresh, rtol=2e-5,
                               atol=2e-6 * float(np.abs(fresh).max()))
    again = _layer(shape, steps)
    again.rebuild(raw, w, n_ctx)
    np.testing.assert_array_equal(to_host(again.pooled)[:n_rows], g_pooled)


def test_topk_at_maximum_candidates():
    n_full = qsa.topk_max_candidates()
    k_blk = 512
    rng = np.random.default_rng(640)
    s = rng.standard_normal(n_full).astype(np.float32)
    s[rng.choice(n_full, 5000, replace=False)] = s[rng.choice(n_full, 5000)]
    blocks = torch.zeros((1, k_blk), dtype=torch.int32, device="cuda")
    counts = torch.zeros(1, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(to_dev(s[None]), n_full, k_blk, blocks, counts)
    want = oracle.topk(s.astype(np.float64), n_full, k_blk)
    np.testing.assert_array_equal(to_host(blocks)[0], want)


def test_prefill_chunk_1024_queries_at_255181_sampled():
    """The 1024-query chunk after 255,181 tokens: tensor-core scores of sampled queries
    against the oracle's bf16-operand scores, their selections under the tie band rule,
    and their attention outputs whenever the selections agree."""
    shape = qsa_synth.CONFIGS["prefill_256k"]
    inp = qsa_synth.prefill_inputs(shape, seed=1024)
    H, d, n_q, n_rows, n_ctx = shape.H_idx, shape.d_idx, shape.n_q, shape.n_rows, shape.n_ctx
    pooled = torch.zeros(n_rows, H * d, device="cuda")
    qsa.pool_update(to_dev(inp["raw_k"]), n_ctx, H, d, to_dev(inp["norm_w"]), shape.eps,
                    shape.rope_base, pooled, 0)
    q_pos = to_dev(inp["q_pos"])
    scale_idx = 1.0 / math.sqrt(d)
    scores = torch.empty(n_q, n_rows, device="cuda")
    ws = torch.zeros(qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC),
                     dtype=torch.uint8, device="cuda")
    qsa.index_score(to_dev(inp["q_idx"]), pooled, n_rows, H, d, scale_idx, scores, q_pos=q_pos,
                    precision=qsa.QSA_PREC_BF16_TC, workspace=ws)
    blocks = torch.empty(n_q, shape.k_blk, dtype=torch.int32, device="cuda")
    counts = torch.empty(n_q, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(scores, n_ctx // 4, shape.k_blk, blocks, counts, q_pos=q_pos)
    pos = torch.empty(n_q, shape.max_cells, dtype=torch.int32, device="cuda")
    n_cells = torch.empty(n_q, dtype=torch.int32, device="cuda")
    qsa.gather_kv(blocks, counts, shape.k_blk, pos, n_cells, shape.max_cells, q_pos=q_pos,
                  n_kv=n_ctx)
    out = torch.empty(n_q, shape.H_q, shape.d, device="cuda")
    aws = torch.empty(max(qsa.sparse_attn_workspace_size(n_q, shape.H_q, shape.H_kv, shape.d,
                                                          shape.max_cells) // 4, 1),
                      device="cuda")
    qsa.sparse_attn(to_dev(inp["q"]), to_dev(inp["K"]), to_dev(inp["V"]), n_cells,
                    shape.max_cells, out, shape.H_kv, shape.d, shape.d, 1.0 / math.sqrt(shape.d),
                    pos=pos, workspace=aws)
    g_scores, g_blocks, g_counts = to_host(scores), to_host(blocks), to_host(counts)
    g_out, g_pos = to_host(out), to_host(pos)
    # the oracle's own pooled cache and scores for a few queries (first, last, random)
    o_pooled = oracle.pool_rows(inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps,
                                shape.rope_base, 0, n_rows)
    sample = np.array([0, 1, 511, 1022, 1023] + list(np.random.default_rng(5).choice(1024, 3)))
    o_scores = oracle.scores(inp["q_idx"][sample], o_pooled, n_rows, H, d, scale_idx,
                             q_pos=inp["q_pos"][sample], round_bf16_operands=True)
    agree = 0
    for j, i in enumerate(sample):
        p = int(inp["q_pos"][i])
        nf = (p + 1) // 4
        vis = np.isfinite(o_scores[j])
        assert np.array_equal(np.isneginf(g_scores[i]), ~vis)
        n_band = check_topk(g_blocks[i], int(g_counts[i]), o_scores[j], nf, shape.k_blk)
        w_blocks = oracle.topk(o_scores[j], nf, shape.k_blk)
        if np.array_equal(g_blocks[i, :g_counts[i]], w_blocks):
            cells = oracle.cells(w_blocks, p)
            np.testing.assert_array_equal(g_pos[i, :cells.shape[0]], cells)
            want, _ = oracle.attention(inp["q"][i], inp["K"], inp["V"], shape.H_q, shape.H_kv,
                                       shape.d, shape.d, shape.H_kv * shape.d,
                                       shape.H_kv * shape.d, cells, 1.0 / math.sqrt(shape.d))
            np.testing.assert_allclose(g_out[i], want, rtol=0, atol=ATOL_ATTN_BF16)
            agree += 1
        else:
            assert n_band > 0
    assert agree >= len(sample) - 1


def test_prefill_selection_with_maxima_at_255181():
    """The 1024-query chunk after 255,181 tokens in the benchmark's launch configuration: the
    score kernel that also writes group maxima gives the same scores bit for bit, and the
    top-k fed by those maxima the same selection, for every query, as the top-k that scans
    whole rows (itself exact against the oracle in the tests above and below)."""
    shape = qsa_synth.CONFIGS["prefill_256k"]
    inp = qsa_synth.prefill_inputs(shape, seed=1025)
    H, d, n_q, n_rows, n_ctx = shape.H_idx, shape.d_idx, shape.n_q, shape.n_rows, shape.n_ctx
    pooled = torch.zeros(n_rows, H * d, device="cuda")
    qsa.pool_update(to_dev(inp["raw_k"]), n_ctx, H, d, to_dev(inp["norm_w"]), shape.eps,
                    shape.rope_base, pooled, 0)
    q_pos, q = to_dev(inp["q_pos"]), to_dev(inp["q_idx"])
    scale_idx = 1.0 / math.sqrt(d)
    ws = torch.zeros(qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC),
                     dtype=torch.uint8, device="cuda")
    ref = torch.empty(n_q, n_rows, device="cuda")
    qsa.index_score(q, pooled, n_rows, H, d, scale_idx, ref, q_pos=q_pos,
                    precision=qsa.QSA_PREC_BF16_TC, workspace=ws)
    scores = torch.empty(n_q, n_rows, device="cuda")
    maxima = torch.empty(n_q, (n_rows + 31) // 32, device="cuda")
    qsa.index_score_maxima(q, pooled, n_rows, H, d, scale_idx, scores, maxima, q_pos=q_pos,
                           workspace=ws)
    assert torch.equal(scores, ref)
    padded = torch.full((n_q, maxima.shape[1] * 32), -math.inf, device="cuda")
    padded[:, :n_rows] = ref
    assert torch.equal(maxima, padded.view(n_q, -1, 32).amax(dim=2))
    blocks = torch.empty(n_q, shape.k_blk, dtype=torch.int32, device="cuda")
    counts = torch.empty(n_q, dtype=torch.int32, device="cuda")
    tws = torch.empty(qsa.topk_blocks_maxima_workspace_size(n_q), dtype=torch.uint8,
                      device="cuda")
    qsa.topk_blocks_maxima(scores, maxima, n_ctx // 4, shape.k_blk, blocks, counts, tws,
                           q_pos=q_pos)
    w_blocks = torch.empty_like(blocks)
    w_counts = torch.empty_like(counts)
    qsa.topk_blocks(ref, n_ctx // 4, shape.k_blk, w_blocks, w_counts, q_pos=q_pos)
    assert torch.equal(counts, w_counts)
    assert torch.equal(blocks, w_blocks)


@pytest.mark.parametrize("store,n_q,steps", [("bf16", 1, 16), ("f32", 3, 6), ("bf16", 3, 6)],
                         ids=["bf16-pooled", "three-queries", "three-queries-bf16-pooled"])
def test_decode_255181_tokens_variants_appending(store, n_q, steps):
    """The benchmarked variants at 255,181 tokens in their launch configuration: a bf16
    pooled cache (half the scan's bytes) and steps carrying three query tokens (a token and
    two drafts), appending n_q tokens per step, against the oracle's multi-query step at
    every step: the recomputed rows (bf16 rows: each stored value a rounding of a value
    within the kernel's fp32 error of the exact one), 2,000 sampled rows at the first step,
    every score of every query, each query's selection (the tie band widened, for bf16 rows,
    by what a rounding the other way can move a score), cell list and output."""
    shape = qsa_synth.CONFIGS["decode_256k"]
    inp = qsa_synth.decode_inputs(shape, seed=2551 + n_q, extra_tokens=n_q * steps,
                                  n_steps=n_q * steps)
    H, d = shape.H_idx, shape.d_idx
    scale = 1.0 / math.sqrt(d)
    raw, w, K, V = (to_dev(inp["raw_k"]), to_dev(inp["norm_w"]), to_dev(inp["K"]),
                    to_dev(inp["V"]))
    bf = store == "bf16"
    lay = qsa.DecodeLayer(cap_tokens=shape.n_ctx + n_q * steps, H_idx=H, d_idx=d,
                          H_q=shape.H_q, H_kv=shape.H_kv, d=shape.d,
                          top_k_tokens=shape.top_k_tokens, eps=shape.eps,
                          rope_base=shape.rope_base,
                          pooled_dtype=torch.bfloat16 if bf else None, max_queries=n_q)
    n0 = shape.n_ctx - n_q
    lay.rebuild(raw, w, n0)
    o_pooled = np.zeros((lay.cap_rows, H * d), np.uint16 if bf else np.float32)
    oracle.pool_rows(inp["raw_k"], n0, H, d, inp["norm_w"], shape.eps, shape.rope_base, 0,
                     (n0 + 3) // 4, o_pooled)
    o_valid = n0 // 4
    q_idx_all = inp["q_idx"].reshape(steps, n_q, -1)
    q_all = inp["q"].reshape(steps, n_q, shape.H_q, shape.d)
    rng = np.random.default_rng(2551)
    agree = 0
    for s in range(steps):
        n_ctx = n0 + n_q * (s + 1)
        n_rows = (n_ctx + 3) // 4
        lay.step(raw, w, K, V, n_ctx, to_dev(q_idx_all[s]), to_dev(q_all[s]))
        res, o_scores = oracle.decode_step_multi(
            inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps, shape.rope_base, o_pooled,
            o_valid, q_idx_all[s], shape.top_k_tokens, q_all[s], inp["K"], inp["V"], shape.H_q,
            shape.H_kv, shape.d)
        rows = np.arange(o_valid, n_rows)
        if s == 0:
            rows = np.concatenate([rng.choice(o_valid, 2000, replace=False), rows])
        o_valid = n_ctx // 4
        g_all = to_host(lay.pooled)
        if bf:
            z = pooled_f64(inp, shape, n_ctx, rows)
            check_bf16_rows(g_all[rows], o_pooled[rows], z, d)
            g_vals = qsa_synth.bf16_bits_to_f32(g_all[:n_rows])
        else:
            np.testing.assert_allclose(g_all[rows], o_pooled[rows], rtol=2e-5,
                                       atol=2e-6 * float(np.abs(o_pooled[rows]).max()))
            g_vals = g_all[:n_rows]
        g_scores = to_host(lay.scores_of(n_q, n_ctx))
        blocks, counts = to_host(lay.blocks), to_host(lay.counts)
        pos, n_cells, out = to_host(lay.pos), to_host(lay.n_cells), to_host(lay.out)
        # the GPU's scores of its own cache against the fp32 summation bound (the bound of
        # score_tolerance, for all queries at once)
        g64 = g_vals.astype(np.float64)
        qs = q_idx_all[s].astype(np.float64).T
        ref_all = (g64 @ qs).T * scale
        chain = H * d / 128 + 8
        tol_all = (2.0 * chain * 2.0 ** -24 * scale * (np.abs(g64) @ np.abs(qs))).T + 1e-30
        del g64
        for i in range(n_q):
            assert np.all(np.abs(g_scores[i] - ref_all[i]) <= tol_all[i]), f"step {s} query {i}"
            p = n_ctx - n_q + i
            n_i = min(n_ctx // 4, (p + 1) // 4)
            band = None
            if bf:
                # what a bf16 rounding the other way can move a score, for the rows near the
                # k-th best oracle score (elsewhere it cannot change the selection)
                srt = np.sort(np.nan_to_num(o_scores[i][:n_i], nan=-np.inf))[::-1]
                s_k = srt[shape.k_blk - 1]
                near = np.flatnonzero(np.abs(o_scores[i][:n_i] - s_k) <= 1e-2 * abs(s_k))
                band = np.zeros(n_i)
                band[near] = flip_band(q_idx_all[s][i], pooled_f64(inp, shape, n_ctx, near), d,
                                       scale)
            n_band = check_topk(blocks[i], int(counts[i]), o_scores[i], n_i, shape.k_blk,
                                band_abs=band)
            o_blocks, o_cells, o_out, _ = res[i]
            if np.array_equal(blocks[i, :counts[i]], o_blocks):
                np.testing.assert_array_equal(pos[i, :n_cells[i]], o_cells)
                np.testing.assert_allclose(out[i], o_out, rtol=0, atol=ATOL_ATTN_BF16)
                agree += 1
            else:
                assert n_band > 0
    assert agree >= n_q * steps - 2
