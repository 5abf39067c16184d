"""GPU parity of the bf16 pooled-key cache and of the multi-query decode step (a token and
its draft tokens verified together) against the fp64 oracle on the same seeded inputs.
Every input and every expected value comes from qsa_synth or the oracle.

bf16 storage rule: the oracle rounds the exact (fp64) pooled value to bf16 once; the
kernel rounds its fp32 value, which lies within delta (BF16_FLIP_REL of the rotation
pair's magnitude) of the exact one.  So each stored value must be the bf16 rounding of
some value within delta of the exact value: away from rounding midpoints (and from zero)
that is the oracle's bits exactly, next to one either neighbour.  Scores and selections
over a kernel-written bf16 cache widen the top-k boundary band by what such roundings
can move a score.
"""
import math

import numpy as np
import pytest
import torch

import gather_qsa_pool_gb300 as qsa
import qsa_synth
from oracle import oracle
from gpu_helpers import (ATOL_ATTN_BF16, ATOL_ATTN_F32, check_bf16_rows, check_topk, flip_band,
                         pooled_f64, score_tolerance, to_dev, to_host)

pytestmark = pytest.mark.gpu

TINY = qsa_synth.CONFIGS["tiny_f32_decode"]
SMALL = qsa_synth.shrink(qsa_synth.CONFIGS["decode_64k"], name="small_bf16", n_ctx=9_003,
                         top_k_tokens=512)
# ------------------------------------------------------------------ bf16 pooled storage

@pytest.mark.parametrize("shape", [TINY, SMALL], ids=lambda s: s.name)
def test_pool_update_bf16_storage(shape):
    inp = qsa_synth.decode_inputs(shape, seed=41)
    n_ctx, H, d = shape.n_ctx, shape.H_idx, shape.d_idx
    want = oracle.pool_rows(inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps,
                            shape.rope_base, 0, shape.n_rows, store="bf16")
    pooled = torch.zeros(shape.n_rows + 3, H * d, dtype=torch.bfloat16, device="cuda")
    pooled[shape.n_rows:] = 5.0
    qsa.pool_update(to_dev(inp["raw_k"]), n_ctx, H, d, to_dev(inp["norm_w"]), shape.eps,
                    shape.rope_base, pooled, 0)
    got = to_host(pooled)
    z = pooled_f64(inp, shape, n_ctx, range(shape.n_rows))
    flips = check_bf16_rows(got[:shape.n_rows], want, z, d)
    assert flips <= 1e-3 * want.size  # rounding disagreements are rare
    assert np.all(got[shape.n_rows:] == 0x40A0)  # rows past the cache end untouched


@pytest.mark.parametrize("n_q", [1, 2, 3, 4])
@pytest.mark.parametrize("store", ["f32", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_index_score_few_queries_one_pass(n_q, store, causal):
    """1-4 queries share one pass over the cache (fp32 or bf16 rows); with q_pos the rows a
    query cannot see are -inf."""
    shape = qsa_synth.shrink(SMALL, n_ctx=20_001)
    inp = qsa_synth.decode_inputs(shape, seed=42, n_steps=n_q)
    H, d, n_rows = shape.H_idx, shape.d_idx, shape.n_rows
    pooled = oracle.pool_rows(inp["raw_k"], shape.n_ctx, H, d, inp["norm_w"], shape.eps,
                              shape.rope_base, 0, n_rows, store=store)
    pvals = qsa_synth.bf16_bits_to_f32(pooled) if store == "bf16" else pooled
    scale = 1.0 / math.sqrt(d)
    q_pos = (np.array([5, 4000, 79_000, 80_000])[:n_q] % shape.n_ctx).astype(np.int32) \
        if causal else None
    want = oracle.scores(inp["q_idx"], pooled, n_rows, H, d, scale, q_pos=q_pos)
    scores = torch.full((n_q, n_rows + 2), 3.0, device="cuda")
    qsa.index_score(to_dev(inp["q_idx"]), to_dev(pooled), n_rows, H, d, scale, scores,
                    q_pos=None if q_pos is None else to_dev(q_pos))
    got = to_host(scores)
    assert np.all(got[:, n_rows:] == 3.0)
    for i in range(n_q):
        vis = np.isfinite(want[i])
        assert np.array_equal(np.isneginf(got[i, :n_rows]), ~vis)
        tol = score_tolerance(inp["q_idx"][i], pvals, n_rows, scale)[vis]
        assert np.all(np.abs(got[i, :n_rows][vis] - want[i][vis]) <= tol)


def test_prefill_scores_on_tensor_cores_read_a_bf16_cache_in_place():
    H, d, depth, n_q = 16, 128, 6000, 300
    shape = qsa_synth.PrefillShape("tc_bf16", depth, n_q, H, d, 8, 2, 128, 256, dtype="bf16")
    inp = qsa_synth.prefill_inputs(shape, seed=43)
    n_rows = shape.n_rows
    pooled = oracle.pool_rows(inp["raw_k"], shape.n_ctx, H, d, inp["norm_w"], shape.eps,
                              shape.rope_base, 0, n_rows, store="bf16")
    scale = 1.0 / math.sqrt(d)
    ws_f32 = qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC)
    ws_b = qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC, qsa.QSA_BF16)
    assert ws_b < ws_f32
    ws = torch.zeros(ws_b, dtype=torch.uint8, device="cuda")
    scores = torch.zeros(n_q, n_rows, device="cuda")
    qsa.index_score(to_dev(inp["q_idx"]), to_dev(pooled), n_rows, H, d, scale, scores,
                    q_pos=to_dev(inp["q_pos"]), precision=qsa.QSA_PREC_BF16_TC, workspace=ws)
    got = to_host(scores)
    rows = np.random.default_rng(4).choice(n_q, 40, replace=False)
    want = oracle.scores(inp["q_idx"][rows], pooled, n_rows, H, d, scale,
                         q_pos=inp["q_pos"][rows], round_bf16_operands=True)
    qb = np.array([oracle.round_bf16(float(x)) for x in inp["q_idx"][rows].reshape(-1)],
                  np.float32).reshape(len(rows), -1)
    pvals = qsa_synth.bf16_bits_to_f32(pooled)
    for j, i in enumerate(rows):
        vis = np.isfinite(want[j])
        assert np.array_equal(np.isneginf(got[i]), ~vis)
        tol = score_tolerance(qb[j], pvals, n_rows, scale, chain=H * d)[vis]
        assert np.all(np.abs(got[i][vis] - want[j][vis]) <= tol)


# ------------------------------------------------------------------ decode steps

def _layer(shape, cap, store, max_queries):
    return qsa.DecodeLayer(cap_tokens=cap, H_idx=shape.H_idx, d_idx=shape.d_idx, H_q=shape.H_q,
                           H_kv=shape.H_kv, d=shape.d, top_k_tokens=shape.top_k_tokens,
                           pooled_dtype=torch.bfloat16 if store == "bf16" else torch.float32,
                           max_queries=max_queries)


@pytest.mark.parametrize("shape", [TINY, SMALL], ids=lambda s: s.name)
@pytest.mark.parametrize("store", ["f32", "bf16"])
def test_multi_query_decode_steps_match_oracle(shape, store):
    """Steps of 3, 1, 4 and 2 query tokens, each appending its tokens, against the oracle's
    multi-query step: per query the selection (boundary band), the cell list and the
    attention output; the pooled cache with the bf16 rule."""
    plan = [3, 1, 4, 2]
    extra = sum(plan)
    inp = qsa_synth.decode_inputs(shape, seed=44, extra_tokens=extra, n_steps=extra)
    H, d = shape.H_idx, shape.d_idx
    raw, w = to_dev(inp["raw_k"]), to_dev(inp["norm_w"])
    K, V = to_dev(inp["K"]), to_dev(inp["V"])
    n0 = shape.n_ctx
    lay = _layer(shape, n0 + extra, store, 4)
    lay.rebuild(raw, w, n0)
    cap_rows = (n0 + extra + 3) // 4
    o_pooled = oracle.pool_rows(inp["raw_k"], n0, H, d, inp["norm_w"], shape.eps,
                                shape.rope_base, 0, (n0 + 3) // 4,
                                np.zeros((cap_rows, H * d),
                                         np.uint16 if store == "bf16" else np.float32))
    o_valid = n0 // 4
    n_ctx, used, n_band = n0, 0, 0
    atol = ATOL_ATTN_BF16 if shape.dtype == "bf16" else ATOL_ATTN_F32
    scale = 1.0 / math.sqrt(d)
    for n_q in plan:
        n_ctx += n_q
        qi = inp["q_idx"][used:used + n_q]
        qa = inp["q"][used:used + n_q]
        used += n_q
        out = to_host(lay.step(raw, w, K, V, n_ctx, to_dev(qi), to_dev(qa)))
        res, o_scores = oracle.decode_step_multi(
            inp["raw_k"], n_ctx, H, d, inp["norm_w"], shape.eps, shape.rope_base, o_pooled,
            o_valid, qi, shape.top_k_tokens, qa, inp["K"], inp["V"], shape.H_q, shape.H_kv,
            shape.d)
        o_valid = n_ctx // 4
        n_rows = (n_ctx + 3) // 4
        if store == "bf16":
            z = pooled_f64(inp, shape, n_ctx, range(n_rows))
            check_bf16_rows(to_host(lay.pooled)[:n_rows], o_pooled[:n_rows], z, d)
        blocks = to_host(lay.blocks)
        counts = to_host(lay.counts)
        n_cells = to_host(lay.n_cells)
        pos = to_host(lay.pos)
        for i in range(n_q):
            p = n_ctx - n_q + i
            n_i = min(n_ctx // 4, (p + 1) // 4)
            band_abs = flip_band(qi[i], z[:n_i], d, scale) if store == "bf16" else None
            n_band += check_topk(blocks[i], int(counts[i]), o_scores[i], n_i, shape.k_blk,
                                 band_abs=band_abs)
            o_blocks, o_cells, o_out, _ = res[i]
            if np.array_equal(np.sort(blocks[i, :counts[i]]), o_blocks):
                np.testing.assert_array_equal(pos[i, :n_cells[i]], o_cells)
                np.testing.assert_allclose(out[i], o_out, rtol=0, atol=atol)
            else:
                assert len(np.sort(blocks[i, :counts[i]])) == len(o_blocks)
    assert n_band < 20


@pytest.mark.parametrize("store", ["f32", "bf16"])
def test_multi_query_composite_equals_separate_calls(store):
    """The fused step and the five calls (top-k and gather with q_pos = the last n_q
    positions) give bit-identical cache, selections, cell lists and outputs."""
    shape = SMALL
    plan = [2, 3, 1, 4]
    extra = sum(plan)
    inp = qsa_synth.decode_inputs(shape, seed=45, extra_tokens=extra, n_steps=extra)
    raw, w = to_dev(inp["raw_k"]), to_dev(inp["norm_w"])
    K, V = to_dev(inp["K"]), to_dev(inp["V"])
    a = _layer(shape, shape.n_ctx + extra, store, 4)
    b = _layer(shape, shape.n_ctx + extra, store, 4)
    a.rebuild(raw, w, shape.n_ctx - 1)
    b.rebuild(raw, w, shape.n_ctx - 1)
    n_ctx, used = shape.n_ctx - 1, 0
    for n_q in plan:
        n_ctx += n_q
        qi = to_dev(inp["q_idx"][used:used + n_q])
        qa = to_dev(inp["q"][used:used + n_q])
        used += n_q
        oa = a.step(raw, w, K, V, n_ctx, qi, qa).clone()
        ob = b.step_separate_calls(raw, w, K, V, n_ctx, qi, qa).clone()
        assert torch.equal(a.pooled, b.pooled)
        assert torch.equal(a.scores_of(n_q, n_ctx), b.scores_of(n_q, n_ctx))
        assert torch.equal(a.blocks[:n_q], b.blocks[:n_q])
        assert torch.equal(a.counts[:n_q], b.counts[:n_q])
        assert torch.equal(a.n_cells[:n_q], b.n_cells[:n_q])
        for i in range(n_q):
            nc = int(a.n_cells[i].item())
            assert torch.equal(a.pos[i, :nc], b.pos[i, :nc])
        assert torch.equal(oa, ob)


def test_multi_query_small_context_takes_every_block():
    """When a query has no more complete blocks than k, all of them are selected (the
    one-CTA form) and its tail still ends at its own position."""
    shape = qsa_synth.shrink(TINY, n_ctx=37)
    inp = qsa_synth.decode_inputs(shape, seed=46, n_steps=3)
    raw, w = to_dev(inp["raw_k"]), to_dev(inp["norm_w"])
    K, V = to_dev(inp["K"]), to_dev(inp["V"])
    lay = _layer(shape, 64, "f32", 3)
    out = to_host(lay.step(raw, w, K, V, 37, to_dev(inp["q_idx"][:3]), to_dev(inp["q"][:3])))
    res, _ = oracle.decode_step_multi(
        inp["raw_k"], 37, shape.H_idx, shape.d_idx, inp["norm_w"], shape.eps, shape.rope_base,
        np.zeros((10, shape.H_idx * shape.d_idx), np.float32), 0, inp["q_idx"][:3],
        shape.top_k_tokens, inp["q"][:3], inp["K"], inp["V"], shape.H_q, shape.H_kv, shape.d)
    for i in range(3):
        o_blocks, o_cells, o_out, _ = res[i]
        assert int(lay.counts[i].item()) == len(o_blocks)
        np.testing.assert_array_equal(to_host(lay.blocks)[i, :len(o_blocks)], o_blocks)
        np.testing.assert_array_equal(to_host(lay.pos)[i, :len(o_cells)], o_cells)
        np.testing.assert_allclose(out[i], o_out, rtol=0, atol=ATOL_ATTN_F32)


@pytest.mark.parametrize("shape,n_q,store,pinned", [
    (SMALL, 1, "f32", True), (SMALL, 3, "bf16", True), (TINY, 2, "f32", True),
    (SMALL, 2, "bf16", False), (TINY, 1, "f32", False)],
    ids=["bf16-1", "bf16-3", "f32-2", "bf16-2-pageable", "f32-1-pageable"])
def test_host_fed_step_equals_device_step(shape, n_q, store, pinned):
    """qsa_decode_step_host (new rows and queries from one packed host buffer, output back
    to host memory) writes the same cache rows and gives bit-identical results to
    qsa_decode_step on caches that already hold the new rows: with page-locked host buffers
    (read and written in place by the copy kernels) and with pageable ones (copy-engine
    transfers)."""
    inp = qsa_synth.decode_inputs(shape, seed=47, extra_tokens=n_q, n_steps=n_q)
    n0 = shape.n_ctx
    n_ctx = n0 + n_q
    raw, w, K, V = (to_dev(inp["raw_k"]), to_dev(inp["norm_w"]), to_dev(inp["K"]),
                    to_dev(inp["V"]))
    qi, qa = to_dev(inp["q_idx"]), to_dev(inp["q"])
    a = _layer(shape, n_ctx, store, n_q)
    a.rebuild(raw, w, n0)
    out_a = a.step(raw, w, K, V, n_ctx, qi, qa).clone()
    raw_b, K_b, V_b = raw.clone(), K.clone(), V.clone()
    raw_b[n0:n_ctx] = 0
    K_b[n0:n_ctx] = 0
    V_b[n0:n_ctx] = 0
    b = _layer(shape, n_ctx, store, n_q)
    b.rebuild(raw_b, w, n0)
    b.enable_host_feed(raw.dtype, K.dtype, pinned=pinned)
    assert b.h_in.is_pinned() == pinned
    b.bind(raw_b, w, K_b, V_b)
    hin = b.host_inputs(n_q)
    hin["raw"].copy_(raw[n0:n_ctx].reshape(n_q, -1).cpu())
    hin["k"].copy_(K[n0:n_ctx].reshape(n_q, -1).cpu())
    hin["v"].copy_(V[n0:n_ctx].reshape(n_q, -1).cpu())
    hin["q_idx"].copy_(qi.cpu())
    hin["q"].copy_(qa.cpu())
    b.step_host(n_ctx, torch.cuda.current_stream().cuda_stream, n_q, with_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(raw_b, raw) and torch.equal(K_b, K) and torch.equal(V_b, V)
    assert torch.equal(a.pooled, b.pooled)
    assert torch.equal(a.blocks[:n_q], b.blocks[:n_q])
    assert torch.equal(a.n_cells[:n_q], b.n_cells[:n_q])
    assert torch.equal(b.h_out[:n_q], out_a.cpu())
    assert torch.equal(b.h_lse[:n_q], a.lse[:n_q].cpu())


@pytest.mark.parametrize("n_q,store", [(1, "f32"), (3, "bf16")])
def test_plan_steps_equal_decode_step(n_q, store):
    """Steps through a qsa_decode_plan (the fixed arguments bound once) equal
    qsa_decode_step with all arguments, bit for bit, over several consecutive steps."""
    shape = SMALL
    steps = 5
    inp = qsa_synth.decode_inputs(shape, seed=61, extra_tokens=steps + n_q, n_steps=n_q)
    raw, w, K, V = (to_dev(inp["raw_k"]), to_dev(inp["norm_w"]), to_dev(inp["K"]),
                    to_dev(inp["V"]))
    qi, qa = to_dev(inp["q_idx"]), to_dev(inp["q"])
    n0 = shape.n_ctx
    a = _layer(shape, n0 + steps + n_q, store, n_q)
    b = _layer(shape, n0 + steps + n_q, store, n_q)
    a.rebuild(raw, w, n0)
    b.rebuild(raw, w, n0)
    b.bind(raw, w, K, V)
    sp = torch.cuda.current_stream().cuda_stream
    for t in range(steps):
        n_ctx = n0 + n_q + t
        out_a = a.step(raw, w, K, V, n_ctx, qi, qa)
        b.step_ptr(n_ctx, qi.data_ptr(), qa.data_ptr(), sp, n_q)
        torch.cuda.synchronize()
        assert torch.equal(a.pooled, b.pooled)
        assert torch.equal(a.counts[:n_q], b.counts[:n_q])
        assert torch.equal(a.blocks[:n_q], b.blocks[:n_q])
        assert torch.equal(a.pos[:n_q], b.pos[:n_q])
        assert torch.equal(out_a, b.out[:n_q])
        assert torch.equal(a.lse[:n_q], b.lse[:n_q])


@pytest.mark.parametrize("n_q,n_rows", [(130, 45_000), (1024, 64_052)])
def test_tensor_core_scores_fp32_cache_equal_bf16_cache(n_q, n_rows):
    """An fp32 cache goes through the tensor-core contraction as its bf16 rounding (a
    rounding pass into the workspace, then the contraction): the result is bit-identical to
    the same call on a bf16 cache holding that rounding (read in place), and rows invisible
    to a query stay -inf.  (The oracle pins the bf16-cache path elsewhere.)"""
    H, d = 16, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(n_rows)
    pooled = torch.randn(n_rows, H * d, device="cuda", generator=g)
    q = torch.randn(n_q, H * d, device="cuda", generator=g)
    depth = 4 * n_rows - n_q - 700  # the last queries see every row, the first do not
    q_pos = torch.arange(depth, depth + n_q, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    out = {}
    for dt in (qsa.QSA_F32, qsa.QSA_BF16):
        src = pooled if dt == qsa.QSA_F32 else pooled.to(torch.bfloat16)
        ws = torch.zeros(qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC,
                                                        dt), dtype=torch.uint8, device="cuda")
        scores = torch.full((n_q, n_rows + 3), 5.0, device="cuda")
        qsa.index_score(q, src, n_rows, H, d, scale, scores, q_pos=q_pos,
                        precision=qsa.QSA_PREC_BF16_TC, workspace=ws)
        out[dt] = scores
    torch.cuda.synchronize()
    a, b = out[qsa.QSA_F32], out[qsa.QSA_BF16]
    assert torch.equal(a, b)
    assert torch.all(a[:, n_rows:] == 5.0)
    lim = (q_pos.long() + 1) // 4
    cols = torch.arange(n_rows, device="cuda")
    invisible = cols[None, :] >= lim[:, None]
    assert torch.all(torch.isneginf(a[:, :n_rows][invisible]))
    assert torch.all(torch.isfinite(a[:, :n_rows][~invisible]))


@pytest.mark.parametrize("store", ["f32", "bf16"])
def test_rejected_drafts_roll_back(store):
    """Speculative decode: a step carries a token and two drafts; the drafts are rejected,
    a different token is written in the first draft's place, the layer is told which rows
    changed, and the next step runs one query.  Its cache, selection and output equal those
    of a layer that never saw the drafts (rebuilt at the accepted length, then stepped)."""
    shape = SMALL
    n0 = shape.n_ctx + 2  # 9,005: the drafts straddle a block boundary (9,004 = 4 * 2,251)
    inp = qsa_synth.decode_inputs(qsa_synth.shrink(shape, n_ctx=n0), seed=71, extra_tokens=4,
                                  n_steps=4)
    raw, w, K, V = (to_dev(inp["raw_k"]), to_dev(inp["norm_w"]), to_dev(inp["K"]),
                    to_dev(inp["V"]))
    qi, qa = to_dev(inp["q_idx"]), to_dev(inp["q"])
    cap = n0 + 8
    # speculative layer: three queries at n0+1 .. n0+3 (token n0, drafts n0+1, n0+2)
    a = _layer(shape, cap, store, 3)
    a.rebuild(raw, w, n0)
    a.step(raw, w, K, V, n0 + 3, qi[:3], qa[:3])
    # the drafts are rejected: token n0+1 is replaced, row n0+2 is dropped
    raw2, K2, V2 = raw.clone(), K.clone(), V.clone()
    raw2[n0 + 1] = raw[n0 + 3]
    K2[n0 + 1], V2[n0 + 1] = K[n0 + 3], V[n0 + 3]
    a.invalidate(n0 + 1)
    out_a = a.step(raw2, w, K2, V2, n0 + 2, qi[3:4], qa[3:4]).clone()
    # reference layer: the accepted context only
    b = _layer(shape, cap, store, 3)
    b.rebuild(raw2, w, n0 + 1)
    out_b = b.step(raw2, w, K2, V2, n0 + 2, qi[3:4], qa[3:4]).clone()
    torch.cuda.synchronize()
    n_rows = (n0 + 2 + 3) // 4
    assert torch.equal(a.pooled[:n_rows], b.pooled[:n_rows])
    assert torch.equal(a.counts[:1], b.counts[:1])
    assert torch.equal(a.blocks[:1], b.blocks[:1])
    assert torch.equal(a.n_cells[:1], b.n_cells[:1])
    assert torch.equal(a.pos[:1, :int(b.n_cells[0])], b.pos[:1, :int(b.n_cells[0])])
    assert torch.equal(out_a, out_b)


def test_plan_steps_with_changing_query_counts():
    """One plan, steps of 1, 3, 1, 4 and 2 queries (the workspace layout moves with the
    count, so the histogram kept for the next step is rebuilt when it no longer matches):
    each equals qsa_decode_step with all arguments, bit for bit."""
    shape = SMALL
    seq = [1, 3, 1, 4, 2]
    total = sum(seq)
    inp = qsa_synth.decode_inputs(shape, seed=83, extra_tokens=total, n_steps=4)
    raw, w, K, V = (to_dev(inp["raw_k"]), to_dev(inp["norm_w"]), to_dev(inp["K"]),
                    to_dev(inp["V"]))
    qi, qa = to_dev(inp["q_idx"]), to_dev(inp["q"])
    n0 = shape.n_ctx
    a = _layer(shape, n0 + total, "f32", 4)
    b = _layer(shape, n0 + total, "f32", 4)
    a.rebuild(raw, w, n0)
    b.rebuild(raw, w, n0)
    b.bind(raw, w, K, V)
    sp = torch.cuda.current_stream().cuda_stream
    n_ctx = n0
    for n_q in seq:
        n_ctx += n_q
        out_a = a.step(raw, w, K, V, n_ctx, qi[:n_q], qa[:n_q])
        b.step_ptr(n_ctx, qi.data_ptr(), qa.data_ptr(), sp, n_q)
        torch.cuda.synchronize()
        assert torch.equal(a.pooled, b.pooled)
        assert torch.equal(a.blocks[:n_q], b.blocks[:n_q])
        assert torch.equal(a.n_cells[:n_q], b.n_cells[:n_q])
        assert torch.equal(out_a, b.out[:n_q])


def test_bf16_mirror_of_an_fp32_cache_is_its_rounding():
    """An fp32 pooled cache kept together with a bf16 mirror (every pool update also written
    into the mirror) for the tensor-core prefill scores: after a rebuild and an incremental
    chunk of 1,024 tokens, the mirror is bit for bit the fp32 cache rounded to bf16 (nearest
    even: the update computes one fp32 value per element and rounds it for bf16 storage), so
    the scores read from the mirror in place equal those of the fp32 cache's own rounding
    pass."""
    shape = qsa_synth.shrink(qsa_synth.CONFIGS["prefill_256k"], depth=40_001)
    inp = qsa_synth.prefill_inputs(shape, seed=4096)
    H, d, n_q, n_rows, n_ctx = shape.H_idx, shape.d_idx, shape.n_q, shape.n_rows, shape.n_ctx
    raw, w = to_dev(inp["raw_k"]), to_dev(inp["norm_w"])
    f32 = torch.zeros(n_rows, H * d, device="cuda")
    mirror = torch.zeros(n_rows, H * d, dtype=torch.bfloat16, device="cuda")
    for cache in (f32, mirror):
        qsa.pool_update(raw, shape.depth, H, d, w, shape.eps, shape.rope_base, cache, 0)
        qsa.pool_update(raw, n_ctx, H, d, w, shape.eps, shape.rope_base, cache, shape.depth // 4)
    torch.cuda.synchronize()
    assert torch.equal(mirror.view(torch.int16), f32.to(torch.bfloat16).view(torch.int16))
    q_pos = to_dev(inp["q_pos"])
    q = to_dev(inp["q_idx"])
    out = []
    for src, dt in ((f32, qsa.QSA_F32), (mirror, qsa.QSA_BF16)):
        ws = torch.zeros(qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC,
                                                        dt), dtype=torch.uint8, device="cuda")
        sc = torch.empty(n_q, n_rows, device="cuda")
        qsa.index_score(q, src, n_rows, H, d, 1.0 / math.sqrt(d), sc, q_pos=q_pos,
                        precision=qsa.QSA_PREC_BF16_TC, workspace=ws)
        out.append(sc)
    torch.cuda.synchronize()
    assert torch.equal(out[0], out[1])
