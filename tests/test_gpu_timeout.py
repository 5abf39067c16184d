"""Bounded device waits reported through qsa_set_wait_options.

Each kernel that waits on its own asynchronous copies or tensor-core work is run with the
pipeline limit at 0 (every such wait gives up at once, without looking).  The kernel must then
store QSA_ERR_TIMEOUT into the status word, stop issuing, wait (with the default limit) for
the copies and MMAs it had issued, return its tensor memory and leave: its outputs are NaN
(attention) or untouched (scores), and a normal call afterwards on the same context gives the
normal result again without touching the status.  No wait here is unbounded and no
kernel is made to fault: the failure is a time limit the caller chose."""
import math

import numpy as np
import pytest
import torch

import gather_qsa_pool_gb300 as qsa
import qsa_synth
from gpu_helpers import to_dev, to_host

pytestmark = pytest.mark.gpu

TIMEOUT = 4  # QSA_ERR_TIMEOUT


@pytest.fixture
def status():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    yield st
    qsa.set_wait_options(None, qsa.QSA_WAIT_DEFAULT_NS)  # later tests get the defaults


def _gave_up_then_recovers(run, status, outputs):
    """run() fills the output tensors; returns (normal outputs, outputs under limit 0)."""
    run()
    torch.cuda.synchronize()
    normal = [to_host(o).copy() for o in outputs]
    qsa.set_wait_options(status, 0)
    for o in outputs:
        o.fill_(float("nan")) if o.dtype.is_floating_point else o.fill_(-7)
    run()
    torch.cuda.synchronize()
    limited = [to_host(o).copy() for o in outputs]
    assert int(status.item()) == TIMEOUT
    # back to the defaults: the normal result again, and the status untouched
    qsa.set_wait_options(status, qsa.QSA_WAIT_DEFAULT_NS)
    status.zero_()
    run()
    torch.cuda.synchronize()
    for o, want in zip(outputs, normal):
        np.testing.assert_array_equal(to_host(o), want)
    assert int(status.item()) == 0
    qsa.set_wait_options(None, qsa.QSA_WAIT_DEFAULT_NS)
    return normal, limited


def _rows_nan_or_equal(got, want):
    """Rows (last axis) either all NaN or bit-identical to the normal result; returns the
    fraction of NaN rows (1 when every part of the kernel gave up, as a limit of 0 makes it)."""
    g = got.reshape(-1, got.shape[-1])
    w = want.reshape(-1, want.shape[-1])
    nan_rows = np.isnan(g).all(axis=1)
    assert np.array_equal(g[~nan_rows], w[~nan_rows])
    return float(nan_rows.mean())


def _decode_attn_case(n_q, seed):
    shape = qsa_synth.CONFIGS["decode_64k"]
    rng = np.random.default_rng(seed)
    n_ctx, H_q, H_kv, d = 20000, shape.H_q, shape.H_kv, shape.d
    K = to_dev(qsa_synth.to_bf16_bits(rng.standard_normal((n_ctx, H_kv, d)).astype(np.float32)))
    V = to_dev(qsa_synth.to_bf16_bits(rng.standard_normal((n_ctx, H_kv, d)).astype(np.float32)))
    q = to_dev(rng.standard_normal((n_q, H_q, d)).astype(np.float32))
    max_cells = shape.max_cells
    pos = to_dev(np.stack([np.sort(rng.choice(n_ctx, max_cells, replace=False))
                           for _ in range(n_q)]).astype(np.int32))
    n = to_dev(np.full(n_q, max_cells, np.int32))
    return K, V, q, pos, n, max_cells, H_kv, d


def test_decode_attention_gives_up_and_recovers(status):
    """The decode shape (one query, 32 / 4 heads, 2,051 cells): the tensor-core kernel whose
    splits merge in a thread-block cluster."""
    K, V, q, pos, n, max_cells, H_kv, d = _decode_attn_case(1, 11)
    out = torch.empty(1, 32, d, device="cuda")
    lse = torch.empty(1, 32, device="cuda")

    def run():
        qsa.sparse_attn(q, K, V, n, max_cells, out, H_kv, d, d, 1 / math.sqrt(d), pos=pos,
                        lse=lse)

    (w_out, w_lse), (g_out, g_lse) = _gave_up_then_recovers(run, status, [out, lse])
    assert _rows_nan_or_equal(g_out, w_out) == 1.0
    assert np.array_equal(np.isnan(g_lse), np.isnan(g_out).all(axis=-1))


def test_many_query_attention_gives_up_and_recovers(status):
    """152 queries of the prefill form (one CTA per query, a producer warp feeding a ring)."""
    K, V, q, pos, n, max_cells, H_kv, d = _decode_attn_case(152, 12)
    out = torch.empty(152, 32, d, device="cuda")

    def run():
        qsa.sparse_attn(q, K, V, n, max_cells, out, H_kv, d, d, 1 / math.sqrt(d), pos=pos)

    (w_out,), (g_out,) = _gave_up_then_recovers(run, status, [out])
    assert _rows_nan_or_equal(g_out, w_out) == 1.0


def test_union_attention_gives_up_and_recovers(status):
    K, V, q, pos, n, max_cells, H_kv, d = _decode_attn_case(48, 13)
    out = torch.empty(48, 32, d, device="cuda")
    ws = torch.empty(qsa.sparse_attn_union_workspace_size(48, max_cells), dtype=torch.uint8,
                     device="cuda")

    def run():
        qsa.sparse_attn_union(q, K, V, n, max_cells, out, H_kv, d, 1 / math.sqrt(d), pos,
                              workspace=ws)

    (w_out,), (g_out,) = _gave_up_then_recovers(run, status, [out])
    assert _rows_nan_or_equal(g_out, w_out) == 1.0


def test_latent_mask_attention_gives_up_and_recovers(status):
    shape = qsa_synth.CONFIGS["mask_32k"]
    inp = qsa_synth.mask_attn_inputs(shape, seed=14)
    mask = to_dev(qsa_synth.mask_rows(shape.n_q, shape.n_kv, seed=15))
    q, KV = to_dev(inp["q"]), to_dev(inp["KV"])
    out = torch.empty(shape.n_q, shape.H_q, shape.d_v, device="cuda")
    counts = torch.empty(shape.n_q, dtype=torch.int32, device="cuda")

    def run():
        qsa.mask_sparse_attn(q, KV, mask, shape.max_list, out, 1.0 / math.sqrt(shape.d_k),
                             counts_out=counts)

    (w_out, w_cnt), (g_out, g_cnt) = _gave_up_then_recovers(run, status, [out, counts])
    np.testing.assert_array_equal(g_cnt, w_cnt)  # the counts need no wait
    assert _rows_nan_or_equal(g_out, w_out) == 1.0


@pytest.mark.parametrize("n_q", [512, 200])
def test_tensor_core_scores_give_up_and_recover(status, n_q):
    """The tcgen05 score contraction, in clusters of two CTA pairs sharing each pooled tile
    (512 queries: two query blocks of 256) and of one pair (200 queries): no tile is stored,
    so every score keeps the NaN it was filled with."""
    rng = np.random.default_rng(16)
    n_rows, H, d = 6000, 16, 128
    q = to_dev(rng.standard_normal((n_q, H * d)).astype(np.float32))
    pooled = to_dev(rng.standard_normal((n_rows, H * d)).astype(np.float32))
    scores = torch.empty(n_q, n_rows, device="cuda")
    ws = torch.zeros(qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC),
                     dtype=torch.uint8, device="cuda")

    def run():
        qsa.index_score(q, pooled, n_rows, H, d, 1 / math.sqrt(d), scores,
                        precision=qsa.QSA_PREC_BF16_TC, workspace=ws)

    (w_sc,), (g_sc,) = _gave_up_then_recovers(run, status, [scores])
    assert np.isnan(g_sc).all()  # no tile was stored


def test_decode_step_gives_up_and_recovers(status):
    """A whole decode step at 61,789 tokens: the score and top-k kernels have no waits, the
    attention gives up; the selection is unaffected."""
    shape = qsa_synth.CONFIGS["decode_64k"]
    inp = qsa_synth.decode_inputs(shape, seed=17, extra_tokens=1, n_steps=1)
    raw, w, K, V = (to_dev(inp["raw_k"]), to_dev(inp["norm_w"]), to_dev(inp["K"]),
                    to_dev(inp["V"]))
    q_idx, q = to_dev(inp["q_idx"][0]), to_dev(inp["q"][0])
    lay = qsa.DecodeLayer(cap_tokens=shape.n_ctx + 1, H_idx=shape.H_idx, d_idx=shape.d_idx,
                          H_q=shape.H_q, H_kv=shape.H_kv, d=shape.d,
                          top_k_tokens=shape.top_k_tokens, eps=shape.eps,
                          rope_base=shape.rope_base)
    n_ctx = shape.n_ctx

    def run():
        lay.rebuild(raw, w, n_ctx - 1)
        lay.step(raw, w, K, V, n_ctx, q_idx, q)

    (w_out, w_blk), (g_out, g_blk) = _gave_up_then_recovers(run, status, [lay.out, lay.blocks])
    np.testing.assert_array_equal(g_blk, w_blk)
    assert _rows_nan_or_equal(g_out, w_out) == 1.0


def test_tensor_core_scores_with_maxima_give_up_and_recover(status):
    """The score contraction that also writes the group maxima: when it gives up, neither
    scores nor maxima are stored (both keep the NaN they were filled with); afterwards the
    normal result, maxima included, comes back bit for bit."""
    rng = np.random.default_rng(18)
    n_q, n_rows, H, d = 300, 5000, 16, 128
    q = to_dev(rng.standard_normal((n_q, H * d)).astype(np.float32))
    pooled = to_dev(rng.standard_normal((n_rows, H * d)).astype(np.float32))
    scores = torch.empty(n_q, n_rows, device="cuda")
    maxima = torch.empty(n_q, (n_rows + 31) // 32, device="cuda")
    ws = torch.zeros(qsa.index_score_workspace_size(n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC),
                     dtype=torch.uint8, device="cuda")

    def run():
        qsa.index_score_maxima(q, pooled, n_rows, H, d, 1 / math.sqrt(d), scores, maxima,
                               workspace=ws)

    (w_sc, w_mx), (g_sc, g_mx) = _gave_up_then_recovers(run, status, [scores, maxima])
    assert np.isnan(g_sc).all() and np.isnan(g_mx).all()
    assert np.isfinite(w_mx).all()
