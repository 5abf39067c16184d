"""GPU parity of the pieces of the pages' earlier decode path, which the benchmark times
against the QSA path (the A/B the pages ran with same-binary switches): the block score
expanded to cells followed by a cell-level top-k, and attention over every cell of the
context.  Inputs and expected values come from qsa_synth and the oracle only."""
import math

import numpy as np
import pytest
import torch

import gather_qsa_pool_gb300 as qsa
import qsa_synth
from oracle import oracle
from gpu_helpers import ATOL_ATTN_BF16, to_dev, to_host

pytestmark = pytest.mark.gpu


def test_expand_block_scores_bit_exact():
    rng = np.random.default_rng(51)
    n_q, n_full, ld = 3, 5003, 5010
    s = rng.standard_normal((n_q, ld)).astype(np.float32)
    s[1, 7] = np.nan
    s[2, 9] = -0.0
    cells = torch.full((n_q, 4 * n_full + 6), 8.0, device="cuda")
    qsa.expand_block_scores(to_dev(s), n_full, cells)
    got = to_host(cells)
    for i in range(n_q):
        want = oracle.expand_block_scores(s[i].astype(np.float64), n_full).astype(np.float32)
        np.testing.assert_array_equal(got[i, :4 * n_full].view(np.uint32), want.view(np.uint32))
    assert np.all(got[:, 4 * n_full:] == 8.0)


@pytest.mark.parametrize("n_full,k_tokens", [(15_447, 2048), (63_795, 2048), (3_000, 64)])
def test_cell_level_topk_is_the_pages_old_path(n_full, k_tokens):
    """GPU expansion + GPU top-k over cells equals the oracle's top-k over the oracle's
    expanded cells (identical fp32 scores: exact), and the cells form the blocks of the
    block-domain top-k."""
    rng = np.random.default_rng(52 + n_full)
    s = rng.standard_normal(n_full).astype(np.float32)
    d_s = to_dev(s[None])
    cells = torch.empty(1, 4 * n_full, device="cuda")
    qsa.expand_block_scores(d_s, n_full, cells)
    sel = torch.empty(1, k_tokens, dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(cells, 4 * n_full, k_tokens, sel, cnt)
    got = to_host(sel)[0, :int(cnt.item())]
    want = oracle.topk(oracle.expand_block_scores(s.astype(np.float64), n_full), 4 * n_full,
                       k_tokens)
    np.testing.assert_array_equal(got, want)
    blk = torch.empty(1, k_tokens // 4, dtype=torch.int32, device="cuda")
    qsa.topk_blocks(d_s, n_full, k_tokens // 4, blk, cnt)
    np.testing.assert_array_equal(np.unique(got // 4), to_host(blk)[0])


def test_full_kv_attention_is_dense_attention():
    """qsa_sparse_attn over a list of every position of the context (the attention before
    the selected-K/V gather) equals the oracle's attention over every cell."""
    shape = qsa_synth.shrink(qsa_synth.CONFIGS["decode_64k"], n_ctx=9_003)
    inp = qsa_synth.decode_inputs(shape, seed=53)
    n = shape.n_ctx
    pos = torch.arange(n, dtype=torch.int32, device="cuda").view(1, n)
    n_cells = torch.tensor([n], dtype=torch.int32, device="cuda")
    out = torch.empty(1, shape.H_q, shape.d, device="cuda")
    ws = torch.zeros(max(qsa.sparse_attn_workspace_size(1, shape.H_q, shape.H_kv, shape.d, n)
                         // 4, 1), device="cuda")
    scale = 1.0 / math.sqrt(shape.d)
    qsa.sparse_attn(to_dev(inp["q"][:1]), to_dev(inp["K"]), to_dev(inp["V"]), n_cells, n, out,
                    shape.H_kv, shape.d, shape.d, scale, pos=pos, workspace=ws)
    want, _ = oracle.attention(inp["q"][0], inp["K"], inp["V"], shape.H_q, shape.H_kv, shape.d,
                               shape.d, shape.H_kv * shape.d, shape.H_kv * shape.d,
                               np.arange(n, dtype=np.int32), scale)
    np.testing.assert_allclose(to_host(out)[0], want, rtol=0, atol=ATOL_ATTN_BF16)
