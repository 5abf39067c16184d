"""Pins of the oracle's sparse attention and mask -> position-list steps."""
import math

import numpy as np
import pytest
import torch

from oracle import oracle
import qsa_synth


def _kv(rng, n, H_kv, d):
    return (rng.standard_normal((n, H_kv, d)).astype(np.float32),
            rng.standard_normal((n, H_kv, d)).astype(np.float32))


def test_all_blocks_selected_equals_library_dense_causal_attention():
    """With k_blk >= n_full the selected set is every cell up to the query, so the
    sparse result must equal dense causal attention (torch SDPA, fp64, GQA by repeating
    each KV head for its consecutive query heads)."""
    rng = np.random.default_rng(40)
    H_q, H_kv, d, n_ctx = 8, 2, 32, 23
    K, V = _kv(rng, n_ctx, H_kv, d)
    q = rng.standard_normal((H_q, d)).astype(np.float32)
    n_full = n_ctx // 4
    blocks = oracle.topk(rng.standard_normal(n_full), n_full, 64)
    cl = oracle.cells(blocks, n_ctx - 1)
    np.testing.assert_array_equal(cl, np.arange(n_ctx))
    out, lse = oracle.attention(q, K, V, H_q, H_kv, d, d, H_kv * d, H_kv * d, cl, d ** -0.5)
    Kt = torch.from_numpy(K.astype(np.float64)).permute(1, 0, 2).repeat_interleave(H_q // H_kv, 0)
    Vt = torch.from_numpy(V.astype(np.float64)).permute(1, 0, 2).repeat_interleave(H_q // H_kv, 0)
    qt = torch.from_numpy(q.astype(np.float64))[:, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt)[:, 0, :].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    ref_lse = torch.logsumexp((qt @ Kt.transpose(1, 2))[:, 0, :] * d ** -0.5, dim=-1).numpy()
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12)


def test_single_cell_returns_its_value_row():
    rng = np.random.default_rng(41)
    K, V = _kv(rng, 10, 2, 16)
    q = rng.standard_normal((4, 16)).astype(np.float32)
    out, lse = oracle.attention(q, K, V, 4, 2, 16, 16, 32, 32, np.array([7], np.int32), 0.25)
    for h in range(4):
        g = h * 2 // 4
        np.testing.assert_array_equal(out[h], V[7, g].astype(np.float64))
        assert lse[h] == pytest.approx(0.25 * float(q[h].astype(np.float64) @ K[7, g]), rel=1e-14)


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(42)
    K, V = _kv(rng, 30, 1, 8)
    cl = np.array([1, 4, 9, 29, 17], np.int32)
    out, lse = oracle.attention(np.zeros((2, 8), np.float32), K, V, 2, 1, 8, 8, 8, 8, cl, 1.0)
    np.testing.assert_allclose(out[0], V[cl, 0].astype(np.float64).mean(0), rtol=1e-14)
    assert lse[0] == pytest.approx(math.log(5.0), rel=1e-15)


def test_permutation_invariance_and_gqa_mapping():
    rng = np.random.default_rng(43)
    H_q, H_kv, d = 8, 2, 16
    K, V = _kv(rng, 50, H_kv, d)
    V[:, 0, :] = -5.0
    V[:, 1, :] = 5.0
    q = rng.standard_normal((H_q, d)).astype(np.float32)
    cl = rng.permutation(50)[:20].astype(np.int32)
    out, _ = oracle.attention(q, K, V, H_q, H_kv, d, d, H_kv * d, H_kv * d, cl, 0.3)
    # consecutive query heads share a KV head: heads 0..3 -> group 0, 4..7 -> group 1
    np.testing.assert_allclose(out[:4], -5.0, rtol=1e-13)
    np.testing.assert_allclose(out[4:], 5.0, rtol=1e-13)
    K2, V2 = _kv(rng, 50, H_kv, d)
    o1, l1 = oracle.attention(q, K2, V2, H_q, H_kv, d, d, H_kv * d, H_kv * d, cl, 0.3)
    o2, l2 = oracle.attention(q, K2, V2, H_q, H_kv, d, d, H_kv * d, H_kv * d, cl[::-1].copy(), 0.3)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)


def test_large_logits_are_stable_and_pick_the_max():
    K = np.zeros((3, 1, 2), np.float32)
    K[:, 0, 0] = [1.0, 3.0, 2.0]
    V = np.arange(6, dtype=np.float32).reshape(3, 1, 2)
    out, lse = oracle.attention(np.array([[1000.0, 0.0]], np.float32), K, V, 1, 1, 2, 2, 2, 2,
                                np.array([0, 1, 2], np.int32), 1.0)
    np.testing.assert_allclose(out[0], V[1, 0], atol=1e-300)
    assert lse[0] == pytest.approx(3000.0, rel=1e-15)


def test_empty_cell_list():
    K = np.zeros((2, 1, 4), np.float32)
    out, lse = oracle.attention(np.ones((2, 4), np.float32), K, K, 2, 1, 4, 4, 4, 4,
                                np.zeros(0, np.int32), 1.0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_bf16_storage_equals_decoded_fp32():
    rng = np.random.default_rng(44)
    Kf, Vf = _kv(rng, 20, 2, 8)
    Kb, Vb = qsa_synth.to_bf16_bits(Kf), qsa_synth.to_bf16_bits(Vf)
    q = rng.standard_normal((4, 8)).astype(np.float32)
    cl = np.array([0, 3, 19, 5], np.int32)
    o_b, l_b = oracle.attention(q, Kb, Vb, 4, 2, 8, 8, 16, 16, cl, 0.5)
    o_f, l_f = oracle.attention(q, qsa_synth.bf16_bits_to_f32(Kb), qsa_synth.bf16_bits_to_f32(Vb),
                                4, 2, 8, 8, 16, 16, cl, 0.5)
    np.testing.assert_array_equal(o_b, o_f)
    np.testing.assert_array_equal(l_b, l_f)


def test_value_rows_may_alias_key_rows_with_a_stride():
    """Latent-KV layout: V is the first d_v columns of each K row (row stride d_k)."""
    rng = np.random.default_rng(45)
    d_k, d_v, n = 12, 8, 9
    KV = rng.standard_normal((n, d_k)).astype(np.float32)
    q = rng.standard_normal((3, d_k)).astype(np.float32)
    cl = np.array([2, 8, 4], np.int32)
    out, _ = oracle.attention(q, KV, KV, 3, 1, d_k, d_v, d_k, d_k, cl, 0.1)
    logits = 0.1 * q.astype(np.float64) @ KV[cl].astype(np.float64).T
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    np.testing.assert_allclose(out, p @ KV[cl, :d_v].astype(np.float64), rtol=1e-12)


# ------------------------------------------------------------------ mask -> list

@pytest.mark.parametrize("n_kv", [32768, 1000, 64, 63, 1])
def test_mask_list_matches_library_nonzero_and_packbits(n_kv):
    m = qsa_synth.mask_rows(1, n_kv, seed=n_kv)[0]
    pos, cnt, bits = oracle.mask_to_list(m, 4096)
    nz = np.flatnonzero(m)
    assert cnt == nz.shape[0]
    np.testing.assert_array_equal(pos, nz[:4096])
    packed = np.packbits(m != 0, bitorder="little")
    packed = np.concatenate([packed, np.zeros((-packed.shape[0]) % 8, np.uint8)])
    np.testing.assert_array_equal(bits, packed.view("<u8"))
    assert sum(bin(int(w)).count("1") for w in bits) == cnt


def test_mask_list_overflow_keeps_true_count():
    m = np.ones(5000, np.uint8)
    pos, cnt, _ = oracle.mask_to_list(m, 2048)
    assert cnt == 5000
    np.testing.assert_array_equal(pos, np.arange(2048))


def test_all_ones_mask_gives_dense_attention():
    rng = np.random.default_rng(46)
    n_kv, d = 40, 8
    KV = rng.standard_normal((n_kv, d)).astype(np.float32)
    q = rng.standard_normal((2, d)).astype(np.float32)
    pos, cnt, _ = oracle.mask_to_list(np.ones(n_kv, np.uint8), 64)
    out, _ = oracle.attention(q, KV, KV, 2, 1, d, d, d, d, pos, 0.5)
    logits = 0.5 * q.astype(np.float64) @ KV.astype(np.float64).T
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    np.testing.assert_allclose(out, p @ KV.astype(np.float64), rtol=1e-12)
