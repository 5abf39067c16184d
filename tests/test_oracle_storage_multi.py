"""Pins of the oracle's bf16 pooled-key storage and of its multi-query decode step.

bf16 storage: the rounding is checked against the library's fp32 -> bf16 conversion,
against a brute-force nearest search over every finite bf16 value, and on a value where
rounding through fp32 first would give a different answer; the stored cache and the
scores over it are checked against the fp32-stored cache and a library matrix product.

Multi-query decode (a token and its draft tokens verified in one step): each query must
give exactly what a one-query decode step at its own position gives, because the
visibility rule makes every query see only the blocks complete at its position.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle
import qsa_synth


def _lib_bf16_bits(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_from_f64_matches_library_on_fp32_values():
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(500) * 1e30).astype(np.float32),
        (rng.standard_normal(500) * 1e-39).astype(np.float32),  # subnormal range
        np.array([0.0, -0.0, 1.0, -2.5, 3.3e38, -3.39e38], np.float32),
    ])
    ours = np.array([oracle.bf16_bits_from_f64(float(v)) for v in x], np.uint16)
    np.testing.assert_array_equal(ours, _lib_bf16_bits(x))


def test_bf16_from_f64_rounds_once_not_through_fp32():
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7; a value just above it rounds up.
    # Through fp32 the 2^-40 is lost, the midpoint ties to even and the result is 1.0.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert oracle.bf16_bits_from_f64(x) == 0x3F81
    assert int(_lib_bf16_bits(np.array([x], np.float32))[0]) == 0x3F80
    assert oracle.bf16_bits_from_f64(1.0 + 2.0 ** -8) == 0x3F80        # tie -> even
    assert oracle.bf16_bits_from_f64(1.0 + 3 * 2.0 ** -8) == 0x3F82    # tie -> even
    assert oracle.bf16_bits_from_f64(-(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 0xBF81
    assert oracle.bf16_bits_from_f64(math.inf) == 0x7F80
    assert oracle.bf16_bits_from_f64(4e38) == 0x7F80                   # overflow


def test_bf16_from_f64_brute_force_nearest():
    # every finite non-negative bf16 value, ascending with the bit pattern
    bits = np.arange(0x7F80, dtype=np.uint32)
    vals = (bits << np.uint32(16)).view(np.float32).astype(np.float64)
    rng = np.random.default_rng(12)
    xs = list(rng.standard_normal(300) * 10.0 ** rng.integers(-30, 30, 300))
    # values right at and around midpoints of neighbouring bf16 values
    for j in rng.integers(1, 0x7F7E, 100):
        mid = 0.5 * (vals[j] + vals[j + 1])
        xs += [mid, math.nextafter(mid, math.inf), math.nextafter(mid, -math.inf)]
    for x in xs:
        a = abs(x)
        dist = np.abs(vals - a)
        best = np.flatnonzero(dist == dist.min())
        want = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
        if x < 0:
            want |= 0x8000
        assert oracle.bf16_bits_from_f64(x) == want, x


def test_pool_rows_bf16_store_is_nearest_to_the_fp32_store():
    shape = qsa_synth.shrink(qsa_synth.CONFIGS["decode_64k"], n_ctx=203)
    inp = qsa_synth.decode_inputs(shape, seed=5)
    args = (inp["raw_k"], shape.n_ctx, shape.H_idx, shape.d_idx, inp["norm_w"], shape.eps,
            shape.rope_base)
    p32 = oracle.pool_rows(*args, 0, shape.n_rows)
    p16 = oracle.pool_rows(*args, 0, shape.n_rows, store="bf16")
    assert p16.dtype == np.uint16
    v16 = qsa_synth.bf16_bits_to_f32(p16).astype(np.float64)
    # half a bf16 unit of the value (8 significant bits), plus the fp32 store's own rounding
    ulp = np.exp2(np.floor(np.log2(np.abs(p32.astype(np.float64)))) - 7)
    assert np.all(np.abs(v16 - p32) <= 0.5 * ulp * (1 + 2.0 ** -16))
    # rows outside the range stay untouched
    p16b = np.full_like(p16, 0x1234)
    oracle.pool_rows(*args, 10, 20, pooled=p16b)
    assert np.all(p16b[:10] == 0x1234) and np.all(p16b[20:] == 0x1234)
    np.testing.assert_array_equal(p16b[10:20], p16[10:20])


def test_scores_over_bf16_pooled_match_library_matmul():
    rng = np.random.default_rng(13)
    H, d, n_rows, n_q = 4, 32, 57, 3
    pooled = qsa_synth.to_bf16_bits(rng.standard_normal((n_rows, H * d)).astype(np.float32))
    q = rng.standard_normal((n_q, H * d)).astype(np.float32)
    s = oracle.scores(q, pooled, n_rows, H, d, 0.25)
    ref = 0.25 * (q.astype(np.float64) @ qsa_synth.bf16_bits_to_f32(pooled).astype(np.float64).T)
    np.testing.assert_allclose(s, ref, rtol=1e-12, atol=1e-12)


def _multi_case(n_ctx, n_q, seed, store="f32"):
    shape = qsa_synth.shrink(qsa_synth.CONFIGS["tiny_f32_decode"], n_ctx=n_ctx)
    inp = qsa_synth.decode_inputs(shape, seed=seed, n_steps=n_q)
    pooled = np.zeros((shape.n_rows, shape.H_idx * shape.d_idx),
                      np.uint16 if store == "bf16" else np.float32)
    return shape, inp, pooled


@pytest.mark.parametrize("n_ctx,n_q", [(2050, 3), (2051, 2), (2052, 4), (2053, 3), (90, 3)])
@pytest.mark.parametrize("store", ["f32", "bf16"])
def test_multi_query_step_equals_one_query_steps_at_each_position(n_ctx, n_q, store):
    shape, inp, pooled = _multi_case(n_ctx, n_q, seed=21 + n_ctx, store=store)
    res, s = oracle.decode_step_multi(
        inp["raw_k"], n_ctx, shape.H_idx, shape.d_idx, inp["norm_w"], shape.eps,
        shape.rope_base, pooled, 0, inp["q_idx"], shape.top_k_tokens, inp["q"], inp["K"],
        inp["V"], shape.H_q, shape.H_kv, shape.d)
    assert s.shape == (n_q, shape.n_rows)
    for i in range(n_q):
        p = n_ctx - n_q + i
        ref_pooled = np.zeros_like(pooled)
        b1, c1, o1, l1, _ = oracle.decode_step(
            inp["raw_k"], p + 1, shape.H_idx, shape.d_idx, inp["norm_w"], shape.eps,
            shape.rope_base, ref_pooled, 0, inp["q_idx"][i], shape.top_k_tokens, inp["q"][i],
            inp["K"], inp["V"], shape.H_q, shape.H_kv, shape.d)
        blocks, cl, out, lse = res[i]
        np.testing.assert_array_equal(blocks, b1)
        np.testing.assert_array_equal(cl, c1)
        np.testing.assert_array_equal(out, o1)
        np.testing.assert_array_equal(lse, l1)
        assert len(cl) == 4 * len(blocks) + (p + 1) % 4 and cl.max() <= p
        if (p + 1) % 4:
            assert cl[-1] == p
        # every row is scored for every query; the ones complete at p agree with the
        # one-query step's scores
        n_i = (p + 1) // 4
        ref_s = oracle.scores(inp["q_idx"][i], ref_pooled, n_i, shape.H_idx, shape.d_idx,
                              1.0 / np.sqrt(shape.d_idx))[0]
        np.testing.assert_array_equal(s[i, :n_i], ref_s)
        assert np.all(np.isfinite(s[i]))


def test_multi_query_single_query_is_the_decode_step():
    shape, inp, pooled = _multi_case(2050, 1, seed=3)
    res, s = oracle.decode_step_multi(
        inp["raw_k"], 2050, shape.H_idx, shape.d_idx, inp["norm_w"], shape.eps,
        shape.rope_base, pooled, 0, inp["q_idx"], shape.top_k_tokens, inp["q"], inp["K"],
        inp["V"], shape.H_q, shape.H_kv, shape.d)
    pooled2 = np.zeros_like(pooled)
    b, c, o, l, s1 = oracle.decode_step(
        inp["raw_k"], 2050, shape.H_idx, shape.d_idx, inp["norm_w"], shape.eps,
        shape.rope_base, pooled2, 0, inp["q_idx"][0], shape.top_k_tokens, inp["q"][0],
        inp["K"], inp["V"], shape.H_q, shape.H_kv, shape.d)
    np.testing.assert_array_equal(res[0][0], b)
    np.testing.assert_array_equal(res[0][1], c)
    np.testing.assert_array_equal(res[0][2], o)
    np.testing.assert_array_equal(res[0][3], l)
    np.testing.assert_array_equal(s[0], s1)
