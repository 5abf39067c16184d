"""Pins of the oracle's pooled-key steps: pooling, RMS norm, RoPE and their composition.

Each test checks the oracle against something other than itself: exact arithmetic on
integer-valued keys, closed forms, the textbook 2-D rotation, group properties of
rotations, and a hand-worked example stored under tests/golden/.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import oracle
import qsa_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _eval(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"sqrt": math.sqrt, "cos": math.cos,
                                                   "sin": math.sin}))


# ------------------------------------------------------------------ pooling

@pytest.mark.parametrize("store", ["f32", "bf16"])
def test_pool_mean_is_exact_mean_of_present_tokens(store):
    H, d = 2, 4
    n_ctx = 6  # block 0 = tokens 0..3, block 1 = tokens 4..5 (open block, 2 tokens)
    t = np.arange(n_ctx, dtype=np.float32)[:, None, None]
    e = np.arange(H * d, dtype=np.float32).reshape(1, H, d)
    raw = 10.0 * t + e  # small integers: exact in fp32 and in bf16
    raw = qsa_synth.to_bf16_bits(raw) if store == "bf16" else raw.astype(np.float32)
    p0, c0 = oracle.pool_mean(raw, n_ctx, H, d, 0)
    p1, c1 = oracle.pool_mean(raw, n_ctx, H, d, 1)
    assert c0 == 4 and c1 == 2
    # tokens 0..3: 10*(0+1+2+3)/4 + e = 15 + e ; tokens 4,5: 10*(4+5)/2 + e = 45 + e
    np.testing.assert_array_equal(p0, 15.0 + np.arange(H * d))
    np.testing.assert_array_equal(p1, 45.0 + np.arange(H * d))


def test_pool_mean_single_present_token_is_that_token():
    H, d = 1, 8
    raw = np.random.default_rng(1).standard_normal((9, H, d)).astype(np.float32)
    p, c = oracle.pool_mean(raw, 9, H, d, 2)  # block 2 holds only token 8
    assert c == 1
    np.testing.assert_array_equal(p, raw[8].reshape(-1).astype(np.float64))


# ------------------------------------------------------------------ RMS norm

def test_rmsnorm_unit_rms_without_eps_and_weight():
    p = np.random.default_rng(2).standard_normal(128)
    y = oracle.rmsnorm(p, np.ones(128, np.float32), 0.0)
    assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-14


def test_rmsnorm_rms_before_weight_closed_form():
    """rms(y / w) = sqrt(ms / (ms + eps)) for any p, eps and nonzero w."""
    rng = np.random.default_rng(3)
    p = rng.standard_normal(64) * 0.01
    w = (1.0 + 0.1 * rng.standard_normal(64)).astype(np.float32)
    eps = 1e-6
    y = oracle.rmsnorm(p, w, eps)
    ms = np.mean(p * p)
    got = math.sqrt(np.mean((y / w.astype(np.float64)) ** 2))
    assert abs(got - math.sqrt(ms / (ms + eps))) < 1e-14


def test_rmsnorm_constant_vector_with_eps():
    # p = c everywhere: y = c / sqrt(c^2 + eps) * w ; c = 1e-3, eps = 1e-6 -> 1/sqrt(2)
    y = oracle.rmsnorm(np.full(16, 1e-3), np.full(16, 2.0, np.float32), 1e-6)
    np.testing.assert_allclose(y, 2.0 / math.sqrt(2.0), rtol=1e-14)


def test_rmsnorm_weight_is_elementwise():
    y = oracle.rmsnorm(np.array([3.0, 4.0]), np.array([2.0, 0.5], np.float32), 0.0)
    np.testing.assert_allclose(y, [6.0 / math.sqrt(12.5), 2.0 / math.sqrt(12.5)], rtol=1e-15)


# ------------------------------------------------------------------ RoPE

def test_rope_position_zero_is_identity():
    x = np.random.default_rng(4).standard_normal(128)
    np.testing.assert_array_equal(oracle.rope(x, 0.0, 10000.0), x)


@pytest.mark.parametrize("phi", [0.3, 1.0, 2.5, -0.7, 100.0])
def test_rope_d2_is_textbook_rotation(phi):
    # d = 2: theta_0 = base^0 = 1, so position phi rotates by phi radians, counter-clockwise
    np.testing.assert_allclose(oracle.rope(np.array([1.0, 0.0]), phi, 10000.0),
                               [math.cos(phi), math.sin(phi)], atol=1e-15)
    np.testing.assert_allclose(oracle.rope(np.array([0.0, 1.0]), phi, 10000.0),
                               [-math.sin(phi), math.cos(phi)], atol=1e-15)


def test_rope_frequency_and_half_split_pairing():
    # d = 4, base = 100: theta_1 = 100^(-2/4) = 0.1; dim 1 pairs with dim 3 (i + d/2)
    e1 = np.array([0.0, 1.0, 0.0, 0.0])
    np.testing.assert_allclose(oracle.rope(e1, 10.0, 100.0), [0.0, math.cos(1.0), 0.0,
                                                              math.sin(1.0)], atol=1e-15)
    # dim 0 pairs with dim 2 at theta_0 = 1
    e0 = np.array([1.0, 0.0, 0.0, 0.0])
    np.testing.assert_allclose(oracle.rope(e0, 10.0, 100.0), [math.cos(10.0), 0.0,
                                                              math.sin(10.0), 0.0], atol=1e-15)


def test_rope_preserves_each_pair_norm():
    d = 128
    x = np.random.default_rng(5).standard_normal(d)
    y = oracle.rope(x, 255180.0, 10000.0)
    half = d // 2
    np.testing.assert_allclose(x[:half] ** 2 + x[half:] ** 2, y[:half] ** 2 + y[half:] ** 2,
                               rtol=1e-12)


def test_rope_composes_additively():
    x = np.random.default_rng(6).standard_normal(64)
    a, b = 1234.0, 56789.0
    np.testing.assert_allclose(oracle.rope(oracle.rope(x, a, 10000.0), b, 10000.0),
                               oracle.rope(x, a + b, 10000.0), atol=1e-9)


def test_rope_dot_depends_only_on_relative_position():
    rng = np.random.default_rng(7)
    x, y = rng.standard_normal(128), rng.standard_normal(128)
    m, n, t = 40.0, 12.0, 99991.0
    lhs = oracle.rope(x, m, 10000.0) @ oracle.rope(y, n, 10000.0)
    rhs = oracle.rope(x, m + t, 10000.0) @ oracle.rope(y, n + t, 10000.0)
    assert abs(lhs - rhs) < 1e-9


# ------------------------------------------------------------------ composition

def test_pool_rows_hand_worked_example():
    with open(os.path.join(GOLDEN, "pool_worked_example.json")) as f:
        g = json.load(f)
    raw = np.array(g["tokens"], np.float32).reshape(g["n_ctx"], g["H"], g["d"])
    w = np.array(g["norm_w"], np.float32)
    rows = oracle.pool_rows(raw, g["n_ctx"], g["H"], g["d"], w, g["eps"], g["rope_base"],
                            0, 3)
    want = np.array([[_eval(e) for e in r] for r in g["expected_rows"]])
    np.testing.assert_allclose(rows, want, rtol=0, atol=2e-7)  # fp32 storage
    # the fp64 row before storage matches to rounding of the closed form
    for b in range(3):
        z = oracle.pool_row_f64(raw, g["n_ctx"], g["H"], g["d"], w, g["eps"],
                                g["rope_base"], b)
        np.testing.assert_allclose(z, want[b], atol=1e-14)


def test_pool_row_order_is_pool_then_norm_then_rope():
    """With a non-uniform weight, RMS norm and RoPE do not commute and pooling does not
    commute with RMS norm: the row must equal RoPE(RMS(mean)) at position 4b."""
    rng = np.random.default_rng(8)
    H, d, n_ctx = 3, 16, 23
    raw = rng.standard_normal((n_ctx, H, d)).astype(np.float32)
    w = (1.0 + 0.3 * rng.standard_normal(d)).astype(np.float32)
    for b in (0, 1, 4, 5):  # block 5 is the open block (tokens 20..22)
        z = oracle.pool_row_f64(raw, n_ctx, H, d, w, 1e-6, 10000.0, b)
        p, _ = oracle.pool_mean(raw, n_ctx, H, d, b)
        for h in range(H):
            y = oracle.rmsnorm(p[h * d:(h + 1) * d], w, 1e-6)
            np.testing.assert_allclose(z[h * d:(h + 1) * d], oracle.rope(y, 4.0 * b, 1e4),
                                       atol=1e-14)
        # the other orders give different vectors
        alt = oracle.rmsnorm(oracle.rope(p[:d], 4.0 * b, 1e4), w, 1e-6)
        if b > 0:
            assert np.max(np.abs(alt - z[:d])) > 1e-3


def test_pool_rows_store_fp32_rounding_and_touch_only_requested_rows():
    rng = np.random.default_rng(9)
    H, d, n_ctx = 2, 8, 30
    raw = qsa_synth.to_bf16_bits(rng.standard_normal((n_ctx, H, d)).astype(np.float32))
    w = np.ones(d, np.float32)
    pooled = np.full((8, H * d), 7.0, np.float32)
    oracle.pool_rows(raw, n_ctx, H, d, w, 1e-6, 1e4, 3, 6, pooled)
    for b in range(8):
        if 3 <= b < 6:
            z = oracle.pool_row_f64(raw, n_ctx, H, d, w, 1e-6, 1e4, b)
            np.testing.assert_array_equal(pooled[b], z.astype(np.float32))
        else:
            assert np.all(pooled[b] == 7.0)


def test_incremental_cache_equals_full_rebuild():
    """The incremental update (recompute only rows from the first invalid block) gives
    the same cache as rebuilding every row after each appended token."""
    rng = np.random.default_rng(10)
    H, d = 2, 8
    n_end = 41
    raw = rng.standard_normal((n_end, H, d)).astype(np.float32)
    w = (1.0 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    n_ctx = 17
    cache = oracle.pool_rows(raw, n_ctx, H, d, w, 1e-6, 1e4, 0, (n_ctx + 3) // 4,
                             np.zeros((11, H * d), np.float32))
    while n_ctx < n_end:
        n_valid_full = n_ctx // 4   # rows of complete blocks stay valid
        n_ctx += 1
        oracle.pool_rows(raw, n_ctx, H, d, w, 1e-6, 1e4, n_valid_full, (n_ctx + 3) // 4, cache)
        full = oracle.pool_rows(raw, n_ctx, H, d, w, 1e-6, 1e4, 0, (n_ctx + 3) // 4,
                                np.zeros((11, H * d), np.float32))
        np.testing.assert_array_equal(cache[:(n_ctx + 3) // 4], full[:(n_ctx + 3) // 4])
