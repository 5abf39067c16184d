"""qsa_sparse_attn_noalloc: sparse attention for callers that cannot allocate device
memory (for instance a plugin whose host framework owns every device allocation, or a
real-time loop that may not risk a cudaMalloc).  It keeps its split-K scratch in a fixed
array inside the library instead of a caller workspace.  Checked here, through the C ABI,
against qsa_sparse_attn with a caller workspace on two calls in a row, and for its size
limit.  This file is collected last on purpose."""
import ctypes
import math

import numpy as np
import pytest
import torch

import gather_qsa_pool_gb300 as qsa
import qsa_synth
from gpu_helpers import ATOL_ATTN_BF16, ATOL_ATTN_F32, to_dev, to_host
from oracle import oracle

pytestmark = pytest.mark.gpu

_p, _i64, _int, _f = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float


def _entry():
    fn = qsa.load().qsa_sparse_attn_noalloc
    fn.restype = _int
    fn.argtypes = [_p, _i64, _int, _int, _int, _int, _f, _p, _p, _int, _i64, _i64, _i64, _p, _p,
                   _i64, _p, _p, _p]
    return fn


def _cells(rng, n_ctx, k_blk, max_cells):
    blocks = np.sort(rng.choice(n_ctx // 4, k_blk, replace=False)).astype(np.int32)
    cl = oracle.cells(blocks, n_ctx - 1)
    pos = np.full((1, max_cells), -1, np.int32)
    pos[0, :cl.shape[0]] = cl
    return pos, np.array([cl.shape[0]], np.int32)


def _compare_two_calls(dtype, H_q, H_kv, d, n_ctx, k_blk, tol):
    fn = _entry()
    rng = np.random.default_rng(2024 + H_q)
    max_cells = 4 * k_blk + 3
    scale = 1.0 / math.sqrt(d)

    def store(x):
        return qsa_synth.to_bf16_bits(x) if dtype == "bf16" else x

    K = to_dev(store(rng.standard_normal((n_ctx, H_kv, d)).astype(np.float32)))
    V = to_dev(store(rng.standard_normal((n_ctx, H_kv, d)).astype(np.float32)))
    cases = []
    for _ in range(2):  # two different queries and cell lists
        pos, n = _cells(rng, n_ctx, k_blk, max_cells)
        q = rng.standard_normal((1, H_q, d)).astype(np.float32)
        cases.append((to_dev(q), to_dev(pos), to_dev(n)))
    # reference: the existing entry point with a caller workspace
    ws_bytes = qsa.sparse_attn_workspace_size(1, H_q, H_kv, d, max_cells)
    assert 0 < ws_bytes <= 4 << 20
    want = []
    for q, pos, n in cases:
        ws = torch.empty(ws_bytes // 4, device="cuda")
        out = torch.empty(1, H_q, d, device="cuda")
        lse = torch.empty(1, H_q, device="cuda")
        qsa.sparse_attn(q, K, V, n, max_cells, out, H_kv, d, d, scale, pos=pos, lse=lse,
                        workspace=ws)
        want.append((to_host(out), to_host(lse)))
    # the entry point under test, called twice in a row through the C ABI
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dt = 1 if dtype == "bf16" else 0
    got = []
    for q, pos, n in cases:
        out = torch.full((1, H_q, d), float("nan"), device="cuda")
        lse = torch.full((1, H_q), float("nan"), device="cuda")
        st = fn(q.data_ptr(), 1, H_q, H_kv, d, d, scale, K.data_ptr(), V.data_ptr(), dt, n_ctx,
                H_kv * d, H_kv * d, pos.data_ptr(), n.data_ptr(), max_cells, out.data_ptr(),
                lse.data_ptr(), stream)
        assert st == 0, qsa.status_str(st)
        got.append((out, lse))
    torch.cuda.synchronize()
    for (o, l), (wo, wl) in zip(got, want):
        np.testing.assert_allclose(to_host(o), wo, rtol=0, atol=tol)
        np.testing.assert_allclose(to_host(l), wl, rtol=1e-5, atol=1e-5)
    assert not np.allclose(want[0][0], want[1][0])  # the two calls really differ


def test_noalloc_matches_workspace_call_fp32_split_k():
    """fp32 K/V, 4 query heads per KV head: the split-K partials go through the scratch."""
    _compare_two_calls("f32", 8, 2, 128, 2050, 16, ATOL_ATTN_F32)


def test_noalloc_matches_workspace_call_bf16_decode():
    """The 61,789-token decode shape (32 / 4 heads, 2,051 cells)."""
    _compare_two_calls("bf16", 32, 4, 128, 61789, 512, ATOL_ATTN_BF16)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    fn = _entry()
    # 4 mask rows, 16 heads on one KV head, d_v 512, 2048 positions: 8.4 MB of scratch
    need = qsa.sparse_attn_workspace_size(4, 16, 1, 512, 2048)
    assert need > 4 << 20
    q = torch.zeros(4, 16, 576, device="cuda")
    kv = torch.zeros(4096, 576, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(4, 2048, dtype=torch.int32, device="cuda")
    n = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.zeros(4, 16, 512, device="cuda")
    st = fn(q.data_ptr(), 4, 16, 1, 576, 512, 0.05, kv.data_ptr(), kv.data_ptr(), 1, 4096, 576,
            576, pos.data_ptr(), n.data_ptr(), 2048, out.data_ptr(), None,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert qsa.status_str(st) == "QSA_ERR_UNSUPPORTED"
