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


def _run_pair(dtype, H_q, H_kv, d, n_ctx, k_blks, tol):
    """Two calls in a row (cell lists of k_blks[0] and k_blks[1] blocks, each with its own
    capacity 4*k_blk + 3 and so its own split count), first through qsa_sparse_attn with a
    caller workspace, then through the entry point under test with no synchronisation
    between its two calls; the outputs and log-sum-exps must agree."""
    fn = _entry()
    rng = np.random.default_rng(2024 + H_q + 7 * H_kv)
    scale = 1.0 / math.sqrt(d)

    def store(x):
        return qsa_synth.to_bf16_bits(x) if dtype == "bf16" else x

    K = to_dev(store(rng.standard_normal((n_ctx, H_kv, d)).astype(np.float32)))
    V = to_dev(store(rng.standard_normal((n_ctx, H_kv, d)).astype(np.float32)))
    cases = []
    for k_blk in k_blks:  # two different queries and cell lists
        max_cells = 4 * k_blk + 3
        pos, n = _cells(rng, n_ctx, k_blk, max_cells)
        q = rng.standard_normal((1, H_q, d)).astype(np.float32)
        cases.append((to_dev(q), to_dev(pos), to_dev(n), max_cells))
    # reference: the existing entry point with a caller workspace
    want = []
    for q, pos, n, max_cells in cases:
        ws_bytes = qsa.sparse_attn_workspace_size(1, H_q, H_kv, d, max_cells)
        assert ws_bytes <= 4 << 20
        ws = torch.empty(max(ws_bytes // 4, 1), device="cuda")
        out = torch.empty(1, H_q, d, device="cuda")
        lse = torch.empty(1, H_q, device="cuda")
        qsa.sparse_attn(q, K, V, n, max_cells, out, H_kv, d, d, scale, pos=pos, lse=lse,
                        workspace=ws)
        want.append((to_host(out), to_host(lse)))
    # the entry point under test, called twice in a row through the C ABI
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dt = 1 if dtype == "bf16" else 0
    got = []
    for q, pos, n, max_cells in cases:
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


def _splits(H_q, H_kv, d, k_blk):
    """Split count of a one-query call, read off the (upper-bound) workspace size: 0 bytes
    means one split, otherwise one partial record of (d + 4) floats per head and split."""
    ws = qsa.sparse_attn_workspace_size(1, H_q, H_kv, d, 4 * k_blk + 3)
    return ws // (4 * H_q * (d + 4)) if ws else 1


def test_noalloc_matches_workspace_call_fp32_split_k():
    """fp32 K/V, 4 query heads per KV head: the general kernel writes its split-K partial
    records into the fixed scratch and the combine kernel reads them back."""
    assert _splits(8, 2, 128, 16) > 1
    _run_pair("f32", 8, 2, 128, 2050, (16, 16), ATOL_ATTN_F32)


def test_noalloc_bf16_split_k_more_splits_then_fewer():
    """bf16 K/V with 4 query heads per KV head (16 / 4 heads) also takes the kernel whose
    splits meet in the scratch.  The first call uses more splits than the second, so the
    second runs over records the first left behind."""
    s0, s1 = _splits(16, 4, 128, 512), _splits(16, 4, 128, 64)
    assert s0 > s1 > 1
    _run_pair("bf16", 16, 4, 128, 61789, (512, 64), ATOL_ATTN_BF16)


def test_noalloc_matches_workspace_call_bf16_decode():
    """The 61,789-token decode shape (32 / 4 heads, 2,051 cells), whose kernel merges its
    splits inside a thread-block cluster and leaves the scratch untouched."""
    _run_pair("bf16", 32, 4, 128, 61789, (512, 512), ATOL_ATTN_BF16)


def test_noalloc_latent_shape_needs_no_scratch():
    """Four latent-shape queries (16 heads on one KV head, DKQ 576, d_v 512, V = K[:, :512])
    over 2,048 listed keys: the shape-only workspace bound is above the fixed array, but the
    kernel merges its splits in a cluster, so the call is accepted and equals the
    workspace call."""
    n_q, H_q, n_kv, max_list = 4, 16, 4096, 2048
    assert qsa.sparse_attn_workspace_size(n_q, H_q, 1, 512, max_list) > 4 << 20
    fn = _entry()
    rng = np.random.default_rng(576)
    kv = to_dev(qsa_synth.to_bf16_bits(rng.standard_normal((n_kv, 576)).astype(np.float32)))
    q = to_dev(rng.standard_normal((n_q, H_q, 576)).astype(np.float32))
    pos = to_dev(np.stack([np.sort(rng.choice(n_kv, max_list, replace=False))
                           for _ in range(n_q)]).astype(np.int32))
    n = to_dev(np.array([max_list, 1500, 7, 0], np.int32))
    scale = 1.0 / math.sqrt(576)
    want = torch.empty(n_q, H_q, 512, device="cuda")
    ws = torch.empty(qsa.sparse_attn_workspace_size(n_q, H_q, 1, 512, max_list) // 4,
                     device="cuda")
    qsa.sparse_attn(q, kv, kv, n, max_list, want, 1, 576, 512, scale, pos=pos, workspace=ws,
                    ld_k=576, ld_v=576)
    got = torch.full((n_q, H_q, 512), float("nan"), device="cuda")
    st = fn(q.data_ptr(), n_q, H_q, 1, 576, 512, scale, kv.data_ptr(), kv.data_ptr(), 1, n_kv,
            576, 576, pos.data_ptr(), n.data_ptr(), max_list, got.data_ptr(), None,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, qsa.status_str(st)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_host(got), to_host(want), rtol=0, atol=ATOL_ATTN_BF16)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """Eight queries of 16 heads on one KV head with d 256 (bf16, not the latent shape, so
    the general kernel's partial records): 4.26 MB of scratch, above the fixed 4 MiB."""
    fn = _entry()
    n_q, H_q, d, max_list = 8, 16, 256, 2048
    need = qsa.sparse_attn_workspace_size(n_q, H_q, 1, d, max_list)
    assert need > 4 << 20
    q = torch.zeros(n_q, H_q, d, device="cuda")
    k = torch.zeros(4096, d, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(4096, d, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(n_q, max_list, dtype=torch.int32, device="cuda")
    n = torch.zeros(n_q, dtype=torch.int32, device="cuda")
    out = torch.zeros(n_q, H_q, d, device="cuda")
    st = fn(q.data_ptr(), n_q, H_q, 1, d, d, 0.0625, k.data_ptr(), v.data_ptr(), 1, 4096, d, d,
            pos.data_ptr(), n.data_ptr(), max_list, out.data_ptr(), None,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert qsa.status_str(st) == "QSA_ERR_UNSUPPORTED"
