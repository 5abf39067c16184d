"""Python face of the fp64 CPU oracle (``qsa_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's CPU
baseline are the only callers.  The CUDA library never imports this module and this
module never imports the CUDA library; the two share only the seeded input generator,
which holds none of the method's arithmetic.

The C file is compiled with gcc on first use (``-O2 -ffp-contract=off`` so that no
multiply-add is fused and the fp64 results are the same on x86-64 and AArch64).

Each function restates one step of QSA two-stage sparse attention as the source pages
describe it (Qiita, ariera, EVO-X2 llama.cpp series part 10, "QSA and the QSA
indexer", "incremental pooled-key cache (COMMON-004)", "selected K/V gather
(COMMON-005)", "block-domain top-k (COMMON-006)"; devotd.net, "llama.cpp CDNA sparse
attention", sections 2-3).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int
_d = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (plain gcc, no GPU)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        sig = {
            "oracle_round_bf16": (ctypes.c_float, [ctypes.c_float]),
            "oracle_bf16_bits_from_f64": (ctypes.c_uint16, [_d]),
            "oracle_pool_mean": (_i32, [_p, _i32, _i64, _i32, _i32, _i64, _p]),
            "oracle_rmsnorm": (None, [_p, _i32, _p, _d, _p]),
            "oracle_rope": (None, [_p, _i32, _d, _d]),
            "oracle_pool_row_f64": (None, [_p, _i32, _i64, _i32, _i32, _p, _d, _d, _i64, _p]),
            "oracle_pool_rows": (None, [_p, _i32, _i64, _i32, _i32, _p, _d, _d, _i64, _i64, _i32,
                                        _p]),
            "oracle_scores": (None, [_p, _i64, _p, _i32, _i64, _i32, _i32, _d, _p, _i32, _p]),
            "oracle_topk": (_i64, [_p, _i64, _i64, _p]),
            "oracle_cells": (_i64, [_p, _i64, _i64, _p]),
            "oracle_expand_block_scores": (None, [_p, _i64, _p]),
            "oracle_get_rows": (None, [_p, _i32, _i64, _i64, _p, _i64, _p]),
            "oracle_attention": (None, [_p, _i32, _i32, _i32, _i32, _p, _p, _i32, _i64, _i64,
                                        _p, _i64, _d, _p, _p]),
            "oracle_mask_to_list": (_i64, [_p, _i64, _i64, _p, _p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _raw_dtype(a: np.ndarray) -> int:
    """fp32 arrays are fp32; uint16 arrays hold bf16 bit patterns."""
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle inputs are float32 or bf16 bits (uint16), got {a.dtype}")


# ----------------------------------------------------------------------------- pieces

def round_bf16(x: float) -> float:
    return float(_load().oracle_round_bf16(ctypes.c_float(x)))


def bf16_bits_from_f64(x: float) -> int:
    """Bit pattern of the bf16 value nearest to the fp64 value x (ties to even)."""
    return int(_load().oracle_bf16_bits_from_f64(float(x)))


def pool_mean(raw: np.ndarray, n_ctx: int, H: int, d: int, b: int):
    """Mean of the present raw indexer keys of block b; returns (p [H*d] f64, count)."""
    raw = np.ascontiguousarray(raw)
    p = np.zeros(H * d, np.float64)
    c = _load().oracle_pool_mean(_ptr(raw), _raw_dtype(raw), n_ctx, H, d, b, _ptr(p))
    return p, int(c)


def rmsnorm(p: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    p = _c(p, np.float64)
    w = _c(w, np.float32)
    y = np.zeros_like(p)
    _load().oracle_rmsnorm(_ptr(p), p.shape[0], _ptr(w), eps, _ptr(y))
    return y


def rope(y: np.ndarray, pos: float, base: float) -> np.ndarray:
    y = _c(y, np.float64).copy()
    _load().oracle_rope(_ptr(y), y.shape[0], float(pos), float(base))
    return y


def pool_row_f64(raw, n_ctx, H, d, w, eps, base, b) -> np.ndarray:
    raw = np.ascontiguousarray(raw)
    w = _c(w, np.float32)
    z = np.zeros(H * d, np.float64)
    _load().oracle_pool_row_f64(_ptr(raw), _raw_dtype(raw), n_ctx, H, d, _ptr(w), eps, base,
                                b, _ptr(z))
    return z


def pool_rows(raw, n_ctx, H, d, w, eps, base, row_begin, row_end, pooled=None, store="f32"):
    """Recompute pooled-cache rows [row_begin, row_end) into ``pooled``: an fp32 array, or
    a uint16 array of bf16 bit patterns (``store="bf16"`` when a new one is made)."""
    raw = np.ascontiguousarray(raw)
    w = _c(w, np.float32)
    if pooled is None:
        pooled = np.zeros((row_end, H * d), np.uint16 if store == "bf16" else np.float32)
    assert pooled.flags.c_contiguous
    assert pooled.shape[0] >= row_end and pooled.shape[1] == H * d
    _load().oracle_pool_rows(_ptr(raw), _raw_dtype(raw), n_ctx, H, d, _ptr(w), eps, base,
                             row_begin, row_end, _raw_dtype(pooled), _ptr(pooled))
    return pooled


def scores(q, pooled, n_rows, H, d, scale, q_pos=None, round_bf16_operands=False):
    """Index scores [n_q][n_rows] in fp64 (pooled: fp32, or uint16 bf16 bit patterns)."""
    q = _c(q, np.float32).reshape(-1, H * d)
    pooled = np.ascontiguousarray(pooled).reshape(-1, H * d)
    assert pooled.shape[0] >= n_rows
    n_q = q.shape[0]
    out = np.zeros((n_q, n_rows), np.float64)
    qp = None if q_pos is None else _c(q_pos, np.int32)
    _load().oracle_scores(_ptr(q), n_q, _ptr(pooled), _raw_dtype(pooled), n_rows, H, d, scale,
                          None if qp is None else _ptr(qp), int(bool(round_bf16_operands)),
                          _ptr(out))
    return out


def topk(score_row, n_full, k_blk) -> np.ndarray:
    """Ascending block indices of the k_blk best full blocks (ties -> lower index)."""
    s = _c(score_row, np.float64)
    assert s.shape[0] >= n_full
    out = np.zeros(max(min(k_blk, n_full), 1), np.int32)
    k = _load().oracle_topk(_ptr(s), n_full, k_blk, _ptr(out))
    return out[:k].copy()


def expand_block_scores(score_row, n_full) -> np.ndarray:
    """Each full block's score copied to its 4 cells (the selection path before the block
    domain): [4*n_full] fp64."""
    s = _c(score_row, np.float64)
    assert s.shape[0] >= n_full
    out = np.zeros(max(4 * n_full, 1), np.float64)
    _load().oracle_expand_block_scores(_ptr(s), n_full, _ptr(out))
    return out[:4 * n_full].copy()


def cells(blocks, p) -> np.ndarray:
    """Cells of the selected blocks, then the tail 4*floor((p+1)/4) .. p."""
    blocks = _c(blocks, np.int32)
    out = np.zeros(4 * blocks.shape[0] + 4, np.int32)
    n = _load().oracle_cells(_ptr(blocks), blocks.shape[0], int(p), _ptr(out))
    return out[:n].copy()


def get_rows(src: np.ndarray, row_elems: int, ld: int, cell_list) -> np.ndarray:
    src = np.ascontiguousarray(src)
    cl = _c(cell_list, np.int32)
    dst = np.zeros(cl.shape[0] * row_elems, src.dtype)
    _load().oracle_get_rows(_ptr(src), src.dtype.itemsize, row_elems, ld, _ptr(cl),
                            cl.shape[0], _ptr(dst))
    return dst.reshape(cl.shape[0], row_elems)


def attention(q, K, V, H_q, H_kv, d_k, d_v, ld_k, ld_v, cell_list, scale):
    """Attention of one query token over the listed cells; returns (out f64, lse f64)."""
    q = _c(q, np.float32).reshape(H_q, d_k)
    K = np.ascontiguousarray(K)
    V = np.ascontiguousarray(V)
    dt = _raw_dtype(K)
    assert _raw_dtype(V) == dt
    cl = _c(cell_list, np.int32)
    out = np.zeros((H_q, d_v), np.float64)
    lse = np.zeros(H_q, np.float64)
    _load().oracle_attention(_ptr(q), H_q, H_kv, d_k, d_v, _ptr(K), _ptr(V), dt, ld_k, ld_v,
                             _ptr(cl), cl.shape[0], scale, _ptr(out), _ptr(lse))
    return out, lse


def mask_to_list(mask_row, max_list):
    """(positions[:min(count, max_list)], true count, 64-bit words)."""
    m = _c(mask_row, np.uint8)
    n_kv = m.shape[0]
    pos = np.zeros(max(max_list, 1), np.int32)
    bits = np.zeros((n_kv + 63) // 64, np.uint64)
    cnt = _load().oracle_mask_to_list(_ptr(m), n_kv, max_list, _ptr(pos), _ptr(bits))
    return pos[:min(cnt, max_list)].copy(), int(cnt), bits


# ----------------------------------------------------------------------- composites

def decode_step(raw_k, n_ctx, H_idx, d_idx, w, eps, base, pooled, n_valid_full,
                q_idx, top_k_tokens, q, K, V, H_q, H_kv, d, kv_dtype_ld=None):
    """One decode step of one QSA layer, in the pages' order.

    Updates ``pooled`` rows [n_valid_full, n_rows) in place, scores every row, takes
    the block-domain top-k over full blocks, expands to cells plus the open tail and
    attends over those cells.  Returns (blocks, cells, out [H_q][d] f64, lse, scores).
    """
    n_full = n_ctx // 4
    n_rows = (n_ctx + 3) // 4
    pool_rows(raw_k, n_ctx, H_idx, d_idx, w, eps, base, n_valid_full, n_rows, pooled)
    s = scores(q_idx, pooled, n_rows, H_idx, d_idx, 1.0 / np.sqrt(d_idx))[0]
    blocks = topk(s, n_full, top_k_tokens // 4)
    cl = cells(blocks, n_ctx - 1)
    ld = H_kv * d if kv_dtype_ld is None else kv_dtype_ld
    out, lse = attention(q, K, V, H_q, H_kv, d, d, ld, ld, cl, 1.0 / np.sqrt(d))
    return blocks, cl, out, lse, s


def decode_step_multi(raw_k, n_ctx, H_idx, d_idx, w, eps, base, pooled, n_valid_full,
                      q_idx, top_k_tokens, q, K, V, H_q, H_kv, d):
    """A decode step for n_q query tokens at once: the last n_q tokens of the context,
    positions n_ctx - n_q .. n_ctx - 1 (a token and the draft tokens that follow it,
    verified together), sharing one pooled-cache update.

    Every query scores every pooled row (as the one-query step does), but query i at
    position p_i = n_ctx - n_q + i only selects among what is causal for it: the blocks
    complete at p_i (b < floor((p_i+1)/4)) compete in its top-k, and its tail is
    4*floor((p_i+1)/4) .. p_i.  Returns per-query lists (blocks, cells, out, lse) and
    the score matrix [n_q][n_rows].
    """
    q_idx = _c(q_idx, np.float32).reshape(-1, H_idx * d_idx)
    n_q = q_idx.shape[0]
    q = _c(q, np.float32).reshape(n_q, H_q, d)
    n_full = n_ctx // 4
    n_rows = (n_ctx + 3) // 4
    pool_rows(raw_k, n_ctx, H_idx, d_idx, w, eps, base, n_valid_full, n_rows, pooled)
    q_pos = np.arange(n_ctx - n_q, n_ctx, dtype=np.int32)
    s = scores(q_idx, pooled, n_rows, H_idx, d_idx, 1.0 / np.sqrt(d_idx))
    res = []
    for i in range(n_q):
        p = int(q_pos[i])
        blocks = topk(s[i], min(n_full, (p + 1) // 4), top_k_tokens // 4)
        cl = cells(blocks, p)
        out, lse = attention(q[i], K, V, H_q, H_kv, d, d, H_kv * d, H_kv * d, cl,
                             1.0 / np.sqrt(d))
        res.append((blocks, cl, out, lse))
    return res, s
