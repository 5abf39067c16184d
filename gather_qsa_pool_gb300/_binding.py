"""ctypes binding of ``libqsa.so``: argument marshalling only.

Every function here has the name of the C entry point it calls (without the ``qsa_``
prefix), takes torch tensors that already live on the GPU, passes their data pointers,
sizes and the current CUDA stream, and raises :class:`QSAError` when the call returns a
non-OK status.  All computation happens in the library's CUDA kernels; there is no
fallback of any kind: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libqsa.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "qsa.h")

QSA_OK, QSA_ERR_INVALID_ARG, QSA_ERR_UNSUPPORTED, QSA_ERR_CUDA, QSA_ERR_TIMEOUT = range(5)
QSA_F32, QSA_BF16 = 0, 1
QSA_PREC_F32, QSA_PREC_BF16_TC = 0, 1
QSA_WAIT_DEFAULT_NS = 2_000_000_000

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_f = ctypes.c_float
_d = ctypes.c_double
_sz = ctypes.c_size_t

_SIGNATURES = {
    "qsa_status_str": (ctypes.c_char_p, [_int]),
    "qsa_version": (_int, []),
    "qsa_set_wait_options": (None, [_p, ctypes.c_uint64]),
    "qsa_pool_update": (_int, [_p, _int, _i64, _int, _int, _p, _f, _d, _p, _int, _i64, _i64,
                               _p]),
    "qsa_index_score": (_int, [_p, _i64, _i64, _p, _p, _int, _i64, _int, _int, _f, _p, _i64,
                               _int, _p, _sz, _p]),
    "qsa_index_score_workspace_size": (_sz, [_i64, _i64, _int, _int, _int, _int]),
    "qsa_topk_blocks": (_int, [_p, _i64, _i64, _p, _i64, _i64, _p, _p, _p]),
    "qsa_topk_max_candidates": (_i64, []),
    "qsa_index_score_maxima": (_int, [_p, _i64, _i64, _p, _p, _int, _i64, _int, _int, _f, _p,
                                      _i64, _p, _i64, _p, _sz, _p]),
    "qsa_topk_blocks_maxima": (_int, [_p, _i64, _i64, _p, _i64, _i64, _p, _i64, _p, _p, _p,
                                      _sz, _p]),
    "qsa_topk_blocks_maxima_workspace_size": (_sz, [_i64]),
    "qsa_expand_block_scores": (_int, [_p, _i64, _i64, _i64, _p, _i64, _p]),
    "qsa_gather_kv": (_int, [_p, _p, _int, _i64, _int, _int, _int, _i64, _i64, _p, _p, _i64,
                             _i64, _p, _i64, _p, _p, _p, _p, _i64, _p]),
    "qsa_sparse_attn": (_int, [_p, _i64, _int, _int, _int, _int, _f, _p, _p, _int, _i64, _i64,
                               _i64, _p, _p, _i64, _p, _p, _p, _sz, _p]),
    "qsa_sparse_attn_workspace_size": (_sz, [_i64, _int, _int, _int, _i64]),
    "qsa_sparse_attn_union": (_int, [_p, _i64, _int, _int, _int, _f, _p, _p, _int, _i64, _i64,
                                     _i64, _p, _p, _i64, _p, _p, _p, _sz, _p]),
    "qsa_sparse_attn_union_workspace_size": (_sz, [_i64, _i64]),
    "qsa_decode_step": (_int, [_p, _int, _i64, _int, _int, _p, _f, _d, _p, _int, _i64, _i64,
                               _i64, _p, _f, _p, _i64, _p, _p, _p, _p, _int, _i64, _int, _int,
                               _i64, _p, _p, _i64, _p, _int, _f, _p, _p, _p, _sz, _p]),
    "qsa_decode_step_workspace_size": (_sz, [_i64, _int, _int, _int, _i64, _i64]),
    "qsa_decode_step_host": (_int, [_p, _p, _p, _p, _int, _i64, _int, _int, _p, _f, _d, _p, _int,
                                    _i64, _i64, _i64, _f, _p, _i64, _p, _p, _p, _p, _int, _i64,
                                    _int, _int, _i64, _p, _p, _i64, _int, _f, _p, _p, _p, _sz,
                                    _p]),
    "qsa_decode_step_host_layout": (_sz, [_i64, _int, _int, _int, _int, _int, _int, _int, _p]),
    "qsa_decode_step_host_workspace_size": (_sz, [_i64, _int, _int, _int, _i64, _i64, _int, _int,
                                                  _int, _int]),
    "qsa_decode_plan_create": (_int, [ctypes.POINTER(_p), _p, _int, _int, _int, _p, _f, _d, _p,
                                      _int, _i64, _i64, _f, _p, _i64, _p, _p, _p, _p, _int, _i64,
                                      _int, _int, _i64, _p, _p, _i64, _int, _f, _p, _p, _p, _sz]),
    "qsa_decode_plan_destroy": (None, [_p]),
    "qsa_decode_plan_step": (_int, [_p, _i64, _i64, _i64, _p, _p, _p]),
    "qsa_decode_plan_step_host": (_int, [_p, _i64, _i64, _i64, _p, _p, _p, _p]),
    "qsa_mask_to_list": (_int, [_p, _i64, _i64, _i64, _i64, _p, _p, _p, _p]),
    "qsa_mask_sparse_eligible": (_int, [_int, _f, _f, _i64, _i64]),
    "qsa_mask_sparse_attn": (_int, [_p, _i64, _int, _int, _int, _int, _f, _p, _int, _i64, _i64,
                                    _p, _i64, _i64, _p, _p, _p, _p]),
}

_lib = None


class QSAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {status_str(status)}")


def header_functions() -> list[str]:
    """Names of every function that include/qsa.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(qsa_\w+)\s*\(", text, re.M)))


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library (building it first when its sources are newer)."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        from . import build as _build

        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"QSA CUDA library not found at {path}")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def set_wait_options(status=None, limit_ns=QSA_WAIT_DEFAULT_NS):
    """qsa_set_wait_options: for later launches from this thread, the int32 device tensor a
    kernel whose bounded wait gave up stores QSA_ERR_TIMEOUT into (or None), and the limit of
    the waits inside a kernel's pipeline (0: give up unless already complete)."""
    load().qsa_set_wait_options(_ptr(status), int(limit_ns))


def status_str(status: int) -> str:
    return load().qsa_status_str(status).decode()


def _check(fn: str, status: int):
    if status != QSA_OK:
        raise QSAError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ld(t) -> int:
    """Element stride between rows of a row-major tensor (a single-row tensor may carry an
    arbitrary stride on its size-1 leading dim: use its row length)."""
    if t.dim() < 2 or t.shape[0] <= 1:
        return t[0].numel() if t.dim() >= 2 else t.numel()
    return t.stride(0)


def _dtype(t) -> int:
    import torch

    if t.dtype == torch.float32:
        return QSA_F32
    if t.dtype == torch.bfloat16:
        return QSA_BF16
    raise TypeError(f"QSA tensors are float32 or bfloat16, got {t.dtype}")


# --------------------------------------------------------------------------- entry points

def pool_update(raw_k, n_ctx, H, d, norm_w, eps, rope_base, pooled, n_valid_full, stream=None):
    """qsa_pool_update: recompute pooled rows [n_valid_full, ceil(n_ctx/4)) of a float32 or
    bfloat16 cache."""
    _check("qsa_pool_update", load().qsa_pool_update(
        _ptr(raw_k), _dtype(raw_k), n_ctx, H, d, _ptr(norm_w), eps, rope_base, _ptr(pooled),
        _dtype(pooled), pooled.shape[0], n_valid_full, _stream(stream)))


def index_score_workspace_size(n_q, n_rows, H, d, precision=QSA_PREC_F32,
                               pooled_dtype=QSA_F32) -> int:
    return int(load().qsa_index_score_workspace_size(n_q, n_rows, H, d, pooled_dtype,
                                                     precision))


def index_score(q, pooled, n_rows, H, d, scale, scores, q_pos=None, precision=QSA_PREC_F32,
                workspace=None, stream=None):
    """qsa_index_score: scores[i][b] for b < n_rows (q: [n_q][>= H*d] fp32; pooled float32
    or bfloat16)."""
    n_q = q.shape[0] if q.dim() > 1 else 1
    ld_q = _ld(q) if q.dim() > 1 else H * d
    ld_s = _ld(scores) if scores.dim() > 1 else n_rows
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("qsa_index_score", load().qsa_index_score(
        _ptr(q), n_q, ld_q, _ptr(q_pos), _ptr(pooled), _dtype(pooled), n_rows, H, d, scale,
        _ptr(scores), ld_s, precision, _ptr(workspace), ws_bytes, _stream(stream)))


def topk_max_candidates() -> int:
    return int(load().qsa_topk_max_candidates())


def topk_blocks(scores, n_full, k_blk, blocks_out, counts_out, q_pos=None, stream=None):
    """qsa_topk_blocks over the first n_full columns of each score row."""
    n_q = scores.shape[0] if scores.dim() > 1 else 1
    ld = _ld(scores)
    _check("qsa_topk_blocks", load().qsa_topk_blocks(
        _ptr(scores), n_q, ld, _ptr(q_pos), n_full, k_blk, _ptr(blocks_out), _ptr(counts_out),
        _stream(stream)))


def index_score_maxima(q, pooled, n_rows, H, d, scale, scores, maxima, q_pos=None,
                       workspace=None, stream=None):
    """qsa_index_score_maxima: the tensor-core scores plus maxima[i][g], the largest score of
    rows 32g .. 32g+31 of query i (maxima: [n_q][>= ceil(n_rows / 32)] fp32)."""
    n_q = q.shape[0] if q.dim() > 1 else 1
    ld_q = _ld(q) if q.dim() > 1 else H * d
    ld_s = _ld(scores) if scores.dim() > 1 else n_rows
    ld_m = _ld(maxima) if maxima.dim() > 1 else maxima.numel()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("qsa_index_score_maxima", load().qsa_index_score_maxima(
        _ptr(q), n_q, ld_q, _ptr(q_pos), _ptr(pooled), _dtype(pooled), n_rows, H, d, scale,
        _ptr(scores), ld_s, _ptr(maxima), ld_m, _ptr(workspace), ws_bytes, _stream(stream)))


def topk_blocks_maxima_workspace_size(n_q) -> int:
    return int(load().qsa_topk_blocks_maxima_workspace_size(n_q))


def topk_blocks_maxima(scores, maxima, n_full, k_blk, blocks_out, counts_out, workspace,
                       q_pos=None, stream=None):
    """qsa_topk_blocks_maxima: qsa_topk_blocks fed with the score kernel's group maxima
    (workspace: topk_blocks_maxima_workspace_size(n_q) bytes of device memory)."""
    n_q = scores.shape[0] if scores.dim() > 1 else 1
    ld = _ld(scores)
    ld_m = _ld(maxima) if maxima.dim() > 1 else maxima.numel()
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("qsa_topk_blocks_maxima", load().qsa_topk_blocks_maxima(
        _ptr(scores), n_q, ld, _ptr(q_pos), n_full, k_blk, _ptr(maxima), ld_m,
        _ptr(blocks_out), _ptr(counts_out), _ptr(workspace), ws_bytes, _stream(stream)))


def expand_block_scores(scores, n_full, cell_scores, stream=None):
    """qsa_expand_block_scores: cell_scores[i][c] = scores[i][c // 4] for c < 4*n_full."""
    n_q = scores.shape[0] if scores.dim() > 1 else 1
    ld_s = _ld(scores) if scores.dim() > 1 else scores.numel()
    ld_c = _ld(cell_scores) if cell_scores.dim() > 1 else cell_scores.numel()
    _check("qsa_expand_block_scores", load().qsa_expand_block_scores(
        _ptr(scores), n_q, ld_s, n_full, _ptr(cell_scores), ld_c, _stream(stream)))


def gather_kv(blocks, counts, k_blk, pos_out, n_cells_out, max_cells, n_ctx=-1, q_pos=None,
              K=None, V=None, K_out=None, V_out=None, H_kv=0, d_k=0, d_v=0, n_kv=None,
              stream=None):
    """qsa_gather_kv: cell positions (and compact K/V rows when K_out / V_out are given)."""
    n_q = counts.shape[0]
    dt = _dtype(K) if K is not None else QSA_BF16
    if n_kv is None:
        n_kv = K.shape[0] if K is not None else (1 << 62)
    ld_k = _ld(K) if K is not None else H_kv * d_k
    ld_v = _ld(V) if V is not None else H_kv * d_v
    _check("qsa_gather_kv", load().qsa_gather_kv(
        _ptr(K), _ptr(V), dt, n_kv, H_kv, d_k, d_v, ld_k, ld_v, _ptr(blocks), _ptr(counts), n_q,
        k_blk, _ptr(q_pos), n_ctx, _ptr(K_out), _ptr(V_out), _ptr(pos_out), _ptr(n_cells_out),
        max_cells, _stream(stream)))


def sparse_attn_workspace_size(n_q, H_q, H_kv, d_v, max_cells) -> int:
    return int(load().qsa_sparse_attn_workspace_size(n_q, H_q, H_kv, d_v, max_cells))


def sparse_attn(q, K, V, n_cells, max_cells, out, H_kv, d_k, d_v, scale, pos=None, lse=None,
                workspace=None, ld_k=None, ld_v=None, n_kv=None, stream=None):
    """qsa_sparse_attn: q [n_q][H_q][d_k] fp32 over listed cells of K/V."""
    n_q, H_q = q.shape[0], q.shape[1]
    ld_k = _ld(K) if ld_k is None else ld_k
    ld_v = _ld(V) if ld_v is None else ld_v
    n_kv = K.shape[0] if n_kv is None else n_kv
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("qsa_sparse_attn", load().qsa_sparse_attn(
        _ptr(q), n_q, H_q, H_kv, d_k, d_v, scale, _ptr(K), _ptr(V), _dtype(K), n_kv, ld_k, ld_v,
        _ptr(pos), _ptr(n_cells), max_cells, _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
        _stream(stream)))


def sparse_attn_union(q, K, V, n_cells, max_cells, out, H_kv, d, scale, pos, lse=None,
                      workspace=None, ld_k=None, ld_v=None, n_kv=None, stream=None):
    """qsa_sparse_attn_union: q [n_q][H_q][d] fp32, groups of 16 consecutive queries over the
    union of their lists (bf16 K/V, d 128, 8 query heads per KV head)."""
    n_q, H_q = q.shape[0], q.shape[1]
    ld_k = _ld(K) if ld_k is None else ld_k
    ld_v = _ld(V) if ld_v is None else ld_v
    n_kv = K.shape[0] if n_kv is None else n_kv
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("qsa_sparse_attn_union", load().qsa_sparse_attn_union(
        _ptr(q), n_q, H_q, H_kv, d, scale, _ptr(K), _ptr(V), _dtype(K), n_kv, ld_k, ld_v,
        _ptr(pos), _ptr(n_cells), max_cells, _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
        _stream(stream)))


def sparse_attn_union_workspace_size(n_q, max_cells) -> int:
    return int(load().qsa_sparse_attn_union_workspace_size(n_q, max_cells))


def decode_step(raw_k, n_ctx, H_idx, d_idx, norm_w, eps, rope_base, pooled, n_valid_full,
                q_idx, scale_idx, scores, k_blk, blocks, counts, K, V, H_kv, d, pos, n_cells,
                max_cells, q, H_q, scale, out, lse=None, workspace=None, n_q=1, stream=None):
    """qsa_decode_step: pool update, score, top-k, cell list and attention in one call, for
    the last n_q tokens of the context (packed per-query buffers)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("qsa_decode_step", load().qsa_decode_step(
        _ptr(raw_k), _dtype(raw_k), n_ctx, H_idx, d_idx, _ptr(norm_w), eps, rope_base,
        _ptr(pooled), _dtype(pooled), pooled.shape[0], n_valid_full, n_q, _ptr(q_idx), scale_idx,
        _ptr(scores), k_blk, _ptr(blocks), _ptr(counts), _ptr(K), _ptr(V), _dtype(K), K.shape[0],
        H_kv, d, _ld(K), _ptr(pos), _ptr(n_cells), max_cells, _ptr(q), H_q, scale, _ptr(out),
        _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)))


def decode_step_workspace_size(H_q, H_kv, d, max_cells, cap_rows, n_q=1) -> int:
    return int(load().qsa_decode_step_workspace_size(n_q, H_q, H_kv, d, max_cells, cap_rows))


def decode_step_host_layout(n_q, raw_dtype, H_idx, d_idx, kv_dtype, H_kv, d, H_q):
    """(total bytes, [5] section offsets) of qsa_decode_step_host's packed input."""
    off = (ctypes.c_int64 * 5)()
    total = int(load().qsa_decode_step_host_layout(n_q, raw_dtype, H_idx, d_idx, kv_dtype, H_kv,
                                                   d, H_q, off))
    return total, list(off)


def decode_step_host_workspace_size(n_q, H_q, H_kv, d, max_cells, cap_rows, raw_dtype, H_idx,
                                    d_idx, kv_dtype) -> int:
    return int(load().qsa_decode_step_host_workspace_size(n_q, H_q, H_kv, d, max_cells, cap_rows,
                                                          raw_dtype, H_idx, d_idx, kv_dtype))


class DecodePlan:
    """A qsa_decode_plan: the fixed arguments of a sequence's decode steps bound once (the
    tensors are kept alive with the plan, which is destroyed with this object)."""

    def __init__(self, raw_k, norm_w, eps, rope_base, pooled, max_queries, scale_idx, scores,
                 k_blk, blocks, counts, K, V, H_idx, d_idx, H_kv, d, pos, n_cells, max_cells, H_q,
                 scale, out, lse, workspace):
        lib = load()
        handle = _p()
        ws_bytes = workspace.numel() * workspace.element_size()
        _check("qsa_decode_plan_create", lib.qsa_decode_plan_create(
            ctypes.byref(handle), _ptr(raw_k), _dtype(raw_k), H_idx, d_idx, _ptr(norm_w), eps,
            rope_base, _ptr(pooled), _dtype(pooled), pooled.shape[0], max_queries, scale_idx,
            _ptr(scores), k_blk, _ptr(blocks), _ptr(counts), _ptr(K), _ptr(V), _dtype(K),
            K.shape[0], H_kv, d, _ld(K), _ptr(pos), _ptr(n_cells), max_cells, H_q, scale,
            _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes))
        self._lib = lib
        self.handle = handle.value
        self._keep = (raw_k, norm_w, pooled, scores, blocks, counts, K, V, pos, n_cells, out, lse,
                      workspace)
        self.step = lib.qsa_decode_plan_step            # (handle, n_ctx, n_valid_full, n_q,
        self.step_host = lib.qsa_decode_plan_step_host  #  ...) -> status, see qsa.h

    def close(self):
        if self.handle:
            self._lib.qsa_decode_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown: the library may already be gone
            pass


def mask_to_list(mask, max_list, pos_out, counts_out, bits_out=None, n_kv=None, stream=None):
    """qsa_mask_to_list over every row of a uint8 mask [n_rows][ld]."""
    n_rows = mask.shape[0]
    n_kv = mask.shape[1] if n_kv is None else n_kv
    _check("qsa_mask_to_list", load().qsa_mask_to_list(
        _ptr(mask), n_rows, n_kv, _ld(mask), max_list, _ptr(pos_out), _ptr(counts_out),
        _ptr(bits_out), _stream(stream)))


def mask_sparse_attn(q, KV, mask, max_list, out, scale, counts_out=None, lse=None, n_kv=None,
                     d_k=576, d_v=512, stream=None):
    """qsa_mask_sparse_attn: q [n_q][16][576] fp32 over the set positions of each query's
    mask row (mask [n_q][ld] uint8), the latent KV rows [n_kv][ld] bf16."""
    n_q, H_q = q.shape[0], q.shape[1]
    n_kv = KV.shape[0] if n_kv is None else n_kv
    _check("qsa_mask_sparse_attn", load().qsa_mask_sparse_attn(
        _ptr(q), n_q, H_q, 1, d_k, d_v, scale, _ptr(KV), _dtype(KV), n_kv, _ld(KV), _ptr(mask),
        _ld(mask), max_list, _ptr(counts_out), _ptr(out), _ptr(lse), _stream(stream)))


def mask_sparse_eligible(has_mask, max_bias, softcap, n_kv, max_list) -> bool:
    st = load().qsa_mask_sparse_eligible(int(bool(has_mask)), max_bias, softcap, n_kv, max_list)
    if st not in (QSA_OK, QSA_ERR_UNSUPPORTED):
        raise QSAError("qsa_mask_sparse_eligible", st)
    return st == QSA_OK
