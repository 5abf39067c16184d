"""GB300 (sm_103a) QSA two-stage sparse attention.

The compute lives in ``libqsa.so`` (hand-written CUDA kernels behind a C ABI declared in
``include/qsa.h``); this package is its ctypes binding plus a small decode-step driver
that owns the per-layer device buffers.  There is no CPU or PyTorch fallback.
"""
from ._binding import (  # noqa: F401
    QSA_BF16,
    QSA_F32,
    QSA_PREC_BF16_TC,
    QSA_PREC_F32,
    QSA_WAIT_DEFAULT_NS,
    QSAError,
    decode_step,
    decode_step_host_layout,
    decode_step_host_workspace_size,
    decode_step_workspace_size,
    expand_block_scores,
    gather_kv,
    header_functions,
    index_score,
    index_score_maxima,
    index_score_workspace_size,
    load,
    mask_sparse_attn,
    mask_sparse_eligible,
    mask_to_list,
    pool_update,
    set_wait_options,
    sparse_attn,
    sparse_attn_union,
    sparse_attn_union_workspace_size,
    sparse_attn_workspace_size,
    status_str,
    topk_blocks,
    topk_blocks_maxima,
    topk_blocks_maxima_workspace_size,
    topk_max_candidates,
)
from .decode import DecodeLayer  # noqa: F401
