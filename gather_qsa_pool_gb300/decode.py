"""One QSA layer's decode step through the C ABI.

``DecodeLayer`` owns the device buffers of one QSA layer (the persistent pooled-key
cache, scores, selected blocks, cell lists, split-K workspace, output) and issues the
five library calls of a decode step on the current stream:

    qsa_pool_update -> qsa_index_score -> qsa_topk_blocks -> qsa_gather_kv
                    -> qsa_sparse_attn

either as the one fused call ``qsa_decode_step`` or one by one.  A step may carry up to
four query tokens (a token and the draft tokens that follow it, verified together): they
are the last ``n_q`` tokens of the context and share one scan of the pooled cache.

The raw indexer-key cache and the K/V cache belong to the caller (the model writes the
new tokens' rows before the step).  The gather call only builds the cell lists; the
attention kernel stages the listed K/V rows straight from the cache.
"""
from __future__ import annotations

import math

from . import _binding as qb


class DecodeLayer:
    def __init__(self, *, cap_tokens, H_idx, d_idx, H_q, H_kv, d, top_k_tokens,
                 eps=1e-6, rope_base=10000.0, pooled_dtype=None, max_queries=1,
                 device="cuda"):
        """pooled_dtype: torch.float32 (default) or torch.bfloat16 storage of the pooled
        cache.  max_queries: the most query tokens one step carries (1..4)."""
        import torch

        self.H_idx, self.d_idx = H_idx, d_idx
        self.H_q, self.H_kv, self.d = H_q, H_kv, d
        self.k_blk = top_k_tokens // 4
        self.eps, self.rope_base = eps, rope_base
        self.max_cells = 4 * self.k_blk + 3
        self.cap_rows = (cap_tokens + 3) // 4
        self.max_queries = max_queries
        f32, i32 = torch.float32, torch.int32
        nq = max_queries
        pdt = f32 if pooled_dtype is None else pooled_dtype
        self.pooled = torch.zeros(self.cap_rows, H_idx * d_idx, dtype=pdt, device=device)
        # scores of a step are packed [n_q][n_rows] at the start of this buffer
        self.scores = torch.zeros(nq * self.cap_rows, dtype=f32, device=device)
        self.blocks = torch.zeros(nq, self.k_blk, dtype=i32, device=device)
        self.counts = torch.zeros(nq, dtype=i32, device=device)
        self.pos = torch.zeros(nq, self.max_cells, dtype=i32, device=device)
        self.n_cells = torch.zeros(nq, dtype=i32, device=device)
        self.out = torch.zeros(nq, H_q, d, dtype=f32, device=device)
        self.lse = torch.zeros(nq, H_q, dtype=f32, device=device)
        ws = qb.decode_step_workspace_size(H_q, H_kv, d, self.max_cells, self.cap_rows, nq)
        # zero-filled once: the step keeps its top-k histograms cleared from then on
        self.workspace = torch.zeros(max(ws // 4, 1), dtype=f32, device=device)
        self.n_valid_full = 0

    def rebuild(self, raw_k, norm_w, n_ctx, stream=None):
        """Recompute every pooled row (state load / sequence edit)."""
        qb.pool_update(raw_k, n_ctx, self.H_idx, self.d_idx, norm_w, self.eps, self.rope_base,
                       self.pooled, 0, stream)
        self.n_valid_full = n_ctx // 4

    def invalidate(self, first_changed_token):
        """Rows from the block holding ``first_changed_token`` on are recomputed next step
        (e.g. after rejected draft tokens are rolled back)."""
        self.n_valid_full = min(self.n_valid_full, first_changed_token // 4)

    def scores_of(self, n_q, n_ctx):
        """The last step's scores as [n_q][n_rows]."""
        n_rows = (n_ctx + 3) // 4
        return self.scores[:n_q * n_rows].view(n_q, n_rows)

    def step(self, raw_k, norm_w, K, V, n_ctx, q_idx, q, stream=None):
        """Decode step at context length n_ctx for the last n_q tokens (the current token
        is position n_ctx-1).

        q_idx: [n_q][H_idx*d_idx] (or [H_idx*d_idx]) fp32, q: [n_q][H_q][d] (or [H_q][d])
        fp32.  Returns the output [n_q][H_q][d] (a view into this layer's buffer,
        overwritten by the next step)."""
        n_q = q_idx.shape[0] if q_idx.dim() > 1 else 1
        qb.decode_step(raw_k, n_ctx, self.H_idx, self.d_idx, norm_w, self.eps, self.rope_base,
                       self.pooled, self.n_valid_full, q_idx, 1.0 / math.sqrt(self.d_idx),
                       self.scores, self.k_blk, self.blocks, self.counts, K, V, self.H_kv,
                       self.d, self.pos, self.n_cells, self.max_cells, q, self.H_q,
                       1.0 / math.sqrt(self.d), self.out, self.lse, self.workspace, n_q, stream)
        self.n_valid_full = n_ctx // 4
        return self.out[:n_q]

    def bind(self, raw_k, norm_w, K, V):
        """Bind the caller-owned caches and this layer's buffers into a qsa_decode_plan for
        ``step_ptr`` / ``step_host`` (per step only the context length, the validity
        watermark, the query count and the query pointers cross the C boundary)."""
        self._bound = (raw_k, norm_w, K, V)
        self._plan = qb.DecodePlan(raw_k, norm_w, self.eps, self.rope_base, self.pooled,
                                   self.max_queries, 1.0 / math.sqrt(self.d_idx), self.scores,
                                   self.k_blk, self.blocks, self.counts, K, V, self.H_idx,
                                   self.d_idx, self.H_kv, self.d, self.pos, self.n_cells,
                                   self.max_cells, self.H_q, 1.0 / math.sqrt(self.d), self.out,
                                   self.lse, self.workspace)

    def step_ptr(self, n_ctx, q_idx_ptr, q_ptr, stream_ptr, n_q=1):
        """Decode step on the caches fixed by ``bind``; q_idx / q given as device pointers."""
        plan = self._plan
        st = plan.step(plan.handle, n_ctx, self.n_valid_full, n_q, q_idx_ptr, q_ptr, stream_ptr)
        if st != 0:
            raise qb.QSAError("qsa_decode_plan_step", st)
        self.n_valid_full = n_ctx // 4

    # ------------------------------------------------------------------ host-fed steps

    def enable_host_feed(self, raw_dtype, kv_dtype, pinned=True):
        """Prepare steps fed from host memory (qsa_decode_step_host): a workspace with room
        for the staging area and the host input / output buffers.  raw_dtype, kv_dtype:
        torch dtypes of the raw indexer-key and K/V caches.  pinned: page-locked buffers,
        which the library's kernels read and write in place; pageable ones go through
        copy-engine transfers instead."""
        import torch

        rd = qb.QSA_BF16 if raw_dtype == torch.bfloat16 else qb.QSA_F32
        kd = qb.QSA_BF16 if kv_dtype == torch.bfloat16 else qb.QSA_F32
        self._host_dtypes = (rd, kd, raw_dtype, kv_dtype)
        nq = self.max_queries
        ws = qb.decode_step_host_workspace_size(nq, self.H_q, self.H_kv, self.d, self.max_cells,
                                                self.cap_rows, rd, self.H_idx, self.d_idx, kd)
        dev = self.workspace.device
        self.workspace = torch.zeros(max(ws // 4, 1), dtype=torch.float32, device=dev)
        total, _ = qb.decode_step_host_layout(nq, rd, self.H_idx, self.d_idx, kd, self.H_kv,
                                              self.d, self.H_q)
        self.h_in = torch.zeros(total, dtype=torch.uint8)
        self.h_out = torch.zeros(nq, self.H_q, self.d, dtype=torch.float32)
        self.h_lse = torch.zeros(nq, self.H_q, dtype=torch.float32)
        if pinned:
            self.h_in, self.h_out, self.h_lse = (self.h_in.pin_memory(), self.h_out.pin_memory(),
                                                 self.h_lse.pin_memory())
        self._host_ptrs = (self.h_in.data_ptr(), self.h_out.data_ptr(), self.h_lse.data_ptr())
        if getattr(self, "_bound", None) is not None:
            self.bind(*self._bound)  # the plan must see the larger workspace

    def host_inputs(self, n_q):
        """Views of the packed host input for a step of n_q queries: dict with 'raw' [n_q]
        [H_idx*d_idx], 'k' and 'v' [n_q][H_kv*d], 'q_idx' [n_q][H_idx*d_idx], 'q' [n_q][H_q]
        [d]; fill them, then call step_host."""
        import torch

        rd, kd, rdt, kdt = self._host_dtypes
        total, off = qb.decode_step_host_layout(n_q, rd, self.H_idx, self.d_idx, kd, self.H_kv,
                                                self.d, self.H_q)
        hd, kvd = self.H_idx * self.d_idx, self.H_kv * self.d

        def view(o, dtype, shape):
            n = 1
            for x in shape:
                n *= x
            es = torch.tensor([], dtype=dtype).element_size()
            return self.h_in[o:o + n * es].view(dtype).view(*shape)

        return {"raw": view(off[0], rdt, (n_q, hd)), "k": view(off[1], kdt, (n_q, kvd)),
                "v": view(off[2], kdt, (n_q, kvd)), "q_idx": view(off[3], torch.float32, (n_q, hd)),
                "q": view(off[4], torch.float32, (n_q, self.H_q, self.d)), "bytes": total}

    def step_host(self, n_ctx, stream_ptr, n_q=1, with_lse=False):
        """Host-fed decode step on the caches fixed by ``bind``: the new tokens' rows and the
        queries come from ``h_in`` (see host_inputs), the output lands in ``h_out`` (and the
        log-sum-exp in ``h_lse`` when with_lse) once the stream has been synchronised."""
        plan = self._plan
        h_in, h_out, h_lse = self._host_ptrs
        st = plan.step_host(plan.handle, n_ctx, self.n_valid_full, n_q, h_in, h_out,
                            h_lse if with_lse else None, stream_ptr)
        if st != 0:
            raise qb.QSAError("qsa_decode_plan_step_host", st)
        self.n_valid_full = n_ctx // 4

    def step_separate_calls(self, raw_k, norm_w, K, V, n_ctx, q_idx, q, stream=None):
        """The same step issued as the five individual C calls."""
        import torch

        q_idx = q_idx.view(-1, self.H_idx * self.d_idx)
        n_q = q_idx.shape[0]
        n_rows = (n_ctx + 3) // 4
        n_full = n_ctx // 4
        qb.pool_update(raw_k, n_ctx, self.H_idx, self.d_idx, norm_w, self.eps, self.rope_base,
                       self.pooled, self.n_valid_full, stream)
        self.n_valid_full = n_full
        scores = self.scores_of(n_q, n_ctx)
        qb.index_score(q_idx, self.pooled, n_rows, self.H_idx, self.d_idx,
                       1.0 / math.sqrt(self.d_idx), scores, stream=stream)
        q_pos = None
        if n_q > 1:
            q_pos = torch.arange(n_ctx - n_q, n_ctx, dtype=torch.int32, device=q_idx.device)
        qb.topk_blocks(scores, n_full, self.k_blk, self.blocks[:n_q], self.counts[:n_q],
                       q_pos=q_pos, stream=stream)
        qb.gather_kv(self.blocks[:n_q], self.counts[:n_q], self.k_blk, self.pos[:n_q],
                     self.n_cells[:n_q], self.max_cells, n_ctx=n_ctx, q_pos=q_pos,
                     n_kv=K.shape[0], stream=stream)
        qb.sparse_attn(q.view(n_q, self.H_q, self.d), K, V, self.n_cells[:n_q], self.max_cells,
                       self.out[:n_q], self.H_kv, self.d, self.d, 1.0 / math.sqrt(self.d),
                       pos=self.pos[:n_q], lse=self.lse[:n_q], workspace=self.workspace,
                       ld_k=self.H_kv * self.d, ld_v=self.H_kv * self.d, stream=stream)
        return self.out[:n_q]
