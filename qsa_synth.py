"""Seeded synthetic inputs for QSA two-stage sparse attention.

This module only draws random numbers and lays them out.  It holds none of the
method's arithmetic (no pooling, normalisation, rotation, scoring, selection or
attention), imports neither the CUDA library nor the CPU oracle, and is the one piece
of code both sides share: the same bytes go to the GPU path and to the oracle.

Workload shapes follow the QSA configuration of the source pages: 4-token blocks,
indexer top-k of 2048 tokens (512 blocks) plus the open tail, context lengths of
61,789 / 126,253 / 255,181 tokens, and for the mask-driven variant DKQ = 576 with
16 query heads per KV head.  Head counts and dims the pages leave open come from the
configurations listed in ``CONFIGS``.

CPU generation uses numpy PCG64; bf16 tensors are returned as uint16 bit patterns
(round-to-nearest-even of an fp32 N(0,1) draw).  ``*_torch`` variants draw the same
distributions on a CUDA device with a seeded torch generator (used by the benchmark,
where multi-GB inputs would take minutes on the host).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import numpy as np


@dataclass(frozen=True)
class DecodeShape:
    name: str
    n_ctx: int            # tokens in the cache including the current one
    H_idx: int            # indexer heads
    d_idx: int            # indexer head dim
    H_q: int              # attention query heads
    H_kv: int             # attention KV heads
    d: int                # attention head dim (d_k = d_v)
    top_k_tokens: int     # indexer top-k in tokens (blocks = top_k_tokens / 4)
    dtype: str            # "f32" or "bf16": raw indexer keys and K/V storage
    eps: float = 1e-6
    rope_base: float = 10000.0
    bias_frac: float = 0.0    # fraction of blocks whose raw indexer keys get +bias_sigma
    bias_sigma: float = 3.0

    @property
    def k_blk(self) -> int:
        return self.top_k_tokens // 4

    @property
    def n_full(self) -> int:
        return self.n_ctx // 4

    @property
    def n_rows(self) -> int:
        return (self.n_ctx + 3) // 4

    @property
    def max_cells(self) -> int:
        return 4 * self.k_blk + 3


@dataclass(frozen=True)
class PrefillShape:
    name: str
    depth: int            # tokens before the chunk; query i sits at position depth + i
    n_q: int              # queries in the chunk
    H_idx: int
    d_idx: int
    H_q: int
    H_kv: int
    d: int
    top_k_tokens: int
    dtype: str = "bf16"
    eps: float = 1e-6
    rope_base: float = 10000.0
    bias_frac: float = 0.01
    bias_sigma: float = 3.0

    @property
    def n_ctx(self) -> int:
        return self.depth + self.n_q

    @property
    def k_blk(self) -> int:
        return self.top_k_tokens // 4

    @property
    def n_rows(self) -> int:
        return (self.n_ctx + 3) // 4

    @property
    def max_cells(self) -> int:
        return 4 * self.k_blk + 3


@dataclass(frozen=True)
class MaskShape:
    name: str
    n_q: int              # query tokens (one mask row each)
    n_kv: int             # key length
    H_q: int              # query heads sharing the single KV head
    d_k: int
    d_v: int
    max_list: int
    runs: int = 15        # contiguous runs of set positions
    run_len: int = 64
    p_set: float = 0.0316 # Bernoulli density elsewhere (about 6% set overall)


CONFIGS = {
    # tiny fp32 decode: 2,050 tokens = 512 full blocks + a 2-token tail
    "tiny_f32_decode": DecodeShape("tiny_f32_decode", 2050, 4, 64, 8, 2, 128, 64, "f32"),
    # bf16 decode at the pages' three context lengths
    "decode_64k": DecodeShape("decode_64k", 61789, 16, 128, 32, 4, 128, 2048, "bf16",
                              bias_frac=0.01),
    "decode_128k": DecodeShape("decode_128k", 126253, 16, 128, 32, 4, 128, 2048, "bf16",
                               bias_frac=0.01),
    "decode_256k": DecodeShape("decode_256k", 255181, 16, 128, 32, 4, 128, 2048, "bf16",
                               bias_frac=0.01),
    # prefill chunk of 1024 queries following 255,181 tokens
    "prefill_256k": PrefillShape("prefill_256k", 255181, 1024, 16, 128, 32, 4, 128, 2048),
    # mask-driven sparse attention, DKQ 576 / d_v 512, 16 heads per KV head
    "mask_32k": MaskShape("mask_32k", 4, 32768, 16, 576, 512, 2048),
}


def shrink(shape, **kw):
    """Same shape with some fields replaced (small parity cases)."""
    return replace(shape, **kw)


# --------------------------------------------------------------------------- helpers

_CHUNK = 1 << 22  # elements per generator stream / conversion chunk


def _pool():
    return ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1))


def _to_bf16_chunk(u: np.ndarray, out: np.ndarray):
    t = (u >> np.uint32(16)) & np.uint32(1)
    t += np.uint32(0x7FFF)
    t += u
    t >>= np.uint32(16)
    out[...] = t


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (inputs hold no NaN)."""
    u = np.ascontiguousarray(x, np.float32).reshape(-1).view(np.uint32)
    out = np.empty(u.shape[0], np.uint16)
    with _pool() as ex:
        list(ex.map(lambda i: _to_bf16_chunk(u[i:i + _CHUNK], out[i:i + _CHUNK]),
                    range(0, u.shape[0], _CHUNK)))
    return out.reshape(np.shape(x))


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal(rng, shape):
    """N(0,1) float32 of the given shape.  Large draws are split into fixed-size chunks,
    each with its own stream seeded from ``rng`` (deterministic for any thread count)."""
    n = int(np.prod(shape))
    if n <= _CHUNK:
        return rng.standard_normal(size=shape, dtype=np.float32)
    out = np.empty(n, np.float32)
    starts = list(range(0, n, _CHUNK))
    seeds = rng.integers(0, 2 ** 63 - 1, size=len(starts))

    def fill(k):
        g = np.random.Generator(np.random.PCG64(int(seeds[k])))
        g.standard_normal(out=out[starts[k]:starts[k] + _CHUNK], dtype=np.float32)

    with _pool() as ex:
        list(ex.map(fill, range(len(starts))))
    return out.reshape(shape)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return to_bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, np.float32)


def _bias_blocks(rng, n_blocks: int, frac: float) -> np.ndarray:
    n = int(round(frac * n_blocks))
    if n <= 0:
        return np.zeros(0, np.int64)
    return np.sort(rng.choice(n_blocks, size=n, replace=False))


# --------------------------------------------------------------------------- decode

def decode_inputs(shape: DecodeShape, seed: int, extra_tokens: int = 0, n_steps: int = 1):
    """Inputs of a decode workload on the host.

    Returns a dict with
      raw_k  [n_ctx+extra][H_idx][d_idx]  raw indexer keys (f32 or bf16 bits)
      norm_w [d_idx] f32                  RMS-norm weight, 1 + 0.1 N(0,1)
      K, V   [n_ctx+extra][H_kv][d]       KV cache (f32 or bf16 bits)
      q_idx  [n_steps][H_idx*d_idx] f32   indexer queries (already position-encoded)
      q      [n_steps][H_q][d] f32        attention queries
      bias_blocks                         blocks whose raw keys carry +bias_sigma
    ``extra_tokens`` rows beyond n_ctx hold the tokens that later decode steps append.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    n_tok = shape.n_ctx + extra_tokens
    raw = _normal(rng, (n_tok, shape.H_idx, shape.d_idx))
    bias = _bias_blocks(rng, n_tok // 4, shape.bias_frac)
    for b in bias:
        raw[4 * b:4 * b + 4] += np.float32(shape.bias_sigma)
    w = (1.0 + 0.1 * _normal(rng, (shape.d_idx,))).astype(np.float32)
    K = _normal(rng, (n_tok, shape.H_kv, shape.d))
    V = _normal(rng, (n_tok, shape.H_kv, shape.d))
    q_idx = _normal(rng, (n_steps, shape.H_idx * shape.d_idx))
    q = _normal(rng, (n_steps, shape.H_q, shape.d))
    return {
        "raw_k": _store(raw, shape.dtype),
        "norm_w": w,
        "K": _store(K, shape.dtype),
        "V": _store(V, shape.dtype),
        "q_idx": q_idx,
        "q": q,
        "bias_blocks": bias,
    }


def decode_inputs_torch(shape: DecodeShape, seed: int, device, extra_tokens: int = 0,
                        n_steps: int = 1):
    """Device-side draw of the same distributions as ``decode_inputs`` (torch tensors)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    n_tok = shape.n_ctx + extra_tokens
    tdt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32

    def normal(*sz):
        return torch.randn(*sz, generator=g, device=device, dtype=torch.float32)

    raw = normal(n_tok, shape.H_idx, shape.d_idx)
    n_bias = int(round(shape.bias_frac * (n_tok // 4)))
    if n_bias:
        idx = torch.randperm(n_tok // 4, generator=g, device=device)[:n_bias]
        tok = (4 * idx[:, None] + torch.arange(4, device=device)[None, :]).reshape(-1)
        raw[tok] += shape.bias_sigma
    raw = raw.to(tdt)
    w = 1.0 + 0.1 * normal(shape.d_idx)
    K = normal(n_tok, shape.H_kv, shape.d).to(tdt)
    V = normal(n_tok, shape.H_kv, shape.d).to(tdt)
    q_idx = normal(n_steps, shape.H_idx * shape.d_idx)
    q = normal(n_steps, shape.H_q, shape.d)
    return {"raw_k": raw, "norm_w": w, "K": K, "V": V, "q_idx": q_idx, "q": q}


def clear_winners_torch(n_rows: int, width: int, n_steps: int, seed: int, device,
                        frac: float = 0.01, sigma: float = 3.0):
    """A decode workload whose block scores have clear winners (a timing variant).

    The keys' bias cannot be lined up with the queries in the raw keys without the
    method's own normalisation and rotation, so this draw acts on the completed rows of
    the pooled-key cache, which a decode step takes as given: a direction u ~ N(0,1)^width,
    queries N(0,1) + u, and a random ``frac`` of the rows [0, n_rows) receive lean * u with
    lean = sigma * sqrt(2 / width).  Against rows of unit-variance entries, the raw dot
    product with such a query has standard deviation sqrt(2 * width) and the lean adds
    about lean * width = sigma of those deviations to a chosen row.
    Returns {"q_idx": [n_steps][width], "rows": sorted row indices, "add": [width] the vector
    to add to each chosen row}."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    u = torch.randn(width, generator=g, device=device, dtype=torch.float32)
    q_idx = torch.randn(n_steps, width, generator=g, device=device, dtype=torch.float32) + u
    n = int(round(frac * n_rows))
    rows = torch.randperm(n_rows, generator=g, device=device)[:n].sort().values
    return {"q_idx": q_idx, "rows": rows, "add": (sigma * (2.0 / width) ** 0.5) * u}


# --------------------------------------------------------------------------- prefill

def prefill_inputs(shape: PrefillShape, seed: int, n_tok: int | None = None):
    """Inputs of a prefill chunk: caches of ``n_ctx`` tokens plus per-query vectors."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n_tok = shape.n_ctx if n_tok is None else n_tok
    raw = _normal(rng, (n_tok, shape.H_idx, shape.d_idx))
    bias = _bias_blocks(rng, n_tok // 4, shape.bias_frac)
    for b in bias:
        raw[4 * b:4 * b + 4] += np.float32(shape.bias_sigma)
    w = (1.0 + 0.1 * _normal(rng, (shape.d_idx,))).astype(np.float32)
    K = _normal(rng, (n_tok, shape.H_kv, shape.d))
    V = _normal(rng, (n_tok, shape.H_kv, shape.d))
    q_idx = _normal(rng, (shape.n_q, shape.H_idx * shape.d_idx))
    q = _normal(rng, (shape.n_q, shape.H_q, shape.d))
    q_pos = (shape.depth + np.arange(shape.n_q)).astype(np.int32)
    return {
        "raw_k": _store(raw, shape.dtype),
        "norm_w": w,
        "K": _store(K, shape.dtype),
        "V": _store(V, shape.dtype),
        "q_idx": q_idx,
        "q": q,
        "q_pos": q_pos,
    }


def prefill_inputs_torch(shape: PrefillShape, seed: int, device):
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    n_tok = shape.n_ctx

    def normal(*sz):
        return torch.randn(*sz, generator=g, device=device, dtype=torch.float32)

    raw = normal(n_tok, shape.H_idx, shape.d_idx)
    n_bias = int(round(shape.bias_frac * (n_tok // 4)))
    if n_bias:
        idx = torch.randperm(n_tok // 4, generator=g, device=device)[:n_bias]
        tok = (4 * idx[:, None] + torch.arange(4, device=device)[None, :]).reshape(-1)
        raw[tok] += shape.bias_sigma
    return {
        "raw_k": raw.to(torch.bfloat16),
        "norm_w": 1.0 + 0.1 * normal(shape.d_idx),
        "K": normal(n_tok, shape.H_kv, shape.d).to(torch.bfloat16),
        "V": normal(n_tok, shape.H_kv, shape.d).to(torch.bfloat16),
        "q_idx": normal(shape.n_q, shape.H_idx * shape.d_idx),
        "q": normal(shape.n_q, shape.H_q, shape.d),
        "q_pos": (shape.depth + torch.arange(shape.n_q, device=device)).to(torch.int32),
    }


# --------------------------------------------------------------------------- mask

def mask_rows(n_rows: int, n_kv: int, seed: int, runs: int = 15, run_len: int = 64,
              p_set: float = 0.0316) -> np.ndarray:
    """uint8 [n_rows][n_kv]: Bernoulli(p_set) positions plus ``runs`` contiguous runs of
    ``run_len`` set positions at unaligned random starts (values 0/1, plus a few 2..255
    so that 'nonzero' rather than '== 1' is what counts)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    m = (rng.random((n_rows, n_kv)) < p_set).astype(np.uint8)
    for r in range(n_rows):
        for s in rng.integers(0, max(n_kv - run_len, 1), size=runs):
            m[r, s:s + run_len] = 1
    big = rng.random((n_rows, n_kv)) < 0.002
    m[big & (m > 0)] = rng.integers(2, 256, size=int((big & (m > 0)).sum()), dtype=np.uint8)
    return m


def mask_attn_inputs(shape: MaskShape, seed: int):
    """Queries [n_q][H_q][d_k] f32 and one KV tensor [n_kv][d_k] bf16 bits; V is the
    first d_v columns of each K row (row stride d_k), as in a latent-KV cache."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _normal(rng, (shape.n_q, shape.H_q, shape.d_k))
    KV = to_bf16_bits(_normal(rng, (shape.n_kv, shape.d_k)))
    return {"q": q, "KV": KV}


# --------------------------------------------------------------------------- shared selections

def overlap_block_lists(n_cand, k_blk: int, group: int, share: float, seed: int):
    """Block lists with a stated overlap inside each group of ``group`` consecutive queries,
    for measuring how attention over a group's union behaves as queries share more blocks.

    n_cand[i] is how many blocks query i may pick from (blocks 0 .. n_cand[i]-1).  Each group
    draws one common set of k_blk blocks from the blocks every member may pick; each query
    takes round(share * k) of them (k = min(k_blk, n_cand[i])) and draws the rest uniformly
    from its other candidates, without repeats.  Returns a list of ascending int32 arrays.
    Only random draws: nothing of the method's arithmetic."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n_cand = np.asarray(n_cand, np.int64)
    out = []
    for g0 in range(0, n_cand.shape[0], group):
        members = n_cand[g0:g0 + group]
        lo = int(members.min())
        common = rng.choice(lo, size=min(k_blk, lo), replace=False) if lo > 0 else np.zeros(0, np.int64)
        for nc in members:
            k = int(min(k_blk, nc))
            n_sh = min(int(round(share * k)), common.shape[0])
            mine = rng.choice(common, size=n_sh, replace=False) if n_sh else np.zeros(0, np.int64)
            taken = np.zeros(int(nc), bool)
            taken[mine] = True
            rest = np.flatnonzero(~taken)
            extra = rng.choice(rest, size=k - n_sh, replace=False) if k > n_sh else np.zeros(0, np.int64)
            out.append(np.sort(np.concatenate([mine, extra])).astype(np.int32))
    return out
