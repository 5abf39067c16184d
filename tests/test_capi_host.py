"""Host-only checks of the C ABI: the library builds for sm_103a, loads without a GPU,
exports every function include/qsa.h declares, and rejects bad arguments before it
launches anything (no call here reaches a kernel)."""
import ctypes

import pytest

import gather_qsa_pool_gb300 as qsa
from gather_qsa_pool_gb300 import _binding as qb

P = ctypes.c_void_p
FAKE = P(0x10000)  # never dereferenced: every call below fails validation first


@pytest.fixture(scope="module")
def lib():
    return qsa.load()


def test_library_exports_every_declared_function(lib):
    names = qb.header_functions()
    assert len(names) >= 12
    for n in ["qsa_pool_update", "qsa_index_score", "qsa_topk_blocks", "qsa_gather_kv",
              "qsa_sparse_attn", "qsa_mask_to_list"]:
        assert n in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert qsa.status_str(0) == "QSA_OK"
    assert qsa.status_str(1) == "QSA_ERR_INVALID_ARG"
    assert qsa.status_str(4) == "QSA_ERR_TIMEOUT"
    assert lib.qsa_version() >> 16 == 2
    assert lib.qsa_version() & 0xFFFF >= 2  # decode plans, the one-call mask attention


def test_pool_update_rejects(lib):
    s = None
    assert lib.qsa_pool_update(None, 0, 10, 4, 64, FAKE, 1e-6, 1e4, FAKE, 0, 10, 0, s) == 1
    assert lib.qsa_pool_update(FAKE, 0, 10, 4, 63, FAKE, 1e-6, 1e4, FAKE, 0, 10, 0, s) == 1  # odd d
    assert lib.qsa_pool_update(FAKE, 0, 41, 4, 64, FAKE, 1e-6, 1e4, FAKE, 0, 10, 0, s) == 1  # cap
    assert lib.qsa_pool_update(FAKE, 0, 10, 4, 64, FAKE, 1e-6, 1e4, FAKE, 0, 10, -1, s) == 1
    assert lib.qsa_pool_update(FAKE, 7, 10, 4, 64, FAKE, 1e-6, 1e4, FAKE, 0, 10, 0, s) == 1  # dtype
    assert lib.qsa_pool_update(FAKE, 0, 10, 4, 64, FAKE, 1e-6, 1e4, FAKE, 5, 10, 0, s) == 1  # pooled
    assert lib.qsa_pool_update(FAKE, 0, 10, 4, 64, FAKE, 1e-6, -1.0, FAKE, 0, 10, 0, s) == 1
    # a bf16 cache must be 2-byte aligned
    assert lib.qsa_pool_update(FAKE, 0, 10, 4, 64, FAKE, 1e-6, 1e4, P(0x10001), 1, 10, 0, s) == 1


def test_index_score_rejects(lib):
    s = None
    args = [FAKE, 1, 256, None, FAKE, 0, 10, 4, 64, 1.0, FAKE, 10, 0, None, 0, s]

    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return lib.qsa_index_score(*a)

    assert call(a0=None) == 1
    assert call(a2=255) == 1           # ld_q < H*d
    assert call(a11=9) == 1            # ld_scores < n_rows
    assert call(a12=9) == 1            # unknown precision
    assert call(a5=3) == 1             # unknown pooled dtype
    assert call(a4=P(0x10002)) == 1    # fp32 cache not 4-byte aligned
    assert lib.qsa_index_score_workspace_size(4, 100, 16, 128, 1, 1) < \
        lib.qsa_index_score_workspace_size(4, 100, 16, 128, 0, 1)  # a bf16 cache is read in place
    assert lib.qsa_index_score_workspace_size(4, 100, 16, 128, 0, 0) == 0


def test_maxima_calls_reject(lib):
    """qsa_index_score_maxima / qsa_topk_blocks_maxima: the checks of the calls they extend,
    plus a missing or misaligned maxima array and a short maxima stride (nothing launched)."""
    s = None
    sa = [FAKE, 1, 256, None, FAKE, 0, 100, 4, 64, 1.0, FAKE, 100, FAKE, 4, None, 0, s]

    def score(**kw):
        a = list(sa)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return lib.qsa_index_score_maxima(*a)

    assert score(a12=None) == 1          # no maxima
    assert score(a12=P(0x10002)) == 1    # maxima not 4-byte aligned
    assert score(a13=3) == 1             # ld_maxima < ceil(100 / 32)
    assert score(a2=255) == 1            # ld_q < H*d
    assert score(a11=99) == 1            # ld_scores < n_rows
    assert score(a15=0) == 1             # workspace smaller than required
    ws = lib.qsa_topk_blocks_maxima_workspace_size(2)
    assert ws >= 256 + 8 and lib.qsa_topk_blocks_maxima_workspace_size(0) == 0
    ta = [FAKE, 2, 70000, None, 70000, 512, FAKE, 2187, FAKE, FAKE, P(0x20000), ws, s]

    def topk(**kw):
        a = list(ta)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return lib.qsa_topk_blocks_maxima(*a)

    assert topk(a6=None) == 1            # no maxima
    assert topk(a7=2186) == 1            # ld_maxima < 70000 / 32
    assert topk(a5=0) == 1               # k_blk < 1
    assert topk(a2=69999) == 1           # ld_scores < n_full
    assert topk(a8=None) == 1            # no output
    assert topk(a11=ws - 1) == 1         # workspace smaller than required
    assert topk(a10=P(0x20010)) == 1     # workspace not 256-byte aligned


def test_decode_step_workspace_and_query_count(lib):
    one = lib.qsa_decode_step_workspace_size(1, 32, 4, 128, 2051, 64000)
    three = lib.qsa_decode_step_workspace_size(3, 32, 4, 128, 2051, 64000)
    assert one > 0 and three > 2 * one
    assert lib.qsa_decode_step_workspace_size(0, 32, 4, 128, 2051, 64000) == 0
    assert lib.qsa_decode_step_workspace_size(5, 32, 4, 128, 2051, 64000) == 0
    st = None

    def step(n_q, n_ctx=1000, ws_bytes=1 << 30):
        return lib.qsa_decode_step(FAKE, 1, n_ctx, 16, 128, FAKE, 1e-6, 1e4, FAKE, 0, 4000, 0,
                                   n_q, FAKE, 0.1, FAKE, 512, FAKE, FAKE, FAKE, FAKE, 1, n_ctx, 4,
                                   128, 512, FAKE, FAKE, 2051, FAKE, 32, 0.1, FAKE, None,
                                   P(0x100000), ws_bytes, st)

    assert step(0) == 1            # no query
    assert step(5) == 1            # more than four
    assert step(3, n_ctx=2) == 1   # more queries than tokens
    assert step(3, ws_bytes=one) == 1  # workspace sized for one query


def test_topk_rejects(lib):
    s = None
    assert lib.qsa_topk_blocks(FAKE, 1, 10, None, 10, 0, FAKE, FAKE, s) == 1      # k < 1
    assert lib.qsa_topk_blocks(FAKE, 1, 9, None, 10, 4, FAKE, FAKE, s) == 1       # ld < n_full
    assert lib.qsa_topk_blocks(None, 1, 10, None, 10, 4, FAKE, FAKE, s) == 1
    big = lib.qsa_topk_max_candidates() + 1
    assert lib.qsa_topk_blocks(FAKE, 1, big, None, big, 4, FAKE, FAKE, s) == 2
    assert lib.qsa_topk_max_candidates() >= 64052  # a 256k-token context fits


def test_expand_block_scores_rejects(lib):
    s = None
    assert lib.qsa_expand_block_scores(None, 1, 10, 10, FAKE, 40, s) == 1
    assert lib.qsa_expand_block_scores(FAKE, 1, 9, 10, FAKE, 40, s) == 1    # ld_scores < n_full
    assert lib.qsa_expand_block_scores(FAKE, 1, 10, 10, FAKE, 39, s) == 1   # ld_cells < 4 n_full
    assert lib.qsa_expand_block_scores(FAKE, -1, 10, 10, FAKE, 40, s) == 1
    assert lib.qsa_expand_block_scores(FAKE, 70000, 10, 10, FAKE, 40, s) == 2


def test_gather_rejects(lib):
    s = None
    # max_cells < 4*k_blk + 3
    assert lib.qsa_gather_kv(None, None, 1, 100, 4, 128, 128, 512, 512, FAKE, FAKE, 1, 16, None,
                             100, None, None, FAKE, FAKE, 66, s) == 1
    # K_out without K
    assert lib.qsa_gather_kv(None, None, 1, 100, 4, 128, 128, 512, 512, FAKE, FAKE, 1, 16, None,
                             100, FAKE, None, FAKE, FAKE, 67, s) == 1
    # decode without n_ctx
    assert lib.qsa_gather_kv(None, None, 1, 100, 4, 128, 128, 512, 512, FAKE, FAKE, 1, 16, None,
                             -1, None, None, FAKE, FAKE, 67, s) == 1


def test_sparse_attn_rejects(lib):
    s = None
    a = P(0x10000)
    ok = dict(q=a, n_q=1, H_q=32, H_kv=4, d_k=128, d_v=128, scale=0.1, K=a, V=a, dt=1, n_kv=100,
              ld_k=512, ld_v=512, pos=None, n_cells=a, max_cells=2051, out=a, lse=None,
              ws=a, ws_bytes=1 << 30, st=s)

    def call(**kw):
        v = dict(ok, **kw)
        return lib.qsa_sparse_attn(*v.values())

    assert call(H_kv=3) == 1                 # H_q % H_kv
    assert call(d_k=100) == 1                # not a multiple of 8
    assert call(ld_k=500) == 1               # ld_k < H_kv*d_k
    assert call(K=P(0x10008)) == 1           # K not 16-byte aligned
    # fp32 K/V: the general kernel writes split-K records, so a workspace is required (the
    # bf16 8-head form merges in a cluster and needs none; a valid call would launch)
    assert call(ws_bytes=0, dt=0) == 1       # workspace too small
    assert call(ws_bytes=64, dt=0) == 1
    assert call(H_q=96) == 2                 # 24 heads per KV head: not built
    assert call(H_q=16, H_kv=1, d_k=576, d_v=512, ld_k=576, ld_v=576, dt=0) == 2  # smem
    need = lib.qsa_sparse_attn_workspace_size(1, 32, 4, 128, 2051)
    assert need > 0
    assert lib.qsa_sparse_attn_workspace_size(1024, 32, 4, 128, 2051) == 0  # one split


def test_sparse_attn_union_rejects(lib):
    s = None
    a = P(0x10000)
    ws_need = lib.qsa_sparse_attn_union_workspace_size(1024, 2051)
    assert ws_need > 0
    assert lib.qsa_sparse_attn_union_workspace_size(0, 2051) == 0
    ok = dict(q=a, n_q=1024, H_q=32, H_kv=4, d=128, scale=0.1, K=a, V=a, dt=1, n_kv=256205,
              ld_k=512, ld_v=512, pos=a, n_cells=a, max_cells=2051, out=a, lse=None,
              ws=P(0x20000), ws_bytes=ws_need, st=s)

    def call(**kw):
        v = dict(ok, **kw)
        return lib.qsa_sparse_attn_union(*v.values())

    # every call below fails validation before anything is launched
    assert call(pos=None) == 1                   # null list
    assert call(q=P(0x10008)) == 1               # q not 16-byte aligned
    assert call(n_q=-1) == 1
    assert call(ws_bytes=ws_need - 1) == 1       # workspace too small
    assert call(ws=P(0x20010)) == 1              # workspace not 256-byte aligned
    assert call(dt=0) == 2                       # fp32 K/V: not built
    assert call(d=64) == 2                       # head dim 64: not built
    assert call(H_q=16) == 2                     # 4 query heads per KV head: not built
    assert call(n_kv=(1 << 20) + 4) == 2         # beyond the union builder's bitmap
    assert call(n_kv=3) == 2
    assert call(max_cells=2101) == 2
    assert call(ld_k=500) == 2                   # stride below the row


def test_mask_to_list_rejects(lib):
    s = None
    assert lib.qsa_mask_to_list(None, 1, 64, 64, 8, FAKE, FAKE, None, s) == 1
    assert lib.qsa_mask_to_list(FAKE, 1, 64, 63, 8, FAKE, FAKE, None, s) == 1
    assert lib.qsa_mask_to_list(FAKE, 1, 64, 64, 8, FAKE, FAKE, P(0x10004), s) == 1
    assert lib.qsa_mask_to_list(FAKE, 1, 1 << 31, 1 << 31, 8, FAKE, FAKE, None, s) == 2


def test_mask_sparse_attn_rejects(lib):
    ok = dict(q=FAKE, n_q=4, H_q=16, H_kv=1, d_k=576, d_v=512, scale=0.04, KV=FAKE, dt=1,
              n_kv=32768, ld_kv=576, mask=FAKE, ld_mask=32768, max_list=2048, counts=FAKE,
              out=FAKE, lse=None, st=None)

    def call(**kw):
        v = dict(ok, **kw)
        return lib.qsa_mask_sparse_attn(*v.values())

    assert call(mask=None) == 1
    assert call(out=None) == 1
    assert call(q=P(0x10004)) == 1                       # q not 8-byte aligned
    assert call(ld_mask=100) == 1                        # ld_mask < n_kv
    assert call(max_list=-1) == 1
    assert call(ld_kv=500) == 1                          # ld_kv < d_k
    assert call(dt=7) == 1                               # no such dtype
    assert call(H_q=32, H_kv=2, ld_kv=1152) == 2         # one latent KV head only
    assert call(d_k=128, d_v=128, ld_kv=128) == 2        # not the latent shape
    assert call(dt=0) == 2                               # fp32 rows
    assert call(KV=P(0x10008)) == 2                      # rows not 16-byte aligned
    assert call(n_kv=65537, ld_mask=65537) == 2          # longer than the in-kernel words
    assert call(n_q=0) == 0                              # nothing to launch


def test_mask_sparse_eligibility_rule():
    # devotd.net, section 3: mask present, no bias, no softcap, n_kv >= 4096, n_kv >= 2*max
    assert qsa.mask_sparse_eligible(True, 0.0, 0.0, 32768, 2048)
    assert not qsa.mask_sparse_eligible(False, 0.0, 0.0, 32768, 2048)
    assert not qsa.mask_sparse_eligible(True, 8.0, 0.0, 32768, 2048)
    assert not qsa.mask_sparse_eligible(True, 0.0, 30.0, 32768, 2048)
    assert not qsa.mask_sparse_eligible(True, 0.0, 0.0, 4095, 16)
    assert not qsa.mask_sparse_eligible(True, 0.0, 0.0, 4096, 2049)
    assert qsa.mask_sparse_eligible(True, 0.0, 0.0, 4096, 2048)


def test_decode_step_host_layout_and_validation(lib):
    import ctypes as C

    off = (C.c_int64 * 5)()
    # 3 queries, bf16 raw keys 16x128, bf16 K/V 4x128, 32 query heads
    total = lib.qsa_decode_step_host_layout(3, 1, 16, 128, 1, 4, 128, 32, off)
    assert list(off) == [0, 12288, 15360, 18432, 43008]
    assert total == 43008 + 3 * 32 * 128 * 4
    assert all(o % 16 == 0 for o in off)
    assert lib.qsa_decode_step_host_layout(0, 1, 16, 128, 1, 4, 128, 32, None) == 0
    assert lib.qsa_decode_step_host_layout(3, 9, 16, 128, 1, 4, 128, 32, None) == 0
    ws = lib.qsa_decode_step_workspace_size(3, 32, 4, 128, 2051, 4000)
    wsh = lib.qsa_decode_step_host_workspace_size(3, 32, 4, 128, 2051, 4000, 1, 16, 128, 1)
    assert wsh == ((ws + 255) // 256) * 256 + ((total + 255) // 256) * 256
    st = None
    # every call below fails validation (cap_rows = 4000 matches the sizes above), so
    # nothing is ever enqueued with the fake pointers

    def step(h_in=FAKE, h_out=FAKE, h_lse=None, lse=None, n_ctx=1000, n_kv=1000, ws_bytes=wsh):
        return lib.qsa_decode_step_host(h_in, h_out, h_lse, FAKE, 1, n_ctx, 16, 128, FAKE, 1e-6,
                                        1e4, FAKE, 0, 4000, 0, 3, 0.1, FAKE, 512, FAKE, FAKE,
                                        FAKE, FAKE, 1, n_kv, 4, 128, 512, FAKE, FAKE, 2051, 32,
                                        0.1, FAKE, lse, P(0x100000), ws_bytes, st)

    assert step(h_in=None) == 1
    assert step(h_out=None) == 1
    assert step(h_lse=FAKE) == 1              # host lse without a device lse
    assert step(n_kv=999) == 1                # the new rows would land past the K/V cache
    assert step(ws_bytes=ws) == 1             # no room for the staging area


def test_decode_plan_create_and_validation(lib):
    import ctypes as C

    ws = lib.qsa_decode_step_workspace_size(3, 32, 4, 128, 2051, 4000)
    wsh = lib.qsa_decode_step_host_workspace_size(3, 32, 4, 128, 2051, 4000, 1, 16, 128, 1)
    WS = P(0x100000)

    def create(handle, max_queries=3, ws_bytes=wsh, raw_dtype=1, K=FAKE, workspace=WS):
        # bf16 raw keys 16x128, fp32 pooled cache of 4000 rows, bf16 K/V 4x128, 32 query heads
        return lib.qsa_decode_plan_create(handle, FAKE, raw_dtype, 16, 128, FAKE, 1e-6, 1e4,
                                          FAKE, 0, 4000, max_queries, 0.1, FAKE, 512, FAKE, FAKE,
                                          K, FAKE, 1, 16000, 4, 128, 512, FAKE, FAKE, 2051, 32,
                                          0.1, FAKE, FAKE, workspace, ws_bytes)

    h = P(0x1234)
    assert create(None) == 1
    for bad in (dict(max_queries=0), dict(max_queries=5), dict(ws_bytes=ws - 1),
                dict(raw_dtype=9), dict(K=None), dict(workspace=P(0x100010))):
        assert create(C.byref(h), **bad) == 1, bad
        assert h.value is None  # *plan is cleared on failure
    lib.qsa_decode_plan_destroy(None)
    # host objects only: creating and destroying a plan touches no device
    plan, plan_dev_only = P(), P()
    assert create(C.byref(plan)) == 0 and plan.value
    assert create(C.byref(plan_dev_only), ws_bytes=ws) == 0 and plan_dev_only.value
    st = None
    try:
        # every step below fails validation before anything is enqueued
        assert lib.qsa_decode_plan_step(None, 1000, 0, 1, FAKE, FAKE, st) == 1
        assert lib.qsa_decode_plan_step(plan, 1000, 0, 4, FAKE, FAKE, st) == 1  # > max_queries
        assert lib.qsa_decode_plan_step(plan, 1000, 0, 0, FAKE, FAKE, st) == 1
        assert lib.qsa_decode_plan_step(plan, 16004, 0, 1, FAKE, FAKE, st) == 1  # 4001 rows
        assert lib.qsa_decode_plan_step(plan, 1000, 0, 1, None, FAKE, st) == 1  # no q_idx
        assert lib.qsa_decode_plan_step_host(None, 1000, 0, 1, FAKE, FAKE, None, st) == 1
        assert lib.qsa_decode_plan_step_host(plan, 1000, 0, 4, FAKE, FAKE, None, st) == 1
        assert lib.qsa_decode_plan_step_host(plan, 1000, 0, 1, None, FAKE, None, st) == 1
        assert lib.qsa_decode_plan_step_host(plan, 1000, 0, 1, FAKE, None, None, st) == 1
        assert lib.qsa_decode_plan_step_host(plan, 16004, 0, 1, FAKE, FAKE, None, st) == 1
        # a plan whose workspace holds no staging area takes no host-fed steps
        assert lib.qsa_decode_plan_step_host(plan_dev_only, 1000, 0, 1, FAKE, FAKE, None,
                                             st) == 1
    finally:
        lib.qsa_decode_plan_destroy(plan)
        lib.qsa_decode_plan_destroy(plan_dev_only)
