"""The C-ABI library on the host: it loads, exports what include/bsattn.h declares, and
rejects bad arguments with the documented status before launching anything. Nothing
here touches a GPU: every call below returns during host-side validation."""
import ctypes

import numpy as np
import pytest

from long_context_serving_gb300 import bsattn as B
from long_context_serving_gb300.build import build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    return B.lib()


def test_exports_every_declared_function():
    names = B.header_functions()
    assert {"bs_build_block_summaries", "bs_score_blocks", "bs_select_topk", "bs_sparse_decode_attn",
            "bs_block_setdiff", "bs_workspace_size", "bs_status_string", "bs_check_head_cfg"} <= set(names)
    for n in names:
        assert hasattr(B.lib(), n), n


def test_status_strings():
    for code in range(8):
        assert B.status_string(code) not in ("", "unknown status")
    assert B.status_string(99) == "unknown status"


def _dims(**kw):
    base = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=16, max_pages_per_unit=64,
                max_blocks_per_unit=32, max_sel_per_unit=16, max_subs_per_unit=128, max_gather_pages_per_unit=32,
                n_pages=128, kv_dtype=B.BS_BF16, q_dtype=B.BS_BF16)
    base.update(kw)
    return B.Dims(**base)


def test_workspace_size():
    d = _dims()
    ws = B.workspace_size(d)
    assert ws > 0 and ws % 16 == 0
    assert B.workspace_size(_dims(batch=4)) == 2 * ws
    for bad in (dict(head_dim=96), dict(page_size=32), dict(n_q_heads=9), dict(n_q_heads=18),
                dict(batch=0), dict(max_blocks_per_unit=20000), dict(kv_dtype=7)):
        assert B.workspace_size(_dims(**bad)) == 0, bad


def test_pool_rows_stay_below_two_to_the_31():
    """Pool rows (16 per page) are signed 32-bit tensor-map coordinates: a pool of 2^27
    pages (2^31 rows) is refused on the host by every call, one page fewer is accepted."""
    assert B.workspace_size(_dims(n_pages=(1 << 27) - 1)) > 0
    big = _dims(n_pages=1 << 27)
    assert B.workspace_size(big) == 0
    L = B.lib()
    kv = B.KV(k_pool=0x10000, v_pool=0x20000, page_table=0x30000, seq_lens=0x40000)
    cfg = B.HeadCfg(*([0x50000] * 9))
    ref = ctypes.byref
    assert L.bs_sparse_decode_attn(ref(big), 0x1000, ref(kv), ref(cfg), 0x2000, 0x3000, None, 0x4000, 0x5000, 0x8000,
                                   1 << 30, 0x6000, None) == B.BS_ERR_CAPACITY
    assert L.bs_sparse_decode_attn_noalloc(ref(big), 0x1000, ref(kv), ref(cfg), 0x2000, 0x3000, None, 0x4000,
                                           0x5000, 0x6000, None) == B.BS_ERR_CAPACITY
    assert L.bs_build_block_summaries(ref(big), ref(kv), ref(cfg), 0x1000, 1, 0x70000, 0x6000, None) == \
        B.BS_ERR_CAPACITY


def _ws(units, G, max_gather, kv=B.BS_BF16):
    return B.workspace_size(_dims(batch=1, n_kv_heads=units, n_q_heads=G * units,
                                  max_gather_pages_per_unit=max_gather, kv_dtype=kv))


def test_workspace_size_modes():
    """Four int32 words per unit (padded to 16 bytes), then per mode as the header states:
    cluster mode the fused step's page lists (4 bytes per gathered page); workspace mode
    32 split records of G x (d + 4) floats per unit. And the 8 MiB limit of the
    no-allocation call that follows from it."""
    def counters(u):
        return (4 * u + 3) // 4 * 4 * 4

    def plist(u, mg):
        return (u * mg + 3) // 4 * 4 * 4

    def workspace(u, G):
        return counters(u) + u * 32 * G * (128 + 4) * 4

    assert _ws(8, 4, 1024) == counters(8) + plist(8, 1024)          # few units: cluster
    assert _ws(19, 4, 1024) == counters(19) + plist(19, 1024)
    assert _ws(20, 4, 256) == counters(20) + plist(20, 256)         # small selections: cluster
    assert _ws(304, 4, 1024) == counters(304) + plist(304, 1024)    # many units: cluster
    assert _ws(8, 4, 1025) == workspace(8, 4)                       # above 1024 pages
    assert _ws(20, 4, 257) == workspace(20, 4)                      # 20..303 units, larger selections
    assert _ws(303, 7, 512) == workspace(303, 7)
    assert _ws(1025, 4, 512) == counters(1025) + plist(1025, 512)   # many units: cluster
    assert _ws(1025, 4, 2048) == workspace(1025, 4)
    # the same rule for fp32 caches
    assert _ws(8, 4, 2048, B.BS_FP32) == workspace(8, 4)
    assert _ws(100, 4, 512, B.BS_FP32) == workspace(100, 4)
    assert _ws(100, 4, 256, B.BS_FP32) == counters(100) + plist(100, 256)
    limit = 8 << 20
    assert _ws(124, 4, 2048) <= limit < _ws(125, 4, 2048)          # workspace mode
    assert _ws(62, 8, 2048) <= limit < _ws(63, 8, 2048)
    assert _ws(2040, 4, 1024) <= limit < _ws(2041, 4, 1024)        # cluster mode


class HostCfg:
    """Head configuration in host memory for bs_check_head_cfg."""

    def __init__(self, U, **kw):
        vals = dict(cls=B.BS_RETRIEVAL, block_tokens=32, sub_tokens=8, k_total=4, k_evict=0, sink_tokens=32,
                    local_tokens=32, sum_off=None, sum_rows=128)
        vals.update(kw)
        self.arrays = {}
        for k, v in vals.items():
            dt = np.int64 if k == "sum_off" else np.int32
            if k == "sum_off" and v is None:
                v = np.arange(U, dtype=np.int64) * 128 * 128
            self.arrays[k] = np.ascontiguousarray(np.broadcast_to(np.asarray(v, dtype=dt), (U,)))
        self.cfg = B.HeadCfg(**{k: a.ctypes.data for k, a in self.arrays.items()})


def _check(dims, U=4, T=1000, **kw):
    hc = HostCfg(U, **kw)
    lens = np.full(dims.batch, T, np.int32)
    return B.check_head_cfg(dims, hc.cfg, lens)


def test_check_head_cfg_rules():
    d = _dims()
    assert _check(d) == B.BS_OK
    assert _check(d, block_tokens=24) == B.BS_ERR_INVALID_ARG          # g % 16
    assert _check(d, sub_tokens=5) == B.BS_ERR_INVALID_ARG             # g % s
    assert _check(d, block_tokens=96, sub_tokens=32) == B.BS_ERR_INVALID_ARG   # g/s = 3
    assert _check(d, block_tokens=1024, sub_tokens=8) == B.BS_ERR_INVALID_ARG  # g/s > 64
    assert _check(d, local_tokens=0) == B.BS_ERR_INVALID_ARG
    assert _check(d, k_total=-1) == B.BS_ERR_INVALID_ARG
    assert _check(d, cls=B.BS_DUAL, k_total=4, k_evict=5) == B.BS_ERR_INVALID_ARG
    assert _check(d, cls=3) == B.BS_ERR_INVALID_ARG
    assert _check(d, sum_off=np.array([0, 6, 12, 18])) == B.BS_ERR_ALIGN
    assert _check(d, sum_rows=100) == B.BS_ERR_CAPACITY                # ceil(1000/8) = 125 rows
    assert _check(d, k_total=20) == B.BS_ERR_CAPACITY                  # more than max_sel
    assert _check(d, T=2000) == B.BS_ERR_CAPACITY                      # more pages than the table row
    assert _check(d, T=0) == B.BS_ERR_INVALID_ARG
    assert B.check_head_cfg(d, HostCfg(4).cfg, None) == B.BS_ERR_INVALID_ARG


def test_calls_reject_bad_arguments_before_launch():
    L = B.lib()
    d = _dims()
    kv = B.KV(k_pool=0x10000, v_pool=0x20000, page_table=0x30000, seq_lens=0x40000)
    cfg = B.HeadCfg(*([0x50000] * 9))
    st = ctypes.c_void_p(0x60000)
    ref = ctypes.byref
    # null pointers
    assert L.bs_build_block_summaries(ref(d), ref(kv), ref(cfg), None, 1, 0x70000, st, None) == B.BS_ERR_INVALID_ARG
    assert L.bs_score_blocks(ref(d), None, ref(cfg), 0x1000, 0x2000, 0, 0x3000, st, None) == B.BS_ERR_INVALID_ARG
    assert L.bs_select_topk(ref(d), ref(cfg), None, 0x1000, None, None, 0x2000, 0x3000, st, None) == \
        B.BS_ERR_INVALID_ARG
    assert L.bs_sparse_decode_attn(ref(d), 0x1000, ref(kv), ref(cfg), 0x2000, 0x3000, None, 0x4000, 0x5000, None,
                                   1 << 30, st, None) == B.BS_ERR_INVALID_ARG
    assert L.bs_block_setdiff(ref(d), 0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, st,
                              None) == B.BS_ERR_INVALID_ARG
    assert L.bs_score_blocks(None, 0x1000, ref(cfg), 0x1000, 0x2000, 0, 0x3000, st, None) == B.BS_ERR_INVALID_ARG
    # bad shapes
    assert L.bs_score_blocks(ref(_dims(head_dim=80)), 0x1000, ref(cfg), 0x1000, 0x2000, 0, 0x3000, st, None) == \
        B.BS_ERR_SHAPE
    assert L.bs_select_topk(ref(_dims(n_q_heads=20)), ref(cfg), 0x1000, 0x1000, None, None, 0x2000, 0x3000, st,
                            None) == B.BS_ERR_SHAPE
    # misaligned pointers
    assert L.bs_sparse_decode_attn(ref(d), 0x1002, ref(kv), ref(cfg), 0x2000, 0x3000, None, 0x4000, 0x5000, 0x8000,
                                   1 << 30, st, None) == B.BS_ERR_ALIGN
    bad_kv = B.KV(k_pool=0x10008, v_pool=0x20000, page_table=0x30000, seq_lens=0x40000)
    assert L.bs_build_block_summaries(ref(d), ref(bad_kv), ref(cfg), 0x1000, 1, 0x70000, st, None) == B.BS_ERR_ALIGN
    assert L.bs_score_blocks(ref(d), 0x1000, ref(cfg), 0x1000, 0x2004, 0, 0x3000, st, None) == B.BS_ERR_ALIGN
    # invalid values
    assert L.bs_score_blocks(ref(d), 0x1000, ref(cfg), 0x1000, 0x2000, 5, 0x3000, st, None) == B.BS_ERR_INVALID_ARG
    assert L.bs_build_block_summaries(ref(d), ref(kv), ref(cfg), 0x1000, 0, 0x70000, st, None) == \
        B.BS_ERR_INVALID_ARG
    # workspace too small
    assert L.bs_sparse_decode_attn(ref(d), 0x1000, ref(kv), ref(cfg), 0x2000, 0x3000, None, 0x4000, 0x5000, 0x8000,
                                   16, st, None) == B.BS_ERR_CAPACITY


def test_offload_and_split_calls_reject_bad_arguments():
    """bs_block_swap, bs_cpu_sparse_attn and bs_lse_merge validate on the host first."""
    L = B.lib()
    ref = ctypes.byref
    d = _dims()
    st = 0x9000
    cfg = B.HeadCfg(cls=0x100, block_tokens=0x200, sub_tokens=0x300, k_total=0x400, k_evict=0x500,
                    sink_tokens=0x600, local_tokens=0x700, sum_off=0x800, sum_rows=0x900)
    host = B.HostKV(k_pool=0x10000, v_pool=0x20000, page_table=0x30000, n_pages=128)
    cache = B.BlockCache(k_pool=0x40000, v_pool=0x50000, page_table=0x60000, slot_block=0x70000,
                         block_slot=0x80000, slots_per_unit=8, pages_per_slot=2)
    swap = L.bs_block_swap
    assert swap(ref(d), ref(cfg), 0x1000, ref(host), ref(cache), None, 0x2000, 0x3000, 0x4000, st,
                None) == B.BS_ERR_INVALID_ARG
    assert swap(ref(d), ref(cfg), 0x1000, ref(B.HostKV(k_pool=0, v_pool=0x20000, page_table=0x30000, n_pages=128)),
                ref(cache), 0x1100, 0x2000, 0x3000, 0x4000, st, None) == B.BS_ERR_INVALID_ARG
    for bad in (dict(slots_per_unit=0), dict(slots_per_unit=5000), dict(pages_per_slot=0)):
        c = B.BlockCache(k_pool=0x40000, v_pool=0x50000, page_table=0x60000, slot_block=0x70000,
                         block_slot=0x80000, **{**dict(slots_per_unit=8, pages_per_slot=2), **bad})
        assert swap(ref(d), ref(cfg), 0x1000, ref(host), ref(c), 0x1100, 0x2000, 0x3000, 0x4000, st,
                    None) == B.BS_ERR_INVALID_ARG, bad
    misaligned = B.BlockCache(k_pool=0x40008, v_pool=0x50000, page_table=0x60000, slot_block=0x70000,
                              block_slot=0x80000, slots_per_unit=8, pages_per_slot=2)
    assert swap(ref(d), ref(cfg), 0x1000, ref(host), ref(misaligned), 0x1100, 0x2000, 0x3000, 0x4000, st,
                None) == B.BS_ERR_ALIGN
    assert swap(ref(_dims(head_dim=80)), ref(cfg), 0x1000, ref(host), ref(cache), 0x1100, 0x2000, 0x3000, 0x4000,
                st, None) == B.BS_ERR_SHAPE
    tables = B.HostTables(page_table=0x1000, seq_lens=0x2000, block_tokens=0x3000)
    assert L.bs_cpu_sparse_attn(ref(d), None, ref(host), ref(tables), 0x4000, 0x5000, 0x6000, 0x7000, 4) == \
        B.BS_ERR_INVALID_ARG
    assert L.bs_cpu_sparse_attn(ref(d), 0x1000, ref(host), ref(B.HostTables(page_table=0, seq_lens=0x2000,
                                                                           block_tokens=0x3000)),
                                0x4000, 0x5000, 0x6000, 0x7000, 4) == B.BS_ERR_INVALID_ARG
    no_row = B.HostTables(page_table=0x1000, seq_lens=0x2000, block_tokens=0x3000, evict_bias=0x8000,
                          max_blocks_per_unit=0)   # block logits without a row length
    assert L.bs_cpu_sparse_attn(ref(d), 0x1000, ref(host), ref(no_row), 0x4000, 0x5000, 0x6000, 0x7000, 4) == \
        B.BS_ERR_INVALID_ARG
    assert L.bs_lse_merge(ref(d), 0x1000, 0x2000, None, 0x4000, 0x5000, 0x6000, None) == B.BS_ERR_INVALID_ARG
    assert L.bs_lse_merge(ref(d), 0x1004, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, None) == B.BS_ERR_ALIGN
    assert L.bs_lse_merge(ref(_dims(page_size=8)), 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, None) == \
        B.BS_ERR_SHAPE


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No fallback: without the built library every call raises."""
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "libbsattn.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        B.lib()
    with pytest.raises(RuntimeError, match="missing"):
        B.workspace_size(_dims())


def test_wait_limit_knob_range():
    """The device-wait limit takes 1 us .. 60 s and keeps its value on a refused call."""
    default = B.wait_limit_ns()
    assert default == 10**9
    assert B.lib().bs_set_wait_limit_ns(0) == B.BS_ERR_INVALID_ARG
    assert B.lib().bs_set_wait_limit_ns(61 * 10**9) == B.BS_ERR_INVALID_ARG
    assert B.wait_limit_ns() == default
    B.set_wait_limit_ns(5000)
    assert B.wait_limit_ns() == 5000
    B.set_wait_limit_ns(default)
