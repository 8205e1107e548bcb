"""Thin ctypes binding of libbsattn.so (include/bsattn.h).

Argument marshalling only: every step of the decode path runs in the library's
CUDA kernels. Tensors are passed as raw device pointers; the stream is the
caller's current torch stream unless one is given. A missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbsattn.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "bsattn.h")

# bs_status
BS_OK = 0
BS_ERR_INVALID_ARG = 1
BS_ERR_SHAPE = 2
BS_ERR_ALIGN = 3
BS_ERR_CAPACITY = 4
BS_ERR_CUDA = 5
BS_ERR_DEVICE_BOUNDS = 6
BS_ERR_TIMEOUT = 7
# bs_dtype, bs_head_class, bs_group_reduce
BS_BF16, BS_FP32 = 0, 1
BS_STREAMING, BS_RETRIEVAL, BS_DUAL = 0, 1, 2
BS_GROUP_MAX, BS_GROUP_MEAN = 0, 1


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages_per_unit", ctypes.c_int32), ("max_blocks_per_unit", ctypes.c_int32),
                ("max_sel_per_unit", ctypes.c_int32), ("max_subs_per_unit", ctypes.c_int32),
                ("max_gather_pages_per_unit", ctypes.c_int32), ("n_pages", ctypes.c_int64),
                ("kv_dtype", ctypes.c_int), ("q_dtype", ctypes.c_int)]


class KV(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p)]


class HeadCfg(ctypes.Structure):
    _fields_ = [("cls", ctypes.c_void_p), ("block_tokens", ctypes.c_void_p), ("sub_tokens", ctypes.c_void_p),
                ("k_total", ctypes.c_void_p), ("k_evict", ctypes.c_void_p), ("sink_tokens", ctypes.c_void_p),
                ("local_tokens", ctypes.c_void_p), ("sum_off", ctypes.c_void_p), ("sum_rows", ctypes.c_void_p)]


class StepIO(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("summaries", ctypes.c_void_p), ("scores", ctypes.c_void_p),
                ("evict_logits", ctypes.c_void_p), ("alive", ctypes.c_void_p), ("evict_bias", ctypes.c_void_p),
                ("prev_idx", ctypes.c_void_p),
                ("prev_cnt", ctypes.c_void_p), ("cur_idx", ctypes.c_void_p), ("cur_cnt", ctypes.c_void_p),
                ("added", ctypes.c_void_p), ("added_cnt", ctypes.c_void_p), ("removed", ctypes.c_void_p),
                ("removed_cnt", ctypes.c_void_p), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("dev_status", ctypes.c_void_p)]


class HostKV(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("n_pages", ctypes.c_int64)]


class BlockCache(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("slot_block", ctypes.c_void_p), ("block_slot", ctypes.c_void_p),
                ("slots_per_unit", ctypes.c_int32), ("pages_per_slot", ctypes.c_int32)]


class HostTables(ctypes.Structure):
    _fields_ = [("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p), ("block_tokens", ctypes.c_void_p),
                ("evict_bias", ctypes.c_void_p), ("max_blocks_per_unit", ctypes.c_int32)]


class BsError(RuntimeError):
    def __init__(self, call: str, status: int, text: str):
        super().__init__(f"{call} returned {status} ({text})")
        self.status = status


_P = ctypes.POINTER
_SIGS = {
    "bs_check_head_cfg": (ctypes.c_int, [_P(Dims), _P(HeadCfg), ctypes.c_void_p]),
    "bs_build_block_summaries": (ctypes.c_int, [_P(Dims), _P(KV), _P(HeadCfg), ctypes.c_void_p, ctypes.c_int32,
                                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "bs_score_blocks": (ctypes.c_int, [_P(Dims), ctypes.c_void_p, _P(HeadCfg), ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "bs_select_topk": (ctypes.c_int, [_P(Dims), _P(HeadCfg), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p]),
    "bs_sparse_decode_attn": (ctypes.c_int, [_P(Dims), ctypes.c_void_p, _P(KV), _P(HeadCfg), ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "bs_block_setdiff": (ctypes.c_int, [_P(Dims), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "bs_sparse_decode_attn_noalloc": (ctypes.c_int, [_P(Dims), ctypes.c_void_p, _P(KV), _P(HeadCfg),
                                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                     ctypes.c_void_p]),
    "bs_decode_step": (ctypes.c_int, [_P(Dims), _P(KV), _P(HeadCfg), _P(StepIO), ctypes.c_int, ctypes.c_void_p]),
    "bs_block_swap": (ctypes.c_int, [_P(Dims), _P(HeadCfg), ctypes.c_void_p, _P(HostKV), _P(BlockCache),
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_void_p]),
    "bs_cpu_sparse_attn": (ctypes.c_int, [_P(Dims), ctypes.c_void_p, _P(HostKV), _P(HostTables), ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]),
    "bs_lse_merge": (ctypes.c_int, [_P(Dims), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "bs_workspace_size": (ctypes.c_size_t, [_P(Dims)]),
    "bs_decode_step_launches": (ctypes.c_int, [_P(Dims)]),
    "bs_set_wait_limit_ns": (ctypes.c_int, [ctypes.c_uint64]),
    "bs_wait_limit_ns": (ctypes.c_uint64, []),
    "bs_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library. Raises when it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; build it with long_context_serving_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/bsattn.h declares."""
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bs_[a-z_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return lib().bs_status_string(status).decode()


def _check(call: str, status: int) -> None:
    if status != BS_OK:
        raise BsError(call, status, status_string(status))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data          # a numpy array (host memory)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def check_head_cfg(dims: Dims, cfg_host: HeadCfg, seq_lens_host) -> int:
    """Host-side check of a head configuration held in host memory; returns the status."""
    return lib().bs_check_head_cfg(ctypes.byref(dims), ctypes.byref(cfg_host), _ptr(seq_lens_host))


def build_block_summaries(dims, kv, cfg, tok_begin, max_new_tokens, summaries, dev_status, stream=None):
    _check("bs_build_block_summaries",
           lib().bs_build_block_summaries(ctypes.byref(dims), ctypes.byref(kv), ctypes.byref(cfg), _ptr(tok_begin),
                                          int(max_new_tokens), _ptr(summaries), _ptr(dev_status), _stream(stream)))


def score_blocks(dims, q, cfg, seq_lens, summaries, group_reduce, scores, dev_status, stream=None):
    _check("bs_score_blocks",
           lib().bs_score_blocks(ctypes.byref(dims), _ptr(q), ctypes.byref(cfg), _ptr(seq_lens), _ptr(summaries),
                                 int(group_reduce), _ptr(scores), _ptr(dev_status), _stream(stream)))


def select_topk(dims, cfg, seq_lens, scores, evict_logits, alive, sel_idx, sel_cnt, dev_status, stream=None):
    _check("bs_select_topk",
           lib().bs_select_topk(ctypes.byref(dims), ctypes.byref(cfg), _ptr(seq_lens), _ptr(scores),
                                _ptr(evict_logits), _ptr(alive), _ptr(sel_idx), _ptr(sel_cnt), _ptr(dev_status),
                                _stream(stream)))


def sparse_decode_attn(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, workspace, dev_status, stream=None,
                       evict_bias=None):
    """a4. evict_bias (None: plain softmax) is the ED-DMA logit bias of every block,
    fp32 [units][max_blocks_per_unit] on the device."""
    nbytes = workspace.numel() * workspace.element_size()
    _check("bs_sparse_decode_attn",
           lib().bs_sparse_decode_attn(ctypes.byref(dims), _ptr(q), ctypes.byref(kv), ctypes.byref(cfg),
                                       _ptr(sel_idx), _ptr(sel_cnt), _ptr(evict_bias), _ptr(out), _ptr(lse),
                                       _ptr(workspace), nbytes, _ptr(dev_status), _stream(stream)))


def block_setdiff(dims, prev_idx, prev_cnt, cur_idx, cur_cnt, added, added_cnt, removed, removed_cnt, dev_status,
                  stream=None):
    _check("bs_block_setdiff",
           lib().bs_block_setdiff(ctypes.byref(dims), _ptr(prev_idx), _ptr(prev_cnt), _ptr(cur_idx), _ptr(cur_cnt),
                                  _ptr(added), _ptr(added_cnt), _ptr(removed), _ptr(removed_cnt), _ptr(dev_status),
                                  _stream(stream)))


def sparse_decode_attn_noalloc(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, dev_status, stream=None,
                               evict_bias=None):
    """bs_sparse_decode_attn for callers that cannot allocate a workspace: the library's
    fixed per-device scratch array stands in for it (see include/bsattn.h)."""
    _check("bs_sparse_decode_attn_noalloc",
           lib().bs_sparse_decode_attn_noalloc(ctypes.byref(dims), _ptr(q), ctypes.byref(kv), ctypes.byref(cfg),
                                               _ptr(sel_idx), _ptr(sel_cnt), _ptr(evict_bias), _ptr(out),
                                               _ptr(lse), _ptr(dev_status), _stream(stream)))


def decode_step(dims, kv, cfg, io: StepIO, group_reduce=BS_GROUP_MAX, stream=None):
    """All five steps of one layer's decode step (two launches)."""
    _check("bs_decode_step", lib().bs_decode_step(ctypes.byref(dims), ctypes.byref(kv), ctypes.byref(cfg),
                                                  ctypes.byref(io), int(group_reduce), _stream(stream)))


def block_swap(dims, cfg, seq_lens, host: HostKV, cache: BlockCache, added, added_cnt, removed, removed_cnt,
               dev_status, stream=None):
    """Move the blocks the set-difference adds from host memory into the GPU block cache."""
    _check("bs_block_swap",
           lib().bs_block_swap(ctypes.byref(dims), ctypes.byref(cfg), _ptr(seq_lens), ctypes.byref(host),
                               ctypes.byref(cache), _ptr(added), _ptr(added_cnt), _ptr(removed), _ptr(removed_cnt),
                               _ptr(dev_status), _stream(stream)))


def cpu_sparse_attn(dims, q, kv: HostKV, tables: HostTables, sel_idx, sel_cnt, out, lse, n_threads: int):
    """Attention of the listed blocks on the host cores (every buffer in host memory)."""
    _check("bs_cpu_sparse_attn",
           lib().bs_cpu_sparse_attn(ctypes.byref(dims), _ptr(q), ctypes.byref(kv), ctypes.byref(tables),
                                    _ptr(sel_idx), _ptr(sel_cnt), _ptr(out), _ptr(lse), int(n_threads)))


def lse_merge(dims, out_a, lse_a, out_b, lse_b, out, lse, stream=None):
    """Merge two partial attention results over disjoint token sets (device memory)."""
    _check("bs_lse_merge", lib().bs_lse_merge(ctypes.byref(dims), _ptr(out_a), _ptr(lse_a), _ptr(out_b),
                                              _ptr(lse_b), _ptr(out), _ptr(lse), _stream(stream)))


def workspace_size(dims) -> int:
    return int(lib().bs_workspace_size(ctypes.byref(dims)))


def decode_step_launches(dims) -> int:
    """Kernels one decode_step call launches for these dims (0 on bad dims)."""
    return int(lib().bs_decode_step_launches(ctypes.byref(dims)))


def set_wait_limit_ns(limit_ns: int) -> None:
    """Limit of every device-side wait of the calls launched from now on (default 1 s)."""
    _check("bs_set_wait_limit_ns", lib().bs_set_wait_limit_ns(int(limit_ns)))


def wait_limit_ns() -> int:
    return int(lib().bs_wait_limit_ns())
