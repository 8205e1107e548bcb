"""Device buffers of one attention layer's decode state, laid out for libbsattn.

PyTorch here only allocates device memory, copies inputs in and scatters logical
tokens into the paged pool; every step of the decode path is a libbsattn call.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import bsattn as B


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def _kv_tensor(arr: np.ndarray, dtype: str, device) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)


class PagedLayer:
    """One layer of a workload: paged K/V pools, head configuration, summaries and the
    per-step buffers of the five calls.

    ``workload`` is any object with the fields of ``workloads.Workload`` (shapes, head
    properties, logical K/V/q arrays, eviction logits, page table).
    ``fill``: value written into pool slots that hold no token yet, so that a kernel
    reading past T would show up (NaN by default).
    ``preload_all``: put every token of every step in the pool now (otherwise tokens
    enter the pool when their step appends them).
    ``q_fp32``: pass the queries as fp32 (the same values, widened) over a bf16 cache.
    """

    def __init__(self, wl, device="cuda", fill=float("nan"), preload_all=False, q_fp32=False, ed_dma=False):
        self.wl = wl
        # ED-DMA attention: the eviction logits also enter the attention as block logits.
        self.ed_dma = bool(ed_dma)
        self.device = torch.device(device)
        U, d, G = wl.U, wl.d, wl.G
        T_cap = wl.T_cap
        g = wl.g.astype(np.int64)
        s = wl.s.astype(np.int64)
        max_pages = int(wl.page_table.shape[1])
        n_sink = np.array([_cdiv(int(wl.sink[u]), int(g[u])) for u in range(U)])
        n_local = np.array([_cdiv(int(wl.local[u]), int(g[u])) + 1 for u in range(U)])
        n_blk_cap = np.array([_cdiv(T_cap, int(g[u])) for u in range(U)])
        sel_u = np.minimum(n_sink + n_local + wl.k.astype(np.int64), n_blk_cap)
        self.max_sel = int(sel_u.max())
        self.max_blocks = int(n_blk_cap.max())
        sub_rows = np.array([_cdiv(T_cap, int(s[u])) for u in range(U)], dtype=np.int64)
        self.dims = B.Dims(batch=wl.B, n_q_heads=wl.Hq, n_kv_heads=wl.Hkv, head_dim=d, page_size=16,
                           max_pages_per_unit=max_pages, max_blocks_per_unit=self.max_blocks,
                           max_sel_per_unit=self.max_sel, max_subs_per_unit=int(sub_rows.max()),
                           max_gather_pages_per_unit=int((sel_u * g // 16).max()), n_pages=int(wl.n_pages),
                           kv_dtype=B.BS_BF16 if wl.dtype == "bf16" else B.BS_FP32,
                           q_dtype=B.BS_BF16 if wl.dtype == "bf16" and not q_fp32 else B.BS_FP32)

        dev = self.device
        i32 = lambda a: torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32), device=dev)  # noqa: E731
        # Head configuration (struct of arrays) and summary offsets.
        sum_off = np.zeros(U, dtype=np.int64)
        sum_off[1:] = np.cumsum(sub_rows * d)[:-1]
        self.cfg_arrays = dict(cls=i32(wl.cls), block_tokens=i32(wl.g), sub_tokens=i32(wl.s), k_total=i32(wl.k),
                               k_evict=i32(wl.k_e), sink_tokens=i32(wl.sink), local_tokens=i32(wl.local),
                               sum_off=torch.as_tensor(sum_off, device=dev), sum_rows=i32(sub_rows))
        self.cfg = B.HeadCfg(**{k: v.data_ptr() for k, v in self.cfg_arrays.items()})
        host = dict(cls=wl.cls, block_tokens=wl.g, sub_tokens=wl.s, k_total=wl.k, k_evict=wl.k_e,
                    sink_tokens=wl.sink, local_tokens=wl.local, sum_off=sum_off, sum_rows=sub_rows)
        self._cfg_host = {k: np.ascontiguousarray(v, dtype=np.int64 if k == "sum_off" else np.int32)
                          for k, v in host.items()}
        cfg_host = B.HeadCfg(**{k: v.ctypes.data for k, v in self._cfg_host.items()})
        T_last = (wl.T_prefill + wl.steps).astype(np.int32)
        st = B.check_head_cfg(self.dims, cfg_host, T_last)
        if st != B.BS_OK:
            raise B.BsError("bs_check_head_cfg", st, B.status_string(st))

        # Paged pools.
        kv_dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        self.page_table = i32(wl.page_table)
        self.k_pool = torch.full((wl.n_pages, 16, d), fill, dtype=kv_dt, device=dev)
        self.v_pool = torch.full((wl.n_pages, 16, d), fill, dtype=kv_dt, device=dev)
        self._pt_long = self.page_table.long()
        self._K = _kv_tensor(wl.K, wl.dtype, dev)          # logical [U][T_cap][d], source of appends
        self._V = _kv_tensor(wl.V, wl.dtype, dev)
        upto = np.full(wl.B, T_cap, np.int64) if preload_all else wl.T_prefill.astype(np.int64)
        self._write_tokens(np.zeros(wl.B, np.int64), upto)

        self.q = _kv_tensor(wl.q, wl.dtype, dev)           # [steps][B][Hq][d]
        if q_fp32:
            self.q = self.q.float().contiguous()
        self.seq_lens = i32(np.stack([wl.T_prefill + i + 1 for i in range(wl.steps)]))  # [steps][B]
        self.tok_begin = self.seq_lens - 1
        self.prefill_lens = i32(wl.T_prefill)
        self.zeros_b = torch.zeros(wl.B, dtype=torch.int32, device=dev)
        self.kv = B.KV(k_pool=self.k_pool.data_ptr(), v_pool=self.v_pool.data_ptr(),
                       page_table=self.page_table.data_ptr(), seq_lens=0)

        # Per-step state and outputs.
        MB, MS = self.max_blocks, self.max_sel
        self.summaries = torch.full((int(sub_rows.sum()) * d,), float("nan"), dtype=torch.float32, device=dev)
        self.scores = torch.zeros((U, MB), dtype=torch.float32, device=dev)
        self.evict = None
        self.alive = None
        if wl.evict is not None:
            ev = np.full((U, MB), -np.inf, np.float32)
            ev[:, :wl.evict.shape[1]] = wl.evict[:, :MB]
            self.evict = torch.as_tensor(ev, device=dev)
            self.alive = torch.ones((U, MB), dtype=torch.uint8, device=dev)
        if self.ed_dma and self.evict is None:
            raise ValueError("ED-DMA attention needs a workload with eviction logits")
        self.sel = [torch.full((U, MS), -1, dtype=torch.int32, device=dev) for _ in range(2)]
        self.cnt = [torch.zeros(U, dtype=torch.int32, device=dev) for _ in range(2)]
        self.cur = 0                                         # index of the buffer the next select writes
        self.added = torch.full((U, MS), -1, dtype=torch.int32, device=dev)
        self.added_cnt = torch.zeros(U, dtype=torch.int32, device=dev)
        self.removed = torch.full((U, MS), -1, dtype=torch.int32, device=dev)
        self.removed_cnt = torch.zeros(U, dtype=torch.int32, device=dev)
        self.out = torch.zeros((wl.B, wl.Hq, d), dtype=torch.float32, device=dev)
        self.lse = torch.zeros((wl.B, wl.Hq), dtype=torch.float32, device=dev)
        self.workspace = torch.zeros(max(B.workspace_size(self.dims) // 4, 4), dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    # -- caller-side KV writes (not a step of the method) --------------------------
    def _write_tokens(self, lo: np.ndarray, hi: np.ndarray) -> None:
        """Copy logical tokens [lo[b], hi[b]) of every unit into their pool pages."""
        wl = self.wl
        for b in range(wl.B):
            if hi[b] <= lo[b]:
                continue
            t = torch.arange(int(lo[b]), int(hi[b]), device=self.device)
            for u in range(b * wl.Hkv, (b + 1) * wl.Hkv):
                phys = self._pt_long[u, t // 16]
                self.k_pool[phys, t % 16] = self._K[u, t]
                self.v_pool[phys, t % 16] = self._V[u, t]

    def append(self, step: int) -> None:
        """Write the token appended at ``step`` (position T_prefill + step) into the pools."""
        lo = self.wl.T_prefill.astype(np.int64) + step
        self._write_tokens(lo, lo + 1)

    # -- the five calls ------------------------------------------------------------
    def kv_at(self, seq_lens: torch.Tensor) -> B.KV:
        return B.KV(k_pool=self.kv.k_pool, v_pool=self.kv.v_pool, page_table=self.kv.page_table,
                    seq_lens=seq_lens.data_ptr())

    def prefill(self, stream=None) -> None:
        """Summaries of every prefilled token."""
        max_new = int(self.wl.T_prefill.max())
        if max_new == 0:       # an empty cache: the first decode step's update covers token 0
            return
        B.build_block_summaries(self.dims, self.kv_at(self.prefill_lens), self.cfg, self.zeros_b, max(max_new, 1),
                                self.summaries, self.status, stream)

    def update_summaries(self, step: int, stream=None) -> None:
        """Recompute the sub-block holding the token appended at ``step``."""
        B.build_block_summaries(self.dims, self.kv_at(self.seq_lens[step]), self.cfg, self.tok_begin[step], 1,
                                self.summaries, self.status, stream)

    def score(self, step: int, group_reduce=B.BS_GROUP_MAX, stream=None) -> None:
        B.score_blocks(self.dims, self.q[step], self.cfg, self.seq_lens[step], self.summaries, group_reduce,
                       self.scores, self.status, stream)

    def select(self, step: int, stream=None) -> None:
        B.select_topk(self.dims, self.cfg, self.seq_lens[step], self.scores, self.evict, self.alive,
                      self.sel[self.cur], self.cnt[self.cur], self.status, stream)

    def attend(self, step: int, stream=None) -> None:
        B.sparse_decode_attn(self.dims, self.q[step], self.kv_at(self.seq_lens[step]), self.cfg, self.sel[self.cur],
                             self.cnt[self.cur], self.out, self.lse, self.workspace, self.status, stream,
                             evict_bias=self.evict if self.ed_dma else None)

    def setdiff(self, stream=None) -> None:
        prev = 1 - self.cur
        B.block_setdiff(self.dims, self.sel[prev], self.cnt[prev], self.sel[self.cur], self.cnt[self.cur],
                        self.added, self.added_cnt, self.removed, self.removed_cnt, self.status, stream)

    def step_io(self, step: int) -> B.StepIO:
        """Buffers of bs_decode_step for ``step`` (current selection buffer ``self.cur``)."""
        prev = 1 - self.cur
        ptr = lambda t: 0 if t is None else t.data_ptr()  # noqa: E731
        return B.StepIO(q=self.q[step].data_ptr(), summaries=self.summaries.data_ptr(),
                        scores=self.scores.data_ptr(), evict_logits=ptr(self.evict), alive=ptr(self.alive),
                        evict_bias=ptr(self.evict) if self.ed_dma else 0,
                        prev_idx=self.sel[prev].data_ptr(), prev_cnt=self.cnt[prev].data_ptr(),
                        cur_idx=self.sel[self.cur].data_ptr(), cur_cnt=self.cnt[self.cur].data_ptr(),
                        added=self.added.data_ptr(), added_cnt=self.added_cnt.data_ptr(),
                        removed=self.removed.data_ptr(), removed_cnt=self.removed_cnt.data_ptr(),
                        out=self.out.data_ptr(), lse=self.lse.data_ptr(), workspace=self.workspace.data_ptr(),
                        workspace_bytes=self.workspace.numel() * 4, dev_status=self.status.data_ptr())

    def fused_step(self, step: int, group_reduce=B.BS_GROUP_MAX, stream=None) -> None:
        """The same decode step through bs_decode_step (two launches), then advance."""
        B.decode_step(self.dims, self.kv_at(self.seq_lens[step]), self.cfg, self.step_io(step), group_reduce,
                      stream)
        self.advance()

    def advance(self) -> None:
        """The current selection becomes the previous one."""
        self.cur = 1 - self.cur

    def step(self, step: int, group_reduce=B.BS_GROUP_MAX, stream=None) -> None:
        """One decode step of this layer (after the caller appended its KV): a1 update,
        a2 scores, a3 selection, a4 attention, a5 set-difference."""
        self.update_summaries(step, stream)
        self.score(step, group_reduce, stream)
        self.select(step, stream)
        self.attend(step, stream)
        self.setdiff(stream)
        self.advance()

    # -- host views ----------------------------------------------------------------
    def set_selection(self, lists: dict, which: int | None = None) -> None:
        """Overwrite selections of some units (unit -> ascending block list)."""
        which = self.cur if which is None else which
        sel = self.sel[which].cpu()
        cnt = self.cnt[which].cpu()
        for u, lst in lists.items():
            sel[u] = -1
            sel[u, :len(lst)] = torch.as_tensor(list(lst), dtype=torch.int32)
            cnt[u] = len(lst)
        self.sel[which].copy_(sel)
        self.cnt[which].copy_(cnt)

    def selection(self, which: int) -> list:
        sel = self.sel[which].cpu().numpy()
        cnt = self.cnt[which].cpu().numpy()
        return [sel[u, :cnt[u]].tolist() for u in range(self.wl.U)]

    def unit_summaries(self, u: int, rows: int) -> np.ndarray:
        off = int(self._cfg_host["sum_off"][u])
        d = self.wl.d
        return self.summaries[off:off + rows * d].view(rows, d).cpu().numpy()

    def read_status(self) -> int:
        return int(self.status.item())
