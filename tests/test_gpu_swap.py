"""Set-difference-driven block swap into a GPU block cache, through the C ABI.

Over multi-step decode runs, after each step's swap: the cache bookkeeping (slot of
every block, block of every slot, cache page table) equals the oracle's exactly, the
cached pages equal the host pool's bytes, and attention over the cache equals
attention over the full pool (bitwise for the separate calls: same values, same split
plan)."""

import numpy as np
import pytest
import torch

from long_context_serving_gb300 import bsattn as B
from long_context_serving_gb300.build import build
from long_context_serving_gb300.layer import PagedLayer
from oracle import bsattn_oracle as O
from workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build()
    B.lib()


class Cache:
    """Device buffers of a block cache with `slots` slots of `pps` pages per unit."""

    def __init__(self, layer: PagedLayer, slots: int, pps: int):
        wl, dev = layer.wl, layer.device
        n = wl.U * slots * pps
        self.k = torch.full((n, 16, wl.d), float("nan"), dtype=layer.k_pool.dtype, device=dev)
        self.v = torch.full_like(self.k, float("nan"))
        self.pt = torch.full_like(layer.page_table, -1)
        self.slot_block = torch.full((wl.U, slots), -1, dtype=torch.int32, device=dev)
        self.block_slot = torch.full((wl.U, layer.max_blocks), -1, dtype=torch.int32, device=dev)
        self.c = B.BlockCache(k_pool=self.k.data_ptr(), v_pool=self.v.data_ptr(), page_table=self.pt.data_ptr(),
                              slot_block=self.slot_block.data_ptr(), block_slot=self.block_slot.data_ptr(),
                              slots_per_unit=slots, pages_per_slot=pps)
        self.dims = B.Dims.from_buffer_copy(layer.dims)
        self.dims.n_pages = n
        self.ws = torch.zeros_like(layer.workspace)
        self.slots, self.pps = slots, pps

    def kv(self, seq_lens) -> B.KV:
        return B.KV(k_pool=self.k.data_ptr(), v_pool=self.v.data_ptr(), page_table=self.pt.data_ptr(),
                    seq_lens=seq_lens.data_ptr())


def host_pool(layer: PagedLayer):
    """Pinned host copies of the layer's pools (device-readable under unified addressing)."""
    hk = layer.k_pool.cpu().pin_memory()
    hv = layer.v_pool.cpu().pin_memory()
    return hk, hv, B.HostKV(k_pool=hk.data_ptr(), v_pool=hv.data_ptr(), page_table=layer.page_table.data_ptr(),
                            n_pages=int(layer.wl.n_pages))


CASES = {"dual-B2-T2000x8": (5, dict(B=2, T=2000, steps=8)),
         "mixed-g-B1-T9000x6": (3, dict(B=1, T=9000, steps=6)),
         "llama-T5000x3": (2, dict(T=5000, steps=3))}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("fused", [False, True])
def test_swap_cache_matches_oracle_and_full_pool(name, fused):
    cfg_id, kw = CASES[name]
    wl = make_workload(cfg_id, seed=21, **kw)
    layer = PagedLayer(wl, preload_all=True)
    layer.prefill()
    torch.cuda.synchronize()
    slots = layer.max_sel
    pps = int(wl.g.max()) // 16
    cache = Cache(layer, slots, pps)
    hk, hv, host = host_pool(layer)
    sb_ref = [np.full(slots, -1) for _ in range(wl.U)]
    bs_ref = [np.full(layer.max_blocks, -1) for _ in range(wl.U)]
    out2, lse2 = torch.zeros_like(layer.out), torch.zeros_like(layer.lse)
    for step in range(wl.steps):
        cur = layer.cur
        (layer.fused_step if fused else layer.step)(step)
        B.block_swap(layer.dims, layer.cfg, layer.seq_lens[step], host, cache.c, layer.added, layer.added_cnt,
                     layer.removed, layer.removed_cnt, layer.status)
        B.sparse_decode_attn(cache.dims, layer.q[step], cache.kv(layer.seq_lens[step]), layer.cfg, layer.sel[cur],
                             layer.cnt[cur], out2, lse2, cache.ws, layer.status)
        torch.cuda.synchronize()
        assert layer.read_status() == 0, step
        # attention over the cache equals attention over the full pool
        if fused:
            assert (out2 - layer.out).abs().max().item() <= 1e-5 and (lse2 - layer.lse).abs().max().item() <= 1e-5
        else:
            assert torch.equal(out2, layer.out) and torch.equal(lse2, layer.lse), step
        # bookkeeping equals the oracle's
        added = layer.added.cpu().numpy()
        added_cnt = layer.added_cnt.cpu().numpy()
        removed = layer.removed.cpu().numpy()
        removed_cnt = layer.removed_cnt.cpu().numpy()
        sb = cache.slot_block.cpu().numpy()
        bsl = cache.block_slot.cpu().numpy()
        pt = cache.pt.cpu().numpy()
        sel = layer.selection(cur)
        for u in range(wl.U):
            T = int(wl.T(step, u // wl.Hkv))
            sb_ref[u], bs_ref[u], _ = O.block_swap(sb_ref[u], bs_ref[u], added[u, :added_cnt[u]].tolist(),
                                                   removed[u, :removed_cnt[u]].tolist())
            assert sb[u].tolist() == sb_ref[u].tolist(), (step, u)
            assert bsl[u].tolist() == bs_ref[u].tolist(), (step, u)
            assert sorted(np.flatnonzero(bsl[u] >= 0).tolist()) == sel[u], (step, u)
            row = O.cache_page_table(bs_ref[u], u, int(wl.g[u]), T, pt.shape[1], slots, pps)
            assert pt[u].tolist() == row.tolist(), (step, u)
        # cached pages hold the host pool's bytes
        mask = torch.as_tensor(pt >= 0, device=layer.device)
        dev_pages = cache.pt[mask].long()
        src_pages = layer.page_table[mask].long()
        assert torch.equal(cache.k[dev_pages].view(torch.int16), layer.k_pool[src_pages].view(torch.int16))
        assert torch.equal(cache.v[dev_pages].view(torch.int16), layer.v_pool[src_pages].view(torch.int16))
    del hk, hv


def test_swap_reports_capacity_and_bounds():
    """Too few slots: BS_ERR_CAPACITY and the excess is not cached; nothing faults."""
    wl = make_workload(2, seed=22, T=3000)
    layer = PagedLayer(wl, preload_all=True)
    layer.prefill()
    layer.step(0)
    torch.cuda.synchronize()
    cache = Cache(layer, 4, 2)                       # 4 slots, fewer than every selection
    hk, hv, host = host_pool(layer)
    B.block_swap(layer.dims, layer.cfg, layer.seq_lens[0], host, cache.c, layer.added, layer.added_cnt,
                 layer.removed, layer.removed_cnt, layer.status)
    torch.cuda.synchronize()
    assert layer.read_status() == B.BS_ERR_CAPACITY
    bsl = cache.block_slot.cpu().numpy()
    added = layer.added.cpu().numpy()
    for u in range(wl.U):
        assert sorted(np.flatnonzero(bsl[u] >= 0).tolist()) == added[u, :4].tolist()
    del hk, hv
