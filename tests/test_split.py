"""CPU/GPU split attention: bs_cpu_sparse_attn (host cores) and bs_lse_merge (GPU).

The CPU side is host code of the library, checked here against the oracle on the CPU;
the GPU test splits every unit's selection between the GPU attention and the CPU,
merges on the GPU and compares with the oracle's attention over the union and with the
GPU's attention over the whole selection."""
import numpy as np
import pytest
import torch

from _parity import ATT_ABS, ATT_REL, LSE_ABS, REL_FLOOR
from long_context_serving_gb300 import bsattn as B
from long_context_serving_gb300.build import build
from long_context_serving_gb300.layer import PagedLayer
from oracle import bsattn_oracle as O
from workloads import make_workload


def _subsets(wl, rng, T_of, MS):
    """Per unit: forced blocks plus random candidates (at most MS blocks in all), then
    a split of that selection into two ascending parts (a: even positions, b: odd)."""
    sel, a, b = {}, {}, {}
    for u in range(wl.U):
        T = T_of(u)
        g = int(wl.g[u])
        F = O.forced_blocks(T, g, int(wl.sink[u]), int(wl.local[u]))
        C = O.candidate_blocks(T, g, int(wl.sink[u]), int(wl.local[u]))
        n = min(len(C), max(0, MS - len(F)), int(rng.integers(0, len(C) + 1)))
        pick = sorted(int(c) for c in rng.choice(C, size=n, replace=False)) if n else []
        s = sorted(set(F) | set(pick))
        sel[u] = s
        a[u] = s[0::2]
        b[u] = s[1::2]
    return sel, a, b


def _rows(lists, U, MS):
    idx = np.full((U, MS), -1, np.int32)
    cnt = np.zeros(U, np.int32)
    for u, l in lists.items():
        idx[u, :len(l)] = l
        cnt[u] = len(l)
    return idx, cnt


def _compare(wl, step, out, lse, lists, T_of):
    for u in range(wl.U):
        T, g = T_of(u), int(wl.g[u])
        b, hk = u // wl.Hkv, u % wl.Hkv
        rows = slice(hk * wl.G, (hk + 1) * wl.G)
        o = np.asarray(out[b, rows], np.float64)
        lv = np.asarray(lse[b, rows], np.float64)
        if not lists[u]:
            assert np.all(o == 0) and np.all(np.isneginf(lv))
            continue
        o_ref, l_ref = O.sparse_attention(wl.q64(step, u), wl.K64(u), wl.V64(u), lists[u], g, T)
        diff = np.abs(o - o_ref)
        assert diff.max() <= ATT_ABS, (u, diff.max())
        assert (diff / np.maximum(np.abs(o_ref), REL_FLOOR)).max() <= ATT_REL, u
        assert np.abs(lv - l_ref).max() <= LSE_ABS, u


@pytest.mark.parametrize("cfg_id,kw", [(3, dict(B=1, T=6000, steps=1)), (1, {})])
def test_cpu_attention_matches_oracle(cfg_id, kw):
    build()
    wl = make_workload(cfg_id, seed=31, **kw)
    layer = PagedLayer(wl, device="cpu", preload_all=True)
    rng = np.random.default_rng(3)
    T_of = lambda u: int(wl.T(0, u // wl.Hkv))  # noqa: E731
    sel, a, _ = _subsets(wl, rng, T_of, layer.max_sel)
    a[0] = []                                   # a unit with nothing to attend
    idx, cnt = _rows(a, wl.U, layer.max_sel)
    out = np.zeros((wl.B, wl.Hq, wl.d), np.float32)
    lse = np.zeros((wl.B, wl.Hq), np.float32)
    seq = layer.seq_lens[0].contiguous()
    host = B.HostKV(k_pool=layer.k_pool.data_ptr(), v_pool=layer.v_pool.data_ptr(), page_table=0,
                    n_pages=int(wl.n_pages))
    tables = B.HostTables(page_table=layer.page_table.data_ptr(), seq_lens=seq.data_ptr(),
                          block_tokens=layer.cfg_arrays["block_tokens"].data_ptr())
    B.cpu_sparse_attn(layer.dims, layer.q[0].contiguous(), host, tables, idx, cnt, out, lse, 4)
    _compare(wl, 0, out, lse, a, T_of)


def test_cpu_attention_ed_dma_matches_oracle():
    """The host attention with ED-DMA block logits (the eviction logits added to the
    logits of each block's tokens; one block per unit at -inf, one unit with every
    listed block at -inf) against the oracle's ed_dma_attention."""
    build()
    wl = make_workload(5, seed=33, B=2, T=3000, steps=1)
    layer = PagedLayer(wl, device="cpu", preload_all=True, ed_dma=True)
    rng = np.random.default_rng(5)
    T_of = lambda u: int(wl.T(0, u // wl.Hkv))  # noqa: E731
    sel, _, _ = _subsets(wl, rng, T_of, layer.max_sel)
    bias = layer.evict.numpy().copy()
    e = {u: np.asarray(wl.evict[u], np.float64).copy() for u in range(wl.U)}
    for u in range(wl.U):
        c = sel[u][len(sel[u]) // 2]
        bias[u, c] = -np.inf
        e[u][c] = -np.inf
    bias[1, :] = -np.inf
    e[1][:] = -np.inf
    idx, cnt = _rows(sel, wl.U, layer.max_sel)
    out = np.zeros((wl.B, wl.Hq, wl.d), np.float32)
    lse = np.zeros((wl.B, wl.Hq), np.float32)
    seq = layer.seq_lens[0].contiguous()
    host = B.HostKV(k_pool=layer.k_pool.data_ptr(), v_pool=layer.v_pool.data_ptr(), page_table=0,
                    n_pages=int(wl.n_pages))
    tables = B.HostTables(page_table=layer.page_table.data_ptr(), seq_lens=seq.data_ptr(),
                          block_tokens=layer.cfg_arrays["block_tokens"].data_ptr(),
                          evict_bias=bias.ctypes.data, max_blocks_per_unit=layer.max_blocks)
    B.cpu_sparse_attn(layer.dims, layer.q[0].contiguous(), host, tables, idx, cnt, out, lse, 4)
    for u in range(wl.U):
        b, hk = u // wl.Hkv, u % wl.Hkv
        rows = slice(hk * wl.G, (hk + 1) * wl.G)
        o_ref, l_ref = O.ed_dma_attention(wl.q64(0, u), wl.K64(u), wl.V64(u), sel[u], int(wl.g[u]), T_of(u), e[u])
        o, lv = np.asarray(out[b, rows], np.float64), np.asarray(lse[b, rows], np.float64)
        if np.all(np.isneginf(l_ref)):
            assert np.all(o == 0) and np.all(np.isneginf(lv)), u
            continue
        diff = np.abs(o - o_ref)
        assert diff.max() <= ATT_ABS, (u, diff.max())
        assert (diff / np.maximum(np.abs(o_ref), REL_FLOOR)).max() <= ATT_REL, u
        assert np.abs(lv - l_ref).max() <= LSE_ABS, u


@pytest.mark.gpu
@pytest.mark.parametrize("cfg_id,kw", [(2, dict(T=5000)), (5, dict(B=2, T=3000, steps=1)),
                                       (3, dict(B=1, T=9000, steps=1))])
def test_split_attention_merged_on_gpu(cfg_id, kw):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build()
    wl = make_workload(cfg_id, seed=32, **kw)
    layer = PagedLayer(wl, preload_all=True)
    layer.prefill()
    rng = np.random.default_rng(4)
    T_of = lambda u: int(wl.T(0, u // wl.Hkv))  # noqa: E731
    sel, a, b = _subsets(wl, rng, T_of, layer.max_sel)
    a[wl.U - 1], b[wl.U - 1] = sel[wl.U - 1], []   # one unit entirely on the GPU
    a[0], b[0] = [], sel[0]                     # one unit entirely on the CPU
    MS = layer.max_sel
    dev = layer.device
    # GPU part
    ia, ca = _rows(a, wl.U, MS)
    ia_d, ca_d = torch.as_tensor(ia, device=dev), torch.as_tensor(ca, device=dev)
    out_a, lse_a = torch.zeros_like(layer.out), torch.zeros_like(layer.lse)
    B.sparse_decode_attn(layer.dims, layer.q[0], layer.kv_at(layer.seq_lens[0]), layer.cfg, ia_d, ca_d, out_a, lse_a,
                         layer.workspace, layer.status)
    # CPU part over host copies
    ib, cb = _rows(b, wl.U, MS)
    hk, hv = layer.k_pool.cpu(), layer.v_pool.cpu()
    pt, seq, gs = layer.page_table.cpu(), layer.seq_lens[0].cpu(), layer.cfg_arrays["block_tokens"].cpu()
    qh = layer.q[0].cpu()
    out_b = np.zeros((wl.B, wl.Hq, wl.d), np.float32)
    lse_b = np.zeros((wl.B, wl.Hq), np.float32)
    B.cpu_sparse_attn(layer.dims, qh, B.HostKV(k_pool=hk.data_ptr(), v_pool=hv.data_ptr(), page_table=0,
                                                n_pages=int(wl.n_pages)),
                      B.HostTables(page_table=pt.data_ptr(), seq_lens=seq.data_ptr(), block_tokens=gs.data_ptr()),
                      ib, cb, out_b, lse_b, 8)
    ob_d, lb_d = torch.as_tensor(out_b, device=dev), torch.as_tensor(lse_b, device=dev)
    # merge in place into the GPU part
    B.lse_merge(layer.dims, out_a, lse_a, ob_d, lb_d, out_a, lse_a)
    # the whole selection on the GPU, for comparison
    i_all, c_all = _rows(sel, wl.U, MS)
    out_w, lse_w = torch.zeros_like(layer.out), torch.zeros_like(layer.lse)
    B.sparse_decode_attn(layer.dims, layer.q[0], layer.kv_at(layer.seq_lens[0]), layer.cfg,
                         torch.as_tensor(i_all, device=dev), torch.as_tensor(c_all, device=dev), out_w, lse_w,
                         layer.workspace, layer.status)
    torch.cuda.synchronize()
    assert layer.read_status() == 0
    assert (out_a - out_w).abs().max().item() <= 1e-4
    assert (lse_a - lse_w).abs().max().item() <= 1e-4
    _compare(wl, 0, out_a.cpu().numpy(), lse_a.cpu().numpy(), sel, T_of)
