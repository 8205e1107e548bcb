"""GPU parity of the five calls against the float64 oracle (through the C ABI)."""
import functools

import numpy as np
import pytest
import torch

from _parity import ATT_ABS, ATT_REL, LSE_ABS, attention_errors, run_parity
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


# Shrunken versions of the five configurations: several tiles, ragged tails, and the
# multi-step ones cross a block boundary during the run.
SMALL = {
    "cfg1-tiny": (1, {}),
    "cfg2-T4133": (2, dict(T=4096 + 37)),
    "cfg3-B2-T9210x12": (3, dict(B=2, T=9210, steps=12)),
    "cfg4-B3-T3000..6000": (4, dict(B=3, T_range=(3000, 6000))),
    "cfg5-B4-T2040x16": (5, dict(B=4, T=2040, steps=16)),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_parity_small(name):
    cfg, kw = SMALL[name]
    rep = run_parity(make_workload(cfg, seed=1, **kw))
    rep.check()


@pytest.mark.parametrize("name", sorted(SMALL))
def test_parity_small_fused_step(name):
    cfg, kw = SMALL[name]
    rep = run_parity(make_workload(cfg, seed=1, **kw), fused=True)
    rep.check()


def test_fused_step_matches_separate_calls():
    """bs_decode_step gives the separate calls' selections, set-differences and
    summaries exactly and their attention within rounding."""
    wl = make_workload(3, seed=13, B=2, T=7000, steps=6)
    a, b = PagedLayer(wl), PagedLayer(wl)
    a.prefill()
    b.prefill()
    for step in range(wl.steps):
        a.append(step)
        b.append(step)
        a.step(step)
        b.fused_step(step)
        torch.cuda.synchronize()
        assert a.selection(1 - a.cur) == b.selection(1 - b.cur), step
        for name in ("added", "removed", "added_cnt", "removed_cnt"):
            assert torch.equal(getattr(a, name), getattr(b, name)), (step, name)
        assert torch.equal(a.summaries.nan_to_num(7.0), b.summaries.nan_to_num(7.0)), step
        assert (a.out - b.out).abs().max().item() <= 1e-5
        assert (a.lse - b.lse).abs().max().item() <= 1e-5
    if a.alive is not None:
        assert torch.equal(a.alive, b.alive)
    assert a.read_status() == 0 and b.read_status() == 0


@pytest.mark.parametrize("fused", [False, True])
def test_parity_large_selection_workspace_merge(fused):
    """Selections above 1024 pages per unit merge their splits through the workspace."""
    wl = make_workload(2, seed=14, T=20000)
    wl.k[4:] = 600                      # ~1200 pages per retrieval unit
    rep = run_parity(wl, fused=fused)
    rep.check()


@pytest.mark.parametrize("B", [10, 40])
@pytest.mark.parametrize("fused", [False, True])
def test_parity_few_splits_per_unit(B, fused):
    """Many units: the attention takes 2 (B=10, 80 units) or 1 (B=40) splits per unit."""
    wl = make_workload(5, seed=3, B=B, T=3000, steps=2)
    wl.k[:] = 20
    wl.k_e[:] = 12
    rep = run_parity(wl, fused=fused)
    rep.check()


@pytest.mark.parametrize("fused", [False, True])
def test_parity_workspace_split_bounds(fused):
    """The workspace plan (24 units, selections above 256 pages) with units whose head
    configuration bounds them to 1, 3, 8 and 14 splits: in the fused step only those
    splits take part, and a unit bounded to one split writes its output without a merge."""
    wl = make_workload(4, seed=21, B=6, T_range=(3000, 6000), steps=2)
    wl.k[:] = 80
    wl.k[0::3] = 1
    wl.sink[0::3] = 0
    wl.k[1::3] = 10
    rep = run_parity(wl, fused=fused)
    rep.check()


@pytest.mark.parametrize("T", [1, 17, 40])
@pytest.mark.parametrize("fused", [False, True])
def test_parity_tiny_lengths(T, fused):
    """One token, a partial first block, a budget larger than the candidates."""
    rep = run_parity(make_workload(2, seed=15, T=T), fused=fused)
    rep.check()


@pytest.mark.parametrize("fused", [False, True])
def test_parity_degenerate_budgets(fused):
    """Dual units with k = 0 (forced blocks only), k_e = k (no query-aware blocks) and
    k_e = 0 (no eviction-driven blocks)."""
    wl = make_workload(5, seed=16, B=2, T=3000, steps=3)
    wl.k[0::2] = 0
    wl.k_e[0::2] = 0
    wl.k_e[1::4] = wl.k[1::4]
    wl.k_e[3::4] = 0
    rep = run_parity(wl, fused=fused)
    rep.check()


@pytest.mark.parametrize("fused", [False, True])
def test_parity_shared_memory_selection_path(fused):
    """More candidates than the register path holds (9,374 blocks of 16 tokens)."""
    wl = make_workload(3, seed=17, B=1, T=150000, steps=1)
    wl.g[:] = 16
    wl.s[:] = 4
    wl.cls[:] = O.RETRIEVAL
    wl.k[:] = 300
    rep = run_parity(wl, units=[0, 5], summary_rows_sample=256, fused=fused)
    rep.check()


# GQA group sizes other than the configurations' 4 and 7 (the kernels are instantiated
# for G = 1..8): all-retrieval (config 4 shape), dual (config 5), streaming + retrieval
# (config 2) and the fp32 cache (config 1, head_dim 64).
GROUPS = {
    "cfg4-G1": (4, dict(B=2, T_range=(6000, 9000), Hq=2, Hkv=2)),
    "cfg4-G2": (4, dict(B=2, T_range=(6000, 9000), Hq=4, Hkv=2)),
    "cfg4-G3": (4, dict(B=2, T_range=(6000, 9000), Hq=6, Hkv=2)),
    "cfg4-G5": (4, dict(B=2, T_range=(6000, 9000), Hq=10, Hkv=2)),
    "cfg4-G6": (4, dict(B=2, T_range=(6000, 9000), Hq=12, Hkv=2)),
    "cfg4-G8": (4, dict(B=2, T_range=(6000, 9000), Hq=16, Hkv=2)),
    "cfg5-G3": (5, dict(B=1, T=2040, steps=6, Hq=6, Hkv=2)),
    "cfg5-G8": (5, dict(B=1, T=2040, steps=6, Hq=16, Hkv=2)),
    "cfg2-G5": (2, dict(T=4133, Hq=40, Hkv=8)),
    "cfg1-G3": (1, dict(Hq=3, Hkv=1)),
    "cfg1-G8": (1, dict(Hq=8, Hkv=1)),
}


@pytest.mark.parametrize("name", sorted(GROUPS))
@pytest.mark.parametrize("fused", [False, True])
def test_parity_group_sizes(name, fused):
    cfg, kw = GROUPS[name]
    rep = run_parity(make_workload(cfg, seed=3, **kw), fused=fused)
    rep.check()


# bf16 caches with head_dim 64 (the configurations use 128 for bf16, 64 only for fp32).
HEAD_DIM_64 = {
    "cfg2-d64": (2, dict(T=4133, d=64)),
    "cfg4-d64-G7": (4, dict(B=2, T_range=(6000, 9000), d=64)),
    "cfg5-d64-G8": (5, dict(B=1, T=2040, steps=6, Hq=16, Hkv=2, d=64)),
}


@pytest.mark.parametrize("name", sorted(HEAD_DIM_64))
@pytest.mark.parametrize("fused", [False, True])
def test_parity_bf16_head_dim_64(name, fused):
    cfg, kw = HEAD_DIM_64[name]
    rep = run_parity(make_workload(cfg, seed=4, **kw), fused=fused)
    rep.check()


@pytest.mark.parametrize("kw", [dict(d=128), dict(d=128, Hq=8, Hkv=1)], ids=["G4", "G8"])
@pytest.mark.parametrize("fused", [False, True])
def test_parity_fp32_head_dim_128(kw, fused):
    """fp32 caches at head_dim 128 (configuration 1 uses 64)."""
    rep = run_parity(make_workload(1, seed=6, **kw), fused=fused)
    rep.check()


@pytest.mark.parametrize("name", ["cfg2-T4133", "cfg5-B4-T2040x16"])
@pytest.mark.parametrize("fused", [False, True])
def test_parity_fp32_queries_over_bf16_cache(name, fused):
    """q_dtype fp32 with a bf16 cache: the same query values, widened."""
    cfg, kw = SMALL[name]
    rep = run_parity(make_workload(cfg, seed=7, **kw), fused=fused, q_fp32=True)
    rep.check()


@pytest.mark.parametrize("fused", [False, True])
def test_parity_group_mean(fused):
    rep = run_parity(make_workload(2, seed=2, T=3000), group_reduce="mean", fused=fused)
    rep.check()


# Full sizes of the configurations, with outputs sampled on a subset of units.
def _sample_units(wl, n):
    rng = np.random.default_rng(7)
    by_cls = {c: [u for u in range(wl.U) if wl.cls[u] == c] for c in (O.STREAMING, O.RETRIEVAL, O.DUAL)}
    pick = []
    for c, us in by_cls.items():
        if us:
            pick += rng.choice(us, size=min(len(us), max(1, n // 2)), replace=False).tolist()
    return sorted(set(pick))[:max(n, 2)]


@functools.lru_cache(maxsize=1)
def _full_workload(cfg):
    return make_workload(cfg, seed=0)


@pytest.mark.parametrize("cfg,fused", [(1, False), (2, False), (2, True), (3, False), (3, True), (4, False),
                                       (4, True), (5, False), (5, True)])
def test_parity_full_size(cfg, fused):
    """Full-size configurations through the five calls and through the fused step:
    summaries (256 sampled rows per unit from config 3 on), scores, selections, alive
    masks and set-differences of every unit at every step; the attention output of every
    unit for configs 1 and 2 and of six sampled units (both classes) for configs 3-5."""
    wl = _full_workload(cfg)
    attend = None if cfg <= 2 else set(_sample_units(wl, 6))
    rep = run_parity(wl, None, summary_rows_sample=None if cfg <= 2 else 256, fused=fused, attend_units=attend)
    assert rep.selection_checks == wl.U * wl.steps
    rep.check()


# ---------------------------------------------------------------------------
# ED-DMA attention: each block's eviction logit added to its tokens' logits
# ("Technisches Resümee: NOSA", Methodik / 1. Algorithmus: NOSA, ED-DMA)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name,cfg,kw", [("cluster-16-units", 5, dict(B=2, T=2040, steps=6)),
                                         ("cluster-32-units", 5, dict(B=4, T=2040, steps=16)),
                                         ("workspace-32-units", 5, dict(B=4, T=8190, steps=4))])
@pytest.mark.parametrize("fused", [False, True])
def test_parity_ed_dma(name, cfg, kw, fused):
    wl = make_workload(cfg, seed=41, **kw)
    if name.startswith("workspace"):
        wl.k[:] = 80                    # selections above 256 pages over 32 units: the workspace plan
        wl.k_e[:] = 60
    rep = run_parity(wl, fused=fused, ed_dma=True)
    rep.check()


@pytest.mark.parametrize("fused", [False, True])
def test_parity_ed_dma_full_size(fused):
    """Config 5 at full size (512 dual units, 16 steps) with ED-DMA attention: every
    unit's selection at every step, the attention of six sampled units."""
    wl = _full_workload(5)
    rep = run_parity(wl, None, summary_rows_sample=256, fused=fused, attend_units=set(_sample_units(wl, 6)),
                     ed_dma=True)
    assert rep.selection_checks == wl.U * wl.steps
    rep.check()


def _random_block_logits(layer, rng, sel):
    """Random logits N(0, 2^2) per block, with one selected block per unit and (with
    more than one unit) every block of unit 1 at -inf."""
    U, MB = layer.wl.U, layer.max_blocks
    e = (rng.standard_normal((U, MB)) * 2).astype(np.float32)
    for u in range(U):
        if sel[u]:
            e[u, sel[u][len(sel[u]) // 2]] = -np.inf
    if U > 1:
        e[1, :] = -np.inf
    return e


@pytest.mark.parametrize("name,cfg,kw", [("fp32-cluster", 1, {}), ("fp32-workspace", 1, dict(B=24, T=9000)),
                                         ("bf16-cluster", 2, dict(T=4133)),
                                         ("bf16-workspace", 4, dict(B=6, T_range=(3000, 6000))),
                                         ("bf16-workspace-1200-pages", 2, dict(T=20000))])
@pytest.mark.parametrize("noalloc", [False, True])
def test_ed_dma_block_logits_every_plan(name, cfg, kw, noalloc):
    """bs_sparse_decode_attn with random block logits (some -inf, one unit all -inf)
    over the oracle's selection, in each attention plan, against ed_dma_attention."""
    wl = make_workload(cfg, seed=42, **kw)
    if name == "fp32-workspace":
        wl.k[:] = 70                     # ~290 pages per unit over 24 units: the workspace plan
    if name == "bf16-workspace":
        wl.k[:] = 80                     # ~330 pages per unit over 24 units: the workspace plan
    if name == "bf16-workspace-1200-pages":
        wl.k[4:] = 600                   # above 1024 pages per unit
    layer = PagedLayer(wl)
    layer.prefill()
    layer.append(0)
    state = O.init_state(wl)
    res = O.decode_step(wl, 0, state, attend_units=set())
    sel = {u: res[u].sel.sel for u in range(wl.U)}
    layer.set_selection(sel)
    e = _random_block_logits(layer, np.random.default_rng(6), sel)
    e_d = torch.as_tensor(e, device=layer.device)
    kv = layer.kv_at(layer.seq_lens[0])
    if noalloc:
        B.sparse_decode_attn_noalloc(layer.dims, layer.q[0], kv, layer.cfg, layer.sel[layer.cur],
                                     layer.cnt[layer.cur], layer.out, layer.lse, layer.status, evict_bias=e_d)
    else:
        B.sparse_decode_attn(layer.dims, layer.q[0], kv, layer.cfg, layer.sel[layer.cur], layer.cnt[layer.cur],
                             layer.out, layer.lse, layer.workspace, layer.status, evict_bias=e_d)
    torch.cuda.synchronize()
    assert layer.read_status() == 0
    out, lse = layer.out.cpu().numpy(), layer.lse.cpu().numpy()
    for u in range(wl.U):
        b, hk = divmod(u, wl.Hkv)
        rows = slice(hk * wl.G, (hk + 1) * wl.G)
        T = int(wl.T(0, b))
        o_ref, l_ref = O.ed_dma_attention(wl.q64(0, u), wl.K64(u), wl.V64(u), sel[u], int(wl.g[u]), T,
                                          e[u].astype(np.float64))
        if np.all(np.isneginf(l_ref)):
            assert np.all(out[b, rows] == 0) and np.all(np.isneginf(lse[b, rows])), u
            continue
        a_abs, a_rel = attention_errors(out[b, rows], o_ref)
        assert a_abs <= ATT_ABS and a_rel <= ATT_REL, (u, a_abs, a_rel)
        assert np.abs(lse[b, rows] - l_ref).max() <= LSE_ABS, u


def test_ed_dma_zero_logits_equal_plain_bitwise():
    """All-zero block logits give bitwise the plain attention (adding 0 changes no
    logit), in the fused step and in the stand-alone call."""
    wl = make_workload(5, seed=43, B=4, T=2040, steps=3)
    a, b = PagedLayer(wl), PagedLayer(wl, ed_dma=True)
    b.evict.zero_()                     # also the selection's logits: both sides select alike
    a.evict.zero_()
    a.prefill()
    b.prefill()
    for step in range(wl.steps):
        a.append(step)
        b.append(step)
        a.fused_step(step)
        b.fused_step(step)
        torch.cuda.synchronize()
        assert a.selection(1 - a.cur) == b.selection(1 - b.cur), step
        assert torch.equal(a.out, b.out) and torch.equal(a.lse, b.lse), step
    a.attend(wl.steps - 1)
    b.attend(wl.steps - 1)
    torch.cuda.synchronize()
    assert torch.equal(a.out, b.out) and torch.equal(a.lse, b.lse)
    assert a.read_status() == 0 and b.read_status() == 0


def test_batch_invariance():
    """A sub-batch gives bitwise the same outputs as the full batch."""
    outs = []
    for Bn in (3, 2):
        layer = PagedLayer(make_workload(4, seed=5, B=Bn, T_range=(3000, 6000)))
        layer.prefill()
        layer.append(0)
        layer.step(0)
        torch.cuda.synchronize()
        outs.append((layer.out.cpu(), layer.lse.cpu(), layer.selection(1 - layer.cur)))
        assert layer.read_status() == 0
    (o3, l3, s3), (o2, l2, s2) = outs
    assert torch.equal(o3[:2], o2) and torch.equal(l3[:2], l2)
    assert s3[:2 * 4] == s2


def test_incremental_summaries_equal_rebuild_bitwise():
    wl = make_workload(3, seed=3, B=1, T=5000, steps=40)
    layer = PagedLayer(wl)
    layer.prefill()
    for step in range(wl.steps):
        layer.append(step)
        layer.update_summaries(step)
    inc = layer.summaries.clone()
    layer.summaries.fill_(float("nan"))
    last = layer.seq_lens[wl.steps - 1].clone()
    B.build_block_summaries(layer.dims, layer.kv_at(last), layer.cfg, layer.zeros_b, int(last.max()),
                            layer.summaries, layer.status)
    torch.cuda.synchronize()
    for u in range(wl.U):
        rows = -(-int(last[0]) // int(wl.s[u]))
        off = int(layer._cfg_host["sum_off"][u])
        a = inc[off:off + rows * wl.d]
        bb = layer.summaries[off:off + rows * wl.d]
        assert torch.equal(a, bb), u
    assert layer.read_status() == 0


def test_select_exact_on_crafted_ties():
    """Scores with many exact ties: the GPU top-k equals the oracle's (lowest index wins)."""
    wl = make_workload(2, seed=4, T=6000)
    layer = PagedLayer(wl)
    rng = np.random.default_rng(0)
    T = int(wl.T(0, 0))
    for trial in range(6):
        vals = rng.integers(-3, 4, size=layer.scores.shape).astype(np.float32)
        if trial == 0:
            vals[:] = 1.0
        if trial == 1:
            vals[:] = -0.0
        layer.scores.copy_(torch.from_numpy(vals))
        layer.select(0)
        torch.cuda.synchronize()
        got = layer.selection(layer.cur)
        for u in range(wl.U):
            ref = O.select_unit(int(wl.cls[u]), T, int(wl.g[u]), int(wl.sink[u]), int(wl.local[u]),
                                int(wl.k[u]), 0, vals[u].astype(np.float64))
            assert got[u] == ref.sel, (trial, u)
    assert layer.read_status() == 0


def test_dual_select_exact_on_crafted_ties():
    """Dual selection over steps with tied logits and scores: exact Gamma_e/Gamma_q and alive."""
    wl = make_workload(5, seed=6, B=2, T=1000, steps=40)
    wl.evict = np.round(wl.evict * 2).astype(np.float32) / 2          # ties in eviction logits
    layer = PagedLayer(wl)
    rng = np.random.default_rng(1)
    alive_ref = {u: np.ones(layer.max_blocks, np.uint8) for u in range(wl.U)}
    for step in range(wl.steps):
        vals = rng.integers(-2, 3, size=layer.scores.shape).astype(np.float32)
        layer.scores.copy_(torch.from_numpy(vals))
        layer.select(step)
        torch.cuda.synchronize()
        got = layer.selection(layer.cur)
        alive = layer.alive.cpu().numpy()
        for u in range(wl.U):
            T = wl.T(step, u // wl.Hkv)
            ref = O.select_unit(O.DUAL, T, int(wl.g[u]), int(wl.sink[u]), int(wl.local[u]), int(wl.k[u]),
                                int(wl.k_e[u]), vals[u].astype(np.float64), wl_evict_row(wl, u, layer.max_blocks),
                                alive_ref[u])
            alive_ref[u] = ref.alive
            assert got[u] == ref.sel, (step, u)
            assert np.array_equal(alive[u], ref.alive), (step, u)
        layer.advance()
    assert layer.read_status() == 0


def wl_evict_row(wl, u, n):
    row = np.full(n, -np.inf)
    row[:min(n, wl.evict.shape[1])] = wl.evict[u, :n]
    return row


def test_setdiff_random_lists():
    wl = make_workload(2, seed=8, T=3000)
    layer = PagedLayer(wl)
    rng = np.random.default_rng(2)
    MS = layer.max_sel
    prev, cur = {}, {}
    for u in range(wl.U):
        prev[u] = sorted(rng.choice(200, size=int(rng.integers(0, MS + 1)), replace=False).tolist())
        cur[u] = sorted(rng.choice(200, size=int(rng.integers(0, MS + 1)), replace=False).tolist())
    layer.set_selection(prev, which=1 - layer.cur)
    layer.set_selection(cur, which=layer.cur)
    layer.setdiff()
    torch.cuda.synchronize()
    a, ac = layer.added.cpu().numpy(), layer.added_cnt.cpu().numpy()
    r, rc = layer.removed.cpu().numpy(), layer.removed_cnt.cpu().numpy()
    for u in range(wl.U):
        ra, rr = O.setdiff(prev[u], cur[u])
        assert a[u, :ac[u]].tolist() == ra and r[u, :rc[u]].tolist() == rr
    assert layer.read_status() == 0


def test_out_of_range_page_reports_and_skips():
    """A page-table entry outside the pool sets BS_ERR_DEVICE_BOUNDS; nothing faults."""
    wl = make_workload(2, seed=9, T=3000)
    layer = PagedLayer(wl, preload_all=True)
    layer.prefill()
    torch.cuda.synchronize()
    assert layer.read_status() == 0
    layer.page_table[4, 0] = wl.n_pages + 5        # sink page of a retrieval unit
    layer.page_table[0, 3] = -7                    # a sink page of a streaming unit
    layer.step(0)
    torch.cuda.synchronize()
    assert layer.read_status() == B.BS_ERR_DEVICE_BOUNDS
    # the context is still usable
    layer.page_table.copy_(torch.from_numpy(wl.page_table))
    layer.status.zero_()
    layer.step(0)
    torch.cuda.synchronize()
    assert layer.read_status() == 0
