"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each ``check_*`` function takes the oracle module so that ``test_oracle_mutations``
can plant a mistake in the oracle and show that some pin fails. None of these
checks re-types the oracle's own formula: each goes through a hand-derived fixture
(tests/golden/), a library routine (torch's scaled_dot_product_attention,
numpy's setdiff1d), a closed form, an invariant the pages state, or brute force.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import _golden
from oracle import bsattn_oracle as O
from workloads import make_workload


# ---------------------------------------------------------------------------
# Hand-derived fixtures
# ---------------------------------------------------------------------------
def check_golden_pooling(orc):
    f = _golden.load("pooling_partial.txt")
    T, s, g, d = _golden.i(f["T"]), _golden.i(f["s"]), _golden.i(f["g"]), _golden.i(f["d"])
    kbar = orc.sub_block_means(f["K"], T, s)
    np.testing.assert_allclose(kbar, f["kbar"], rtol=0, atol=1e-12)
    for reduce, key in (("max", "S_times_sqrt_d_max"), ("mean", "S_times_sqrt_d_mean")):
        S = orc.block_scores(f["q"], kbar, T, g, s, reduce)
        np.testing.assert_allclose(S * math.sqrt(d), f[key], rtol=0, atol=1e-12)


def check_golden_select_retrieval(orc):
    f = _golden.load("select_retrieval.txt")
    for case in ("A", "B"):
        T, g, sink, local, k = (_golden.i(f[f"{case}.{x}"]) for x in ("T", "g", "sink", "local", "k"))
        scores = f[f"{case}.scores"]
        assert orc.forced_blocks(T, g, sink, local) == _golden.ints(f[f"{case}.forced"])
        assert orc.candidate_blocks(T, g, sink, local) == _golden.ints(f[f"{case}.candidates"])
        r = orc.select_unit(orc.RETRIEVAL, T, g, sink, local, k, 0, scores)
        assert r.sel == _golden.ints(f[f"{case}.sel"])
        assert r.gamma_q == _golden.ints(f[f"{case}.topk"])
        assert r.boundary == tuple(float(x) for x in f[f"{case}.boundary"])
    assert orc.select_unit(orc.RETRIEVAL, 40, 4, 4, 6, 3, 0, f["A.scores"]).near_tie
    assert not orc.select_unit(orc.RETRIEVAL, 37, 4, 4, 6, 1, 0, f["B.scores"]).near_tie
    for case in ("C", "D"):
        T, g, sink, local = (_golden.i(f[f"{case}.{x}"]) for x in ("T", "g", "sink", "local"))
        r = orc.select_unit(orc.STREAMING, T, g, sink, local, 0, 0)
        assert r.sel == _golden.ints(f[f"{case}.sel"])
    assert orc.candidate_blocks(10, 4, 8, 8) == []


def check_golden_select_dual(orc):
    f = _golden.load("select_dual.txt")
    g, sink, local, k, k_e = (_golden.i(f[x]) for x in ("g", "sink", "local", "k", "k_e"))
    alive = np.ones(8, np.uint8)
    prev = []
    for st in ("s1", "s2", "s3"):
        T = _golden.i(f[f"{st}.T"])
        r = orc.select_unit(orc.DUAL, T, g, sink, local, k, k_e, f["scores"], f["evict"], alive)
        assert r.gamma_e == _golden.ints(f[f"{st}.gamma_e"]), st
        assert r.gamma_q == _golden.ints(f[f"{st}.gamma_q"]), st
        assert r.sel == _golden.ints(f[f"{st}.sel"]), st
        assert _golden.ints(r.alive) == _golden.ints(f[f"{st}.alive"]), st
        added, removed = orc.setdiff(prev, r.sel)
        assert added == _golden.ints(f[f"{st}.added"]) if f[f"{st}.added"].size else added == []
        assert removed == _golden.ints(f[f"{st}.removed"]) if f[f"{st}.removed"].size else removed == []
        alive, prev = r.alive, r.sel


def check_golden_attention(orc):
    f = _golden.load("attention_closed_form.txt")
    T, g, cap = _golden.i(f["A.T"]), _golden.i(f["A.g"]), _golden.i(f["A.capacity"])
    K = np.stack([np.zeros(cap), np.arange(cap)], axis=1).astype(np.float64)
    V = np.stack([np.arange(cap), np.ones(cap)], axis=1).astype(np.float64)
    o, lse = orc.sparse_attention(f["A.q"][None, :], K, V, _golden.ints(f["A.sel"]), g, T)
    np.testing.assert_allclose(o[0], f["A.o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], _golden.num(f["A.lse"]), rtol=0, atol=1e-12)
    o, lse = orc.sparse_attention(np.atleast_1d(f["B.q"])[None, :], f["B.K"].reshape(-1, 1), f["B.V"].reshape(-1, 1), _golden.ints(f["B.sel"]),
                                  _golden.i(f["B.g"]), _golden.i(f["B.T"]))
    np.testing.assert_allclose(o[0], f["B.o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], _golden.num(f["B.lse"]), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# P1: a budget that covers every block gives dense attention (library routine)
# ---------------------------------------------------------------------------
def _sdpa(q, K, V, mask=None):
    qt = torch.from_numpy(np.ascontiguousarray(q))[None]            # [1][G][d]
    kt = torch.from_numpy(np.ascontiguousarray(K))[None]            # [1][T][d]
    vt = torch.from_numpy(np.ascontiguousarray(V))[None]
    m = None if mask is None else torch.from_numpy(mask)[None, None, :].expand(1, q.shape[0], K.shape[0])
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m)[0].numpy()


def check_p1_full_budget_is_dense(orc):
    rng = np.random.default_rng(11)
    for T, g, s, G, d in ((301, 16, 4, 4, 32), (256, 32, 8, 2, 16), (97, 16, 16, 3, 8)):
        K = rng.standard_normal((T, d))
        V = rng.standard_normal((T, d))
        q = rng.standard_normal((G, d))
        kbar = orc.sub_block_means(K, T, s)
        S = orc.block_scores(q, kbar, T, g, s)
        n_blk = -(-T // g)
        r = orc.select_unit(orc.RETRIEVAL, T, g, g, g, n_blk, 0, S)
        assert r.sel == list(range(n_blk))
        o, lse = orc.sparse_attention(q, K, V, r.sel, g, T)
        np.testing.assert_allclose(o, _sdpa(q, K, V), rtol=0, atol=1e-12)
        # lse closes the softmax: sum_t exp(q.k_t/sqrt(d) - lse) = 1 for every head.
        logits = (q @ K.T) / math.sqrt(d)
        np.testing.assert_allclose(np.exp(logits - lse[:, None]).sum(axis=1), 1.0, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# P2: a streaming head is sink + sliding-window attention (library routine, mask)
# ---------------------------------------------------------------------------
def check_p2_streaming_is_sink_window(orc):
    rng = np.random.default_rng(12)
    G, d, g, sink, local = 4, 16, 32, 128, 2048
    for T in (4096, 4096 + 32 * 7, 4100, 2300):
        K = rng.standard_normal((T, d))
        V = rng.standard_normal((T, d))
        q = rng.standard_normal((G, d))
        r = orc.select_unit(orc.STREAMING, T, g, sink, local, 0, 0)
        start = (max(0, T - local) // g) * g      # the window extended back to its block boundary
        if T % g == 0 and (T - local) % g == 0:
            assert start == T - local              # aligned: exactly the StreamingLLM window
        mask = np.zeros(T, dtype=bool)
        mask[:sink] = True
        mask[start:] = True
        o, _ = orc.sparse_attention(q, K, V, r.sel, g, T)
        np.testing.assert_allclose(o, _sdpa(q, K, V, mask), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# P3: selection equals brute force over all k-subsets (tiny inputs)
# ---------------------------------------------------------------------------
def _brute_topk(keys, pool, k):
    """The unique k-subset A of the pool whose every member beats every non-member,
    'beats' meaning a larger key, or an equal key and a lower index."""
    k = min(k, len(pool))
    winners = []
    for A in itertools.combinations(pool, k):
        rest = [c for c in pool if c not in A]
        if all(keys[a] > keys[b] or (keys[a] == keys[b] and a < b) for a in A for b in rest):
            winners.append(sorted(A))
    assert len(winners) == 1
    return winners[0]


def check_p3_select_brute_force(orc):
    rng = np.random.default_rng(13)
    for trial in range(300):
        g = int(rng.choice([1, 2, 4]))
        T = int(rng.integers(1, 12 * g + 1))
        sink = int(rng.integers(0, 2 * g + 1))
        local = int(rng.integers(1, 3 * g + 1))
        n_blk = -(-T // g)
        keys = rng.integers(-3, 4, size=n_blk).astype(np.float64)      # many ties
        if trial % 7 == 0:
            keys[:] = 1.5                                              # all equal
        C = orc.candidate_blocks(T, g, sink, local)
        forced = orc.forced_blocks(T, g, sink, local)
        # forced set by brute force over tokens: blocks holding a sink or local token
        brute_forced = sorted({t // g for t in range(T) if t < sink or t >= T - local})
        assert forced == brute_forced
        assert C == [c for c in range(n_blk) if c not in brute_forced and (c + 1) * g <= T]
        for k in (0, 1, 2, len(C), len(C) + 3):
            r = orc.select_unit(orc.RETRIEVAL, T, g, sink, local, k, 0, keys)
            want = sorted(set(brute_forced) | set(_brute_topk(keys, C, k)))
            assert r.sel == want
        if len(C) > 2:
            assert orc.select_unit(orc.RETRIEVAL, T, g, sink, local, 2, 0,
                                   np.zeros(n_blk)).gamma_q == C[:2]


# ---------------------------------------------------------------------------
# P4 + P5: eviction monotonicity and the locality bound over multi-step runs
# ---------------------------------------------------------------------------
def check_p4_p5_eviction(orc):
    rng = np.random.default_rng(14)
    for trial in range(40):
        g = int(rng.choice([2, 4, 8]))
        k = int(rng.integers(1, 9))
        k_e = int(rng.integers(0, k + 1))
        local = int(rng.integers(1, 2 * g + 1))
        sink = int(rng.integers(0, g + 1))
        T0 = int(rng.integers(g * (k + 4), g * (k + 12)))
        steps = 3 * g + 2
        n_cap = -(-(T0 + steps) // g)
        evict = rng.standard_normal(n_cap)
        alive = np.ones(n_cap, np.uint8)
        ever_dropped = set()
        prev_e, prev_sel, prev_C = None, None, None
        for t in range(steps):
            T = T0 + t
            scores = rng.standard_normal(n_cap)          # query-aware scores change every step
            C = set(orc.candidate_blocks(T, g, sink, local))
            r = orc.select_unit(orc.DUAL, T, g, sink, local, k, k_e, scores, evict, alive)
            E = set(r.gamma_e)
            assert len(r.gamma_e) <= k_e and len(r.gamma_q) <= k - k_e
            assert E.isdisjoint(r.gamma_q)
            # P4: a block that left Gamma_e's pool never comes back to Gamma_e.
            assert not (E & ever_dropped)
            ever_dropped |= (C - E)
            if prev_e is not None:
                C_new = C - prev_C
                assert E <= (prev_e | C_new)
                # P5: new candidates were forced at the previous step, so Gamma_e(t) lies in
                # S(t-1) and the kept fraction of the budget is at least k_e / k.
                assert C_new <= set(prev_sel)
                if len(E) == k_e:
                    kept = len((E | set(r.gamma_q)) & set(prev_sel))
                    assert kept >= k_e
                    assert kept / k >= k_e / k
            alive, prev_e, prev_sel, prev_C = r.alive, E, r.sel, C


# ---------------------------------------------------------------------------
# P6: pooling special cases
# ---------------------------------------------------------------------------
def check_p6_pooling_special_cases(orc):
    rng = np.random.default_rng(15)
    G, d, g = 3, 16, 8
    for T in (64, 61):
        K = rng.standard_normal((T, d))
        q = rng.standard_normal((G, d))
        n_blk = -(-T // g)
        # s = g: block score is q . (mean key of the block) / sqrt(d), max over heads.
        S = orc.block_scores(q, orc.sub_block_means(K, T, g), T, g, g)
        for c in range(n_blk):
            blk = K[c * g:min((c + 1) * g, T)]
            m = np.add.reduce(blk, axis=0) / blk.shape[0]
            assert abs(S[c] - max(float(q[h] @ m) for h in range(G)) / math.sqrt(d)) < 1e-12
        # s = 1: block score is the block's exact maximum logit over heads and tokens.
        S1 = orc.block_scores(q, orc.sub_block_means(K, T, 1), T, g, 1)
        logits = torch.from_numpy(q) @ torch.from_numpy(K).T / math.sqrt(d)
        for c in range(n_blk):
            assert abs(S1[c] - float(logits[:, c * g:min((c + 1) * g, T)].max())) < 1e-12
        # G = 1: the group reduction is the identity, max and mean agree.
        kbar = orc.sub_block_means(K, T, 4)
        np.testing.assert_array_equal(orc.block_scores(q[:1], kbar, T, g, 4, "max"),
                                      orc.block_scores(q[:1], kbar, T, g, 4, "mean"))
        # identical heads: the group max equals a single head's score
        np.testing.assert_allclose(orc.block_scores(np.repeat(q[:1], 3, 0), kbar, T, g, 4),
                                   orc.block_scores(q[:1], kbar, T, g, 4), rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# P7: set identities of the set-difference (library routine)
# ---------------------------------------------------------------------------
def check_p7_setdiff(orc):
    rng = np.random.default_rng(16)
    for _ in range(200):
        prev = sorted(set(rng.integers(0, 40, size=int(rng.integers(0, 20))).tolist()))
        cur = sorted(set(rng.integers(0, 40, size=int(rng.integers(0, 20))).tolist()))
        added, removed = orc.setdiff(prev, cur)
        assert added == sorted(added) and removed == sorted(removed)
        assert added == np.setdiff1d(np.array(cur, int), np.array(prev, int)).tolist()
        assert removed == np.setdiff1d(np.array(prev, int), np.array(cur, int)).tolist()
        both = np.intersect1d(cur, prev).tolist()
        assert sorted(added + both) == cur and sorted(removed + both) == prev
        assert not set(added) & set(removed)
    assert orc.setdiff([], [3, 5]) == ([3, 5], [])


# ---------------------------------------------------------------------------
# P8: planted structure of the tiny configuration
# ---------------------------------------------------------------------------
def check_p8_planted(orc):
    wl = make_workload(1, seed=0)
    st = orc.init_state(wl)
    res = orc.decode_step(wl, 0, st)[0]
    g = int(wl.g[0])
    needle_blocks = [int(p) // g for p in wl.needles[0]]
    assert set(needle_blocks) <= set(res.sel.gamma_q)          # the needle is in the top-4
    assert 0 in res.sel.sel                                     # the sink block is kept
    assert len(res.sel.gamma_q) == int(wl.k[0]) and len(res.sel.sel) == 6
    # The sink token adds little to the output whatever weight it draws (Fluxion,
    # Kerninzichten item 1: initial tokens with low value norms).
    q, K, V = wl.q64(0, 0), wl.K64(0), wl.V64(0)
    U = orc.selected_tokens(res.sel.sel, g, res.T)
    w = np.exp((q @ K[U].T) / math.sqrt(wl.d) - res.lse[:, None])
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    mean_norm = np.linalg.norm(V[U], axis=1).mean()
    assert (w[:, 0] * np.linalg.norm(V[0]) <= 0.05 * mean_norm).all()


def check_p8_needles_recalled(orc, cfg_id, **kw):
    """At least 3/4 of the planted needles are selected by retrieval units."""
    wl = make_workload(cfg_id, seed=0, **kw)
    units = [u for u in range(wl.U) if wl.cls[u] != orc.STREAMING]
    st = orc.init_state(wl, units)
    res = orc.decode_step(wl, 0, st, units)
    hit = tot = 0
    for u in units:
        g = int(wl.g[u])
        for p in wl.needles[wl.unit_seq(u)]:
            tot += 1
            hit += int(int(p) // g in res[u].sel.sel)
    assert tot > 0 and hit >= 0.75 * tot


# ---------------------------------------------------------------------------
# P9: splitting the selected tokens and merging partials by log-sum-exp
# ---------------------------------------------------------------------------
def check_p9_lse_merge(orc):
    rng = np.random.default_rng(17)
    T, g, G, d = 300, 16, 4, 32
    K = rng.standard_normal((T, d)) * 2
    V = rng.standard_normal((T, d))
    q = rng.standard_normal((G, d))
    sel = sorted(rng.choice(-(-T // g), size=9, replace=False).tolist() + [])
    o, lse = orc.sparse_attention(q, K, V, sel, g, T)
    for n_parts in (2, 3, 9):
        parts = np.array_split(np.array(sel), n_parts)
        outs = [orc.sparse_attention(q, K, V, p.tolist(), g, T) for p in parts]
        lses = np.stack([x[1] for x in outs])                   # [parts][G]
        M = lses.max(axis=0)
        wts = np.exp(lses - M)
        merged_lse = M + np.log(wts.sum(axis=0))
        merged_o = sum(w[:, None] * x[0] for w, x in zip(wts, outs)) / wts.sum(axis=0)[:, None]
        np.testing.assert_allclose(merged_lse, lse, rtol=0, atol=1e-12)
        np.testing.assert_allclose(merged_o, o, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# P10: per-step summary updates equal a rebuild
# ---------------------------------------------------------------------------
def check_p10_incremental(orc):
    rng = np.random.default_rng(18)
    for s in (1, 3, 4, 16):
        K = rng.standard_normal((100, 8))
        T0 = int(rng.integers(1, 40))
        kbar = orc.sub_block_means(K, T0, s)
        for T in range(T0 + 1, 100):
            kbar = orc.update_sub_block(kbar, K, T, s)
            full = orc.sub_block_means(K, T, s)
            assert kbar.shape[0] >= full.shape[0]
            np.testing.assert_allclose(kbar[:full.shape[0]], full, rtol=0, atol=1e-13)
        # sub-block means of a constant sequence are that constant, partial or not
        Kc = np.full((23, 4), 2.5)
        np.testing.assert_array_equal(orc.sub_block_means(Kc, 23, s), 2.5)


def check_golden_block_swap(orc):
    gd = _golden.load("block_swap.txt")
    slots, blocks, g, u = _golden.i(gd["slots"]), _golden.i(gd["blocks"]), _golden.i(gd["g"]), _golden.i(gd["u"])
    sb, bs = np.full(slots, -1), np.full(blocks, -1)
    prev = []
    for step in (1, 2, 3):
        sel = _golden.ints(gd[f"s{step}.sel"])
        added, removed = orc.setdiff(prev, sel)
        sb, bs, copies = orc.block_swap(sb, bs, added, removed)
        assert _golden.ints(sb) == _golden.ints(gd[f"s{step}.slot_block"]), step
        exp = np.atleast_2d(gd[f"s{step}.copies"]).astype(int).tolist()
        assert [list(c) for c in copies] == exp, step
        prev = sel
    row = orc.cache_page_table(bs, u, g, _golden.i(gd["s3.T"]), 20, slots, 2)
    assert _golden.ints(row) == _golden.ints(gd["s3.page_table"])


def check_p11_block_swap_invariants(orc):
    """Over random selection sequences the cache holds exactly the selection, slots and
    blocks map one to one, each added block is copied once and a kept block never
    moves (no re-copy: the point of the locality guarantee)."""
    rng = np.random.default_rng(19)
    for trial in range(30):
        n_blocks, cap = int(rng.integers(5, 60)), int(rng.integers(1, 12))
        sb, bs = np.full(cap, -1), np.full(n_blocks, -1)
        prev = []
        for _ in range(12):
            keep = [c for c in prev if rng.random() < 0.7]
            fresh = [int(c) for c in rng.choice(n_blocks, size=int(rng.integers(0, min(cap, n_blocks) + 1)),
                                                replace=False)]
            sel = sorted(set(keep) | set(fresh))[:cap]
            added, removed = orc.setdiff(prev, sel)
            before = bs.copy()
            sb, bs, copies = orc.block_swap(sb, bs, added, removed)
            cached = sorted(int(c) for c in np.flatnonzero(bs >= 0))
            assert cached == sel
            for s, c in enumerate(sb):
                if c >= 0:
                    assert bs[c] == s
            assert sorted(c for c, _ in copies) == added
            for c in sel:
                if c in prev:
                    assert bs[c] == before[c]
            prev = sel


# ---------------------------------------------------------------------------
# P12: the state decode_step carries from one step to the next
# ---------------------------------------------------------------------------
def _plain_means(K, T, s):
    """Sub-block means by cumulative sums (a different route from a per-block mean)."""
    cs = np.concatenate([np.zeros((1, K.shape[1])), np.cumsum(np.asarray(K[:T], np.float64), axis=0)])
    lo = np.arange(0, T, s)
    hi = np.minimum(lo + s, T)
    return (cs[hi] - cs[lo]) / (hi - lo)[:, None]


def check_p12_decode_step_carry(orc):
    """Multi-step runs through init_state + decode_step on a dual workload that crosses
    a block boundary and on a mixed streaming/retrieval workload whose units have
    different block sizes. At every step the carried state must follow the rules the
    pages fix ("Technisches Resümee: NOSA", Dual-Selection-Mechanismus: a block that
    left Gamma_e's pool never returns to it; Lokalitätsgarantie: at least k_e of the
    k selected blocks were selected at the previous step): the summaries equal a rebuild
    at the current length, the set-difference is the one between this step's and the
    previous step's selections, and the carried alive mask marks exactly the blocks never
    dropped from Gamma_e's pool."""
    cases = [make_workload(5, seed=3, B=2, T=2040, steps=14),      # crosses T = 2048 (g = 64)
             make_workload(3, seed=5, B=1, T=4090, steps=12)]      # crosses T = 4096 for every g
    assert {int(c) for c in cases[1].cls} == {orc.STREAMING, orc.RETRIEVAL}
    assert len({int(x) for x in cases[1].g}) > 1
    for wl in cases:
        state = orc.init_state(wl)
        prev_sel = {u: [] for u in range(wl.U)}
        prev_e = {u: None for u in range(wl.U)}
        prev_C = {u: None for u in range(wl.U)}
        dropped = {u: set() for u in range(wl.U)}
        crossed = False
        for step in range(wl.steps):
            res = orc.decode_step(wl, step, state)
            for u in range(wl.U):
                r, st = res[u], state[u]
                b = wl.unit_seq(u)
                T = wl.T(step, b)
                assert r.T == T
                g, s, k_e = int(wl.g[u]), int(wl.s[u]), int(wl.k_e[u])
                # summaries carried = rebuilt at this length
                n_sub = -(-T // s)
                assert st.kbar.shape[0] >= n_sub
                np.testing.assert_allclose(st.kbar[:n_sub], _plain_means(wl.K64(u), T, s), rtol=0, atol=1e-9)
                # set-difference against the previous step's selection
                cur = np.array(r.sel.sel, dtype=np.int64)
                prv = np.array(prev_sel[u], dtype=np.int64)
                assert r.added == np.setdiff1d(cur, prv).tolist(), (step, u)
                assert r.removed == np.setdiff1d(prv, cur).tolist(), (step, u)
                C = {c for c in range(T // g)
                     if not (c < -(-int(wl.sink[u]) // g) or c >= max(0, T - int(wl.local[u])) // g)}
                if wl.cls[u] == orc.DUAL:
                    E = set(r.sel.gamma_e)
                    assert len(E) <= k_e and E <= C
                    assert not (E & dropped[u]), (step, u)                         # P4
                    if prev_e[u] is not None:
                        C_new = C - prev_C[u]
                        crossed |= bool(C_new)
                        assert E <= prev_e[u] | C_new, (step, u)                   # P4
                        if len(E) == k_e:
                            assert len((E | set(r.sel.gamma_q)) & set(prev_sel[u])) >= k_e, (step, u)  # P5
                    dropped[u] |= C - E
                    n_cap = st.alive.shape[0]
                    want = np.ones(n_cap, np.uint8)
                    want[sorted(dropped[u])] = 0
                    np.testing.assert_array_equal(st.alive, want, err_msg=f"alive, step {step} unit {u}")
                    prev_e[u] = E
                prev_C[u] = C
                prev_sel[u] = list(r.sel.sel)
        if (wl.cls == orc.DUAL).any():
            assert crossed, "the dual run must bring new candidates in"


# ---------------------------------------------------------------------------
# ED-DMA attention: the eviction logit of a block as an additive logit of its tokens
# ("Technisches Resümee: NOSA", Methodik / 1. Algorithmus: NOSA, ED-DMA)
# ---------------------------------------------------------------------------
def check_golden_ed_dma(orc):
    f = _golden.load("ed_dma_bias.txt")
    o, lse = orc.ed_dma_attention(f["A.q"], f["A.K"], f["A.V"], _golden.ints(f["A.sel"]), _golden.i(f["A.g"]),
                                  _golden.i(f["A.T"]), f["A.e"])
    np.testing.assert_allclose(o, f["A.o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, f["A.lse"], rtol=0, atol=1e-12)
    for c in "BC":
        q = np.atleast_1d(f[f"{c}.q"])[None, :]
        K, V = f[f"{c}.K"].reshape(-1, 1), f[f"{c}.V"].reshape(-1, 1)
        o, lse = orc.ed_dma_attention(q, K, V, _golden.ints(f[f"{c}.sel"]), _golden.i(f[f"{c}.g"]),
                                      _golden.i(f[f"{c}.T"]), np.atleast_1d(f[f"{c}.e"]))
        np.testing.assert_allclose(o[0], np.atleast_1d(f[f"{c}.o"]), rtol=0, atol=1e-12)
        np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(np.atleast_1d(f[f"{c}.lse"])))
        fin = np.isfinite(lse)
        np.testing.assert_allclose(lse[fin], np.atleast_1d(f[f"{c}.lse"])[fin], rtol=0, atol=1e-12)


def check_p13_ed_dma(orc):
    rng = np.random.default_rng(23)
    for T, g, G, d, n_sel in ((301, 16, 4, 32, 7), (256, 32, 2, 16, 5), (97, 16, 3, 8, 4)):
        n_blk = -(-T // g)
        K = rng.standard_normal((T + 5, d))
        V = rng.standard_normal((T + 5, d))
        q = rng.standard_normal((G, d))
        e = rng.standard_normal(n_blk) * 2
        sel = sorted(set(rng.choice(n_blk - 1, size=n_sel - 1, replace=False).tolist()) | {n_blk - 1})
        U = np.concatenate([np.arange(c * g, min((c + 1) * g, T)) for c in sel])
        # The library's attention with the blocks' logits as an additive float mask.
        o, lse = orc.ed_dma_attention(q, K, V, sel, g, T, e)
        ref = _sdpa(q, K[U], V[U], (e[U // g]).astype(np.float64))
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
        # lse closes the biased softmax over the selected tokens.
        logits = (q @ K[U].T) / math.sqrt(d) + e[U // g][None, :]
        np.testing.assert_allclose(np.exp(logits - lse[:, None]).sum(axis=1), 1.0, rtol=0, atol=1e-12)
        # A constant logit shifts lse and leaves o alone (plain softmax).
        o0, lse0 = orc.sparse_attention(q, K, V, sel, g, T)
        for c in (0.0, -3.5, 7.25):
            oc, lsec = orc.ed_dma_attention(q, K, V, sel, g, T, np.full(n_blk, c))
            np.testing.assert_allclose(oc, o0, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lsec, lse0 + c, rtol=0, atol=1e-12)
        # e = -inf removes a block: the same as not selecting it.
        drop = sel[len(sel) // 2]
        e2 = e.copy()
        e2[drop] = -np.inf
        o2, lse2 = orc.ed_dma_attention(q, K, V, sel, g, T, e2)
        o3, lse3 = orc.ed_dma_attention(q, K, V, [c for c in sel if c != drop], g, T, e)
        np.testing.assert_allclose(o2, o3, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse2, lse3, rtol=0, atol=1e-12)
    # decode_step(ed_dma=True): the same selections, and every unit's attention is the
    # library's with that unit's eviction logits as the mask of the selected tokens.
    wl = make_workload(5, seed=4, B=1, T=1100, steps=2)
    st_a, st_b = orc.init_state(wl), orc.init_state(wl)
    for step in range(2):
        plain = orc.decode_step(wl, step, st_a)
        ed = orc.decode_step(wl, step, st_b, ed_dma=True)
        for u in range(wl.U):
            assert ed[u].sel.sel == plain[u].sel.sel
            g, T = int(wl.g[u]), ed[u].T
            U = np.concatenate([np.arange(c * g, min((c + 1) * g, T)) for c in ed[u].sel.sel])
            mask = np.asarray(wl.evict[u], np.float64)[U // g]
            ref = _sdpa(wl.q64(step, u), wl.K64(u)[U], wl.V64(u)[U], mask)
            np.testing.assert_allclose(ed[u].o, ref, rtol=0, atol=1e-10)
            assert np.abs(ed[u].o - plain[u].o).max() > 1e-6


def check_p14_selection_size(orc):
    """S = F + top_k(C) with F and C disjoint ("Technisches Resümee: NOSA", Dual-Selection-
    Mechanismus; "Technische Samenvatting: Fluxion", Granularity-Budget Selector): a
    retrieval unit selects |F| + min(k, |C|) blocks, a dual unit |F| + |Gamma_e| +
    |Gamma_q|; neither exceeds min(n_blk, |F| + k), the bound by which the fused step's
    workspace attention sizes its splits. |F| also equals the closed form that bound uses,
    n_sink + n_blk - max(local_lo, n_sink)."""
    rng = np.random.default_rng(14)
    for _ in range(300):
        g = int(rng.choice([4, 8, 16]))
        T = int(rng.integers(1, 400))
        sink, local, k = int(rng.integers(0, 3 * g)), int(rng.integers(1, 4 * g)), int(rng.integers(0, 30))
        n_blk = -(-T // g)
        F, C = orc.forced_blocks(T, g, sink, local), orc.candidate_blocks(T, g, sink, local)
        n_sink, local_lo = min(-(-sink // g), n_blk), max(0, T - local) // g
        assert len(F) == n_sink + n_blk - max(local_lo, n_sink)
        scores = rng.standard_normal(n_blk)
        r = orc.select_unit(orc.RETRIEVAL, T, g, sink, local, k, 0, scores)
        assert len(r.sel) == len(F) + min(k, len(C))
        assert len(r.sel) <= min(n_blk, len(F) + k)
        k_e = int(rng.integers(0, k + 1))
        alive = (rng.random(n_blk) < 0.7).astype(np.uint8)
        d = orc.select_unit(orc.DUAL, T, g, sink, local, k, k_e, scores, rng.standard_normal(n_blk), alive)
        n_e = min(k_e, sum(1 for c in C if alive[c]))
        assert len(d.sel) == len(F) + n_e + min(k - k_e, len(C) - n_e)
        assert len(d.sel) <= min(n_blk, len(F) + k)


ALL_CHECKS = [check_golden_pooling, check_golden_select_retrieval, check_golden_select_dual,
              check_golden_attention, check_p1_full_budget_is_dense, check_p2_streaming_is_sink_window,
              check_p3_select_brute_force, check_p4_p5_eviction, check_p6_pooling_special_cases,
              check_p7_setdiff, check_p8_planted, check_p9_lse_merge, check_p10_incremental,
              check_golden_block_swap, check_p11_block_swap_invariants, check_p12_decode_step_carry,
              check_golden_ed_dma, check_p13_ed_dma, check_p14_selection_size]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(O)


@pytest.mark.parametrize("cfg_id,kw", [(2, dict(T=8192)), (4, dict(B=2, T_range=(6000, 9000))),
                                       (3, dict(B=1, T=20000, steps=1))])
def test_p8_needles_recalled(cfg_id, kw):
    check_p8_needles_recalled(O, cfg_id, **kw)
