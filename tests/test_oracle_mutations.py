"""Planted mistakes in the oracle must each fail at least one pin.

Every mutation below is a plausible slip (a dropped term, a wrong index, a swapped
operand, a reversed tie-break). Each is planted into the oracle module on the CPU
with monkeypatch and the full set of pins from ``test_oracle_pins`` is run: at least
one pin has to fail, which shows the pins constrain that part of the oracle.
"""
import math

import numpy as np
import pytest

from oracle import bsattn_oracle as O
from test_oracle_pins import ALL_CHECKS


def _means_divide_by_s(K, T, s):
    n_sub = -(-T // s)
    out = np.empty((n_sub, K.shape[1]))
    for j in range(n_sub):
        lo, hi = O.sub_block_range(j, s, T)
        out[j] = np.asarray(K[lo:hi], np.float64).sum(axis=0) / s
    return out


def _scores_no_scale(q, kbar, T, g, s, group_reduce="max"):
    return ORIG["block_scores"](q, kbar, T, g, s, group_reduce) * math.sqrt(q.shape[1])


def _scores_mean_pool(q, kbar, T, g, s, group_reduce="max"):
    G, d = q.shape
    n_sub = -(-T // s)
    sigma = (q @ kbar[:n_sub].T) / math.sqrt(d)
    r = g // s
    return np.array([sigma[:, c * r:min((c + 1) * r, n_sub)].mean(axis=1).max()
                     for c in range(-(-T // g))])


def _scores_head0_only(q, kbar, T, g, s, group_reduce="max"):
    return ORIG["block_scores"](q[:1], kbar, T, g, s, group_reduce)


def _topk_high_index(keys, pool, k):
    return [] if k <= 0 else sorted(pool, key=lambda c: (-float(keys[c]), -c))[:k]


def _topk_ascending(keys, pool, k):
    return [] if k <= 0 else sorted(pool, key=lambda c: (float(keys[c]), c))[:k]


def _forced_local_ceil(T, g, sink_tokens, local_tokens):
    n_blk = -(-T // g)
    n_sink = min(-(-sink_tokens // g), n_blk)
    local_lo = -(-max(0, T - local_tokens) // g)
    return sorted(set(range(n_sink)) | set(range(local_lo, n_blk)))


def _forced_sink_floor(T, g, sink_tokens, local_tokens):
    n_blk = -(-T // g)
    local_lo = max(0, T - local_tokens) // g
    return sorted(set(range(min(sink_tokens // g, n_blk))) | set(range(local_lo, n_blk)))


def _candidates_with_forced(T, g, sink_tokens, local_tokens):
    return [c for c in range(-(-T // g)) if (c + 1) * g <= T]


def _attention_no_clip(q, K, V, sel, g, T):
    T2 = min(K.shape[0], max((c + 1) * g for c in sel)) if sel else T
    return ORIG["sparse_attention"](q, K, V, sel, g, T2)


def _attention_values_are_keys(q, K, V, sel, g, T):
    return ORIG["sparse_attention"](q, K, K, sel, g, T)


def _attention_no_scale(q, K, V, sel, g, T):
    return ORIG["sparse_attention"](q * math.sqrt(q.shape[1]), K, V, sel, g, T)


def _attention_lse_no_max(q, K, V, sel, g, T):
    o, lse = ORIG["sparse_attention"](q, K, V, sel, g, T)
    U = O.selected_tokens(sel, g, T)
    m = ((q @ np.asarray(K[U]).T) / math.sqrt(q.shape[1])).max(axis=1)
    return o, lse - m


def _select_no_eviction(cls, T, g, sink_tokens, local_tokens, k, k_e, scores=None, evict=None, alive=None):
    if cls == O.DUAL and alive is not None:
        alive = np.ones_like(alive)
    r = ORIG["select_unit"](cls, T, g, sink_tokens, local_tokens, k, k_e, scores, evict, alive)
    if r.alive is not None:
        r.alive[:] = 1
    return r


def _select_gq_overlaps(cls, T, g, sink_tokens, local_tokens, k, k_e, scores=None, evict=None, alive=None):
    r = ORIG["select_unit"](cls, T, g, sink_tokens, local_tokens, k, k_e, scores, evict, alive)
    if cls == O.DUAL:
        C = O.candidate_blocks(T, g, sink_tokens, local_tokens)
        r.gamma_q = sorted(O.top_k(scores, C, k - k_e))
        r.sel = sorted(set(O.forced_blocks(T, g, sink_tokens, local_tokens)) | set(r.gamma_e) | set(r.gamma_q))
    return r


def _setdiff_swapped(prev, cur):
    a, r = ORIG["setdiff"](prev, cur)
    return r, a


def _update_wrong_sub_block(kbar, K, T, s):
    return ORIG["update_sub_block"](kbar, K, T + 1 if T < K.shape[0] else T, s)


def _swap_no_free(slot_block, block_slot, added, removed):
    return ORIG["block_swap"](slot_block, block_slot, added, [])


def _swap_highest_slot_first(slot_block, block_slot, added, removed):
    sb = np.array(slot_block).copy()
    bs = np.array(block_slot).copy()
    for c in removed:
        if bs[c] >= 0:
            sb[bs[c]] = -1
        bs[c] = -1
    free = [s for s in range(sb.size) if sb[s] < 0][::-1]
    copies = []
    for n, c in enumerate(sorted(added)):
        if n < len(free):
            sb[free[n]], bs[c] = c, free[n]
            copies.append((c, free[n]))
    return sb, bs, copies


def _ed_dma_bias_scaled(q, K, V, sel, g, T, e_blocks):
    return ORIG["ed_dma_attention"](q, K, V, sel, g, T, np.asarray(e_blocks, np.float64) / math.sqrt(q.shape[1]))


def _ed_dma_bias_by_position(q, K, V, sel, g, T, e_blocks):
    e = np.asarray(e_blocks, np.float64)
    e2 = np.full_like(e, -np.inf)      # block sel[i] takes e[i], the logit of its position
    for i, c in enumerate(sel):
        if i < e.size:
            e2[c] = e[i]
    return ORIG["ed_dma_attention"](q, K, V, sel, g, T, e2)


def _ed_dma_bias_negated(q, K, V, sel, g, T, e_blocks):
    e = np.asarray(e_blocks, np.float64)
    return ORIG["ed_dma_attention"](q, K, V, sel, g, T, np.where(np.isneginf(e), e, -e))


def _ed_dma_exp_applied_early(q, K, V, sel, g, T, e_blocks):
    return ORIG["ed_dma_attention"](q, K, V, sel, g, T, np.exp(np.asarray(e_blocks, np.float64)))


def _decode_step_ed_dma_ignored(wl, step, state, units=None, group_reduce="max", attend_units=None, ed_dma=False):
    return ORIG["decode_step"](wl, step, state, units, group_reduce, attend_units)


def _select_forced_within_budget(cls, T, g, sink_tokens, local_tokens, k, k_e, scores=None, evict=None,
                                 alive=None):
    """The budget read as including the forced blocks: top_(k - |F|) of the candidates."""
    kk = max(0, k - len(O.forced_blocks(T, g, sink_tokens, local_tokens)))
    return ORIG["select_unit"](cls, T, g, sink_tokens, local_tokens, kk, min(k_e, kk), scores, evict, alive)


def _decode_step_variant(drop: str):
    """decode_step with one piece of its carried state left out: 'alive' (the eviction
    mask is not carried), 'prev_sel' (the previous selection is not recorded) or 'kbar'
    (the updated summaries are not stored back)."""
    def step(wl, step_i, state, units=None, group_reduce="max", attend_units=None, ed_dma=False):
        units = range(wl.U) if units is None else units
        out = {}
        for u in units:
            st = state[u]
            b = wl.unit_seq(u)
            T = wl.T(step_i, b)
            g, s = int(wl.g[u]), int(wl.s[u])
            K = wl.K64(u)
            kbar = O.update_sub_block(st.kbar if drop != "kbar" else st.kbar.copy(), K, T, s)
            if drop != "kbar":
                st.kbar = kbar
            q = wl.q64(step_i, u)
            cls = int(wl.cls[u])
            scores = O.block_scores(q, kbar, T, g, s, group_reduce) if cls != O.STREAMING else None
            evict = wl.evict[u] if cls == O.DUAL else None
            sel = O.select_unit(cls, T, g, int(wl.sink[u]), int(wl.local[u]), int(wl.k[u]), int(wl.k_e[u]),
                                scores, evict, st.alive)
            if cls == O.DUAL and drop != "alive":
                st.alive = sel.alive
            o = lse = None
            if attend_units is None or u in attend_units:
                if ed_dma:
                    o, lse = O.ed_dma_attention(q, K, wl.V64(u), sel.sel, g, T, wl.evict[u])
                else:
                    o, lse = O.sparse_attention(q, K, wl.V64(u), sel.sel, g, T)
            added, removed = O.setdiff(st.prev_sel, sel.sel)
            if drop != "prev_sel":
                st.prev_sel = list(sel.sel)
            out[u] = O.UnitStep(T=T, sel=sel, scores=scores, o=o, lse=lse, added=added, removed=removed)
        return out
    return step


MUTATIONS = {
    "means_divide_by_s": ("sub_block_means", _means_divide_by_s),
    "scores_no_scale": ("block_scores", _scores_no_scale),
    "scores_mean_pool": ("block_scores", _scores_mean_pool),
    "scores_head0_only": ("block_scores", _scores_head0_only),
    "topk_high_index_ties": ("top_k", _topk_high_index),
    "topk_ascending": ("top_k", _topk_ascending),
    "forced_local_ceil": ("forced_blocks", _forced_local_ceil),
    "forced_sink_floor": ("forced_blocks", _forced_sink_floor),
    "candidates_with_forced": ("candidate_blocks", _candidates_with_forced),
    "attention_no_clip": ("sparse_attention", _attention_no_clip),
    "attention_values_are_keys": ("sparse_attention", _attention_values_are_keys),
    "attention_no_scale": ("sparse_attention", _attention_no_scale),
    "attention_lse_no_max": ("sparse_attention", _attention_lse_no_max),
    "select_no_eviction": ("select_unit", _select_no_eviction),
    "select_gamma_q_overlaps_gamma_e": ("select_unit", _select_gq_overlaps),
    "select_forced_within_budget": ("select_unit", _select_forced_within_budget),
    "setdiff_swapped": ("setdiff", _setdiff_swapped),
    "update_wrong_sub_block": ("update_sub_block", _update_wrong_sub_block),
    "swap_no_free": ("block_swap", _swap_no_free),
    "swap_highest_slot_first": ("block_swap", _swap_highest_slot_first),
    "decode_step_alive_not_carried": ("decode_step", _decode_step_variant("alive")),
    "decode_step_prev_sel_not_carried": ("decode_step", _decode_step_variant("prev_sel")),
    "decode_step_kbar_not_stored": ("decode_step", _decode_step_variant("kbar")),
    "ed_dma_bias_scaled": ("ed_dma_attention", _ed_dma_bias_scaled),
    "ed_dma_bias_by_position": ("ed_dma_attention", _ed_dma_bias_by_position),
    "ed_dma_bias_negated": ("ed_dma_attention", _ed_dma_bias_negated),
    "ed_dma_exp_applied_early": ("ed_dma_attention", _ed_dma_exp_applied_early),
    "decode_step_ed_dma_ignored": ("decode_step", _decode_step_ed_dma_ignored),
}

ORIG = {name: getattr(O, name) for name, _ in MUTATIONS.values()}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(mutation, monkeypatch):
    name, fn = MUTATIONS[mutation]
    monkeypatch.setattr(O, name, fn)
    failed = []
    for check in ALL_CHECKS:
        try:
            check(O)
        except Exception as e:  # noqa: BLE001 - any failure of a pin counts
            failed.append((check.__name__, type(e).__name__))
            break                # one failing pin is enough
    assert failed, f"no pin caught the planted mistake {mutation}"


def test_decode_step_variant_is_faithful_when_nothing_is_dropped():
    """The decode_step copy the carry mutations start from equals the oracle's own when
    nothing is dropped, so each of those mutations differs from the oracle by its one
    left-out assignment only."""
    from workloads import make_workload
    wl = make_workload(5, seed=3, B=1, T=2040, steps=10)
    a, b = O.init_state(wl), O.init_state(wl)
    same = _decode_step_variant("")
    for step in range(wl.steps):
        ra, rb = O.decode_step(wl, step, a), same(wl, step, b)
        for u in range(wl.U):
            assert ra[u].sel.sel == rb[u].sel.sel and ra[u].added == rb[u].added
            assert ra[u].removed == rb[u].removed
            np.testing.assert_array_equal(ra[u].o, rb[u].o)
            np.testing.assert_array_equal(a[u].alive, b[u].alive)
