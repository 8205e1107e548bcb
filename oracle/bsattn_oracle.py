"""Float64 CPU oracle for block-sparse decode attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, links or runs this
file: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it. It shares no code with the CUDA library; the only code
both sides use is the seeded input generator in ``workloads/``.

What it computes, step by step, in the order and notation of the two method pages
("Technisches Resümee: NOSA: Native und Offloadable Sparse Attention", section
"Methodik / 1. Algorithmus: NOSA"; "Technische Samenvatting: Fluxion", sections
"Probleemstelling", "Kerninzichten" and "Systeemcomponenten"):

1. sub-block mean keys, the first stage of NOSA's two-stage pooling
   ("Blockweise Implementierung": mean pooling inside sub-blocks);
2. block scores, the second stage (max pooling at block level), shared across the
   GQA group (Fluxion, "Granularity-Budget Selector": GQA handled at group level);
3. per-unit selection: forced sink and local blocks; streaming heads keep only
   those (Fluxion, "Kerninzichten" item 2); retrieval heads add a top-k of the
   block scores; NOSA dual heads add Gamma_e (top-k_e of query-agnostic
   pre-exponential eviction logits under the strict eviction rule) and Gamma_q
   (query-aware top-(k - k_e)) ("Dual-Selection-Mechanismus", "ED-DMA");
4. softmax attention over only the tokens of the selected blocks (Fluxion,
   "Probleemstelling" item 1: sparse attention over the selected KV blocks); and
   its ED-DMA variant, where each block's pre-exponential eviction logit is added to
   the logits of its tokens, so its exponential is taken only in the attention
   (NOSA, "ED-DMA"; a reading, see ed_dma_attention);
5. the set-difference of the selection against the previous step (NOSA,
   "2. System: NOSI": set-difference kernels for block swapping);
6. the swap that set-difference drives: the bookkeeping of a GPU block cache holding
   exactly the selected blocks (NOSA, "2. System: NOSI"; "Lokalitätsgarantie").

All arithmetic is float64 on logical (unpaged) arrays; bf16 inputs are widened
exactly. The pages give no formulas, so where they are silent the plainest reading
is taken; every such reading is a named argument or constant below:

* group reduction over the G query heads: max (``group_reduce="max"``); the mean
  of the per-head max-pooled scores is the alternative;
* sink and local windows are counted in tokens and covered by whole blocks; forced
  blocks sit outside the budget k; the partial tail block is always forced;
* candidates are the complete blocks outside the forced set;
* ties between equal keys go to the lower block index;
* Gamma_q's budget is k - k_e even when fewer than k_e blocks are eligible for
  Gamma_e; the strict eviction rule applies to Gamma_e's pool only;
* scale 1/sqrt(d) in both scores and attention.

* ED-DMA in attention: the block's eviction logit is an additive logit bias of
  each of its tokens (``ed_dma_attention``); plain softmax over the selection stays
  the default.

Parity unpinned (no page value fixes them; every pin below holds under each
alternative): the group reduction (max vs mean), the sink/local sizes chosen for
the synthetic configurations, the rounding of the budget fraction to k, the
per-block granularity of eviction logits, and the additive-bias reading of ED-DMA
itself (its pins fix the formula as read, not the reading).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# Head classes as encoded in the inputs.
STREAMING = 0
RETRIEVAL = 1
DUAL = 2

# Near-tie rule for parity of selections: the k-th and (k+1)-th keys closer than
# this relative gap (plus an absolute floor) make a unit's selection ambiguous.
NEAR_TIE_REL = 1e-4
NEAR_TIE_ABS = 1e-6


# ---------------------------------------------------------------------------
# 1. Sub-block mean keys (NOSA, "Blockweise Implementierung", first pooling stage)
# ---------------------------------------------------------------------------
def sub_block_range(j: int, s: int, T: int) -> tuple[int, int]:
    """Tokens [lo, hi) of sub-block j of size s when the cache holds T tokens."""
    return j * s, min((j + 1) * s, T)


def sub_block_means(K: np.ndarray, T: int, s: int) -> np.ndarray:
    """kbar[j] = mean of K[t] over the tokens present in sub-block j; shape [ceil(T/s)][d]."""
    n_sub = -(-T // s)
    out = np.empty((n_sub, K.shape[1]), dtype=np.float64)
    for j in range(n_sub):
        lo, hi = sub_block_range(j, s, T)
        out[j] = np.asarray(K[lo:hi], dtype=np.float64).mean(axis=0)
    return out


def update_sub_block(kbar: np.ndarray, K: np.ndarray, T: int, s: int) -> np.ndarray:
    """After appending token T-1, recompute only the sub-block that holds it."""
    j = (T - 1) // s
    n_sub = j + 1
    if kbar.shape[0] < n_sub:
        grown = np.empty((n_sub, kbar.shape[1]), dtype=np.float64)
        grown[:kbar.shape[0]] = kbar
        kbar = grown
    lo, hi = sub_block_range(j, s, T)
    kbar[j] = np.asarray(K[lo:hi], dtype=np.float64).mean(axis=0)
    return kbar


# ---------------------------------------------------------------------------
# 2. Block scores (NOSA second pooling stage; Fluxion GQA group level)
# ---------------------------------------------------------------------------
def block_scores(q: np.ndarray, kbar: np.ndarray, T: int, g: int, s: int,
                 group_reduce: str = "max") -> np.ndarray:
    """S[c] for every block c < ceil(T/g).

    sigma_h(j) = (q_h . kbar_j) / sqrt(d);  per head, max over the present sub-blocks
    of block c; then over the G heads of the group, max (or mean).
    """
    G, d = q.shape
    n_sub = -(-T // s)
    sigma = (np.asarray(q, np.float64) @ kbar[:n_sub].T) / math.sqrt(d)   # [G][n_sub]
    per_block = g // s
    n_blk = -(-T // g)
    S = np.empty(n_blk, dtype=np.float64)
    for c in range(n_blk):
        j_lo, j_hi = c * per_block, min((c + 1) * per_block, n_sub)
        per_head = sigma[:, j_lo:j_hi].max(axis=1)
        if group_reduce == "max":
            S[c] = per_head.max()
        elif group_reduce == "mean":
            S[c] = per_head.mean()
        else:
            raise ValueError(group_reduce)
    return S


# ---------------------------------------------------------------------------
# 3. Selection (Fluxion streaming/retrieval; NOSA dual selection)
# ---------------------------------------------------------------------------
def forced_blocks(T: int, g: int, sink_tokens: int, local_tokens: int) -> list[int]:
    """Sink blocks [0, ceil(sink/g)) united with local blocks [floor(max(0,T-local)/g), ceil(T/g))."""
    n_blk = -(-T // g)
    n_sink = min(-(-sink_tokens // g), n_blk)
    local_lo = max(0, T - local_tokens) // g
    return sorted(set(range(0, n_sink)) | set(range(local_lo, n_blk)))


def candidate_blocks(T: int, g: int, sink_tokens: int, local_tokens: int) -> list[int]:
    """Complete blocks outside the forced set."""
    forced = set(forced_blocks(T, g, sink_tokens, local_tokens))
    n_blk = -(-T // g)
    return [c for c in range(n_blk) if c not in forced and (c + 1) * g <= T]


def top_k(keys, pool, k: int) -> list[int]:
    """The first k of ``pool`` ordered by (key descending, index ascending)."""
    if k <= 0:
        return []
    return sorted(pool, key=lambda c: (-float(keys[c]), c))[:k]


def boundary_pair(keys, pool, k: int):
    """(k-th, (k+1)-th) keys of ``pool`` in selection order, or None when no boundary exists."""
    if k <= 0 or len(pool) <= k:
        return None
    order = sorted(pool, key=lambda c: (-float(keys[c]), c))
    return float(keys[order[k - 1]]), float(keys[order[k]])


def is_near_tie(pair) -> bool:
    if pair is None:
        return False
    a, b = pair
    return abs(a - b) <= NEAR_TIE_REL * max(abs(a), abs(b)) + NEAR_TIE_ABS


@dataclass
class Selection:
    sel: list                      # ascending block indices
    gamma_e: list = field(default_factory=list)
    gamma_q: list = field(default_factory=list)
    alive: np.ndarray | None = None
    boundary: tuple | None = None  # (k-th, (k+1)-th) score of the query-aware top-k

    @property
    def near_tie(self) -> bool:
        return is_near_tie(self.boundary)


def select_unit(cls: int, T: int, g: int, sink_tokens: int, local_tokens: int, k: int, k_e: int,
                scores=None, evict=None, alive=None) -> Selection:
    """Selected blocks of one unit at one step.

    Streaming: S = F.  Retrieval: S = F + top_k(scores over C).
    Dual: Gamma_e = top_{k_e}(evict over C and alive); every other block of C is
    dead from now on; Gamma_q = top_{k-k_e}(scores over C minus Gamma_e);
    S = F + Gamma_e + Gamma_q.
    """
    F = forced_blocks(T, g, sink_tokens, local_tokens)
    if cls == STREAMING:
        return Selection(sel=F)
    C = candidate_blocks(T, g, sink_tokens, local_tokens)
    if cls == RETRIEVAL:
        chosen = top_k(scores, C, k)
        return Selection(sel=sorted(set(F) | set(chosen)), gamma_q=sorted(chosen),
                         boundary=boundary_pair(scores, C, k))
    if cls == DUAL:
        alive = np.array(alive, dtype=np.uint8, copy=True)
        pool_e = [c for c in C if alive[c]]
        gamma_e = top_k(evict, pool_e, k_e)
        in_e = set(gamma_e)
        for c in C:
            alive[c] = 1 if c in in_e else 0
        rest = [c for c in C if c not in in_e]
        gamma_q = top_k(scores, rest, k - k_e)
        return Selection(sel=sorted(set(F) | in_e | set(gamma_q)), gamma_e=sorted(gamma_e),
                         gamma_q=sorted(gamma_q), alive=alive,
                         boundary=boundary_pair(scores, rest, k - k_e))
    raise ValueError(f"unknown head class {cls}")


# ---------------------------------------------------------------------------
# 4. Attention over the selected blocks only
# ---------------------------------------------------------------------------
def selected_tokens(sel, g: int, T: int) -> np.ndarray:
    """Token positions of the selected blocks, each block clipped to t < T."""
    parts = [np.arange(c * g, min((c + 1) * g, T)) for c in sel]
    return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)


def sparse_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, sel, g: int, T: int):
    """o_h = sum_t softmax_t(q_h.K[t]/sqrt(d)) V[t] and lse_h = log sum_t exp(q_h.K[t]/sqrt(d)),
    t over the selected tokens. Returns (o [G][d], lse [G])."""
    G, d = q.shape
    U = selected_tokens(sel, g, T)
    Ku = np.asarray(K[U], dtype=np.float64)
    Vu = np.asarray(V[U], dtype=np.float64)
    logits = (np.asarray(q, np.float64) @ Ku.T) / math.sqrt(d)           # [G][|U|]
    m = logits.max(axis=1, keepdims=True)
    w = np.exp(logits - m)
    l = w.sum(axis=1)
    o = (w @ Vu) / l[:, None]
    lse = m[:, 0] + np.log(l)
    return o, lse


def ed_dma_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, sel, g: int, T: int, e_blocks):
    """Attention of the ED-DMA variant ("Technisches Resümee: NOSA", Methodik /
    1. Algorithmus: NOSA, ED-DMA: blocks are chosen on the eviction head's
    pre-exponential logits, and the exponential is applied only in the attention).

    Reading: the pre-exponential eviction logit e[b] of block b enters the softmax as
    an additive logit of every selected token t of that block, b = t // g:
        logit_h(t) = q_h.K[t]/sqrt(d) + e[t // g]
        o_h = sum_t softmax_t(logit_h(t)) V[t],  lse_h = log sum_t exp(logit_h(t)),
    so exp(e[b]) first appears here, as a factor of the block's attention weights. A
    block with e[b] = -inf drops out; when no token is left, o_h = 0 and lse_h = -inf.
    The tokens are those of sparse_attention (selected blocks clipped to t < T).
    Returns (o [G][d], lse [G])."""
    G, d = q.shape
    U = selected_tokens(sel, g, T)
    e = np.asarray(e_blocks, dtype=np.float64)
    bias = e[U // g] if U.size else np.zeros(0)
    keep = bias > -np.inf
    if not keep.any():
        return np.zeros((G, d)), np.full(G, -np.inf)
    U, bias = U[keep], bias[keep]
    Ku = np.asarray(K[U], dtype=np.float64)
    Vu = np.asarray(V[U], dtype=np.float64)
    logits = (np.asarray(q, np.float64) @ Ku.T) / math.sqrt(d) + bias[None, :]   # [G][|U|]
    m = logits.max(axis=1, keepdims=True)
    w = np.exp(logits - m)
    l = w.sum(axis=1)
    o = (w @ Vu) / l[:, None]
    lse = m[:, 0] + np.log(l)
    return o, lse


# ---------------------------------------------------------------------------
# 5. Set-difference against the previous step
# ---------------------------------------------------------------------------
def setdiff(prev, cur):
    """(added, removed) = (cur minus prev, prev minus cur), both ascending."""
    p, c = set(int(x) for x in prev), set(int(x) for x in cur)
    return sorted(c - p), sorted(p - c)


# ---------------------------------------------------------------------------
# 6. Set-difference-driven block swap into a GPU block cache
# ---------------------------------------------------------------------------
def block_swap(slot_block, block_slot, added, removed):
    """One step's cache bookkeeping ("Technisches Resümee: NOSA", Methodik / 2. System:
    NOSI: the KV cache in minimal block units, set-difference kernels for block
    swapping; Lokalitätsgarantie: blocks kept between steps stay in the GPU cache).

    slot_block[s] is the block held by slot s (-1 free); block_slot[c] the slot of
    block c (-1 not cached). Readings where the page is silent: the removed blocks
    leave first; then the added blocks, in ascending order, take the free slots in
    ascending slot order; a block is cached exactly while it is selected. Returns the
    new (slot_block, block_slot) and the (block, slot) pairs whose pages are copied;
    added blocks beyond the free slots are not placed."""
    sb = np.array(slot_block, dtype=np.int64).copy()
    bs = np.array(block_slot, dtype=np.int64).copy()
    for c in removed:
        s = int(bs[c])
        if s >= 0:
            sb[s] = -1
        bs[c] = -1
    free = [s for s in range(sb.size) if sb[s] < 0]
    copies = []
    for i, c in enumerate(sorted(int(x) for x in added)):
        if i >= len(free):
            break
        sb[free[i]] = c
        bs[c] = free[i]
        copies.append((c, free[i]))
    return sb, bs, copies


def cache_page_table(block_slot, u: int, g: int, T: int, n_row: int, slots: int, pages_per_slot: int):
    """Page-table row of unit u over the cache: logical page p of a cached block c lies
    in device page (u * slots + slot) * pages_per_slot + (p - c * g/16) when it holds
    tokens (16 p < T); every other entry is -1."""
    ppb = g // 16
    row = np.full(n_row, -1, dtype=np.int64)
    for c, s in enumerate(block_slot):
        if s < 0:
            continue
        for j in range(ppb):
            lp = c * ppb + j
            if lp < n_row and lp * 16 < T:
                row[lp] = (u * slots + int(s)) * pages_per_slot + j
    return row


# ---------------------------------------------------------------------------
# One decode step over a workload
# ---------------------------------------------------------------------------
@dataclass
class UnitState:
    kbar: np.ndarray | None = None
    alive: np.ndarray | None = None
    prev_sel: list = field(default_factory=list)


@dataclass
class UnitStep:
    T: int
    sel: Selection
    scores: np.ndarray | None
    o: np.ndarray | None
    lse: np.ndarray | None
    added: list
    removed: list


def init_state(wl, units=None) -> dict:
    """Per-unit state before the first decode step: summaries of the prefilled tokens,
    every block alive, empty previous selection."""
    units = range(wl.U) if units is None else units
    state = {}
    for u in units:
        b = wl.unit_seq(u)
        Tp = int(wl.T_prefill[b])
        st = UnitState()
        st.kbar = sub_block_means(wl.K64(u), Tp, int(wl.s[u])) if Tp > 0 else np.zeros((0, wl.d))
        if wl.cls[u] == DUAL:
            st.alive = np.ones(-(-wl.T_cap // int(wl.g[u])), dtype=np.uint8)
        state[u] = st
    return state


def decode_step(wl, step: int, state: dict, units=None, group_reduce: str = "max", attend_units=None,
                ed_dma: bool = False) -> dict:
    """Run one decode step for ``units`` (default: all); update ``state`` in place.

    ``attend_units``: when given, the attention output (o, lse) is computed only for
    these units and is None for the others; every other result is computed for all
    ``units``. ``ed_dma``: the attention of every unit is ed_dma_attention with the
    unit's eviction logits (``wl.evict[u]``) as the block logits; otherwise plain
    sparse_attention."""
    units = range(wl.U) if units is None else units
    out = {}
    for u in units:
        st = state[u]
        b = wl.unit_seq(u)
        T = wl.T(step, b)
        g, s = int(wl.g[u]), int(wl.s[u])
        K = wl.K64(u)
        st.kbar = update_sub_block(st.kbar, K, T, s)
        q = wl.q64(step, u)
        cls = int(wl.cls[u])
        scores = None
        if cls != STREAMING:
            scores = block_scores(q, st.kbar, T, g, s, group_reduce)
        evict = wl.evict[u] if cls == DUAL else None
        sel = select_unit(cls, T, g, int(wl.sink[u]), int(wl.local[u]), int(wl.k[u]),
                          int(wl.k_e[u]), scores, evict, st.alive)
        if cls == DUAL:
            st.alive = sel.alive
        o = lse = None
        if attend_units is None or u in attend_units:
            if ed_dma:
                o, lse = ed_dma_attention(q, K, wl.V64(u), sel.sel, g, T, wl.evict[u])
            else:
                o, lse = sparse_attention(q, K, wl.V64(u), sel.sel, g, T)
        added, removed = setdiff(st.prev_sel, sel.sel)
        st.prev_sel = list(sel.sel)
        out[u] = UnitStep(T=T, sel=sel, scores=scores, o=o, lse=lse, added=added, removed=removed)
    return out
