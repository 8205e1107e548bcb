"""Step-by-step parity of the CUDA path against the float64 oracle.

Tolerances (floating point; integer outputs are compared exactly):
* attention output: max-abs 2e-3 and max-rel 1e-2, the relative error taken against
  max(|ref|, 0.2) so that near-zero references fall under the absolute bound;
  lse: max-abs 2e-3;
* sub-block means: fp32 sums of at most s bf16 values (|x| <= ~30 with planted
  needles and sink): |err| <= s * 2^-24 * sum|x| well under 1e-4 absolute;
* block scores: dot products of 128 terms on the tensor cores with fp32 operands split
  into tf32 high parts and remainders (each product within 2^-19 of its value) and
  fp32 accumulation: |err| <= (128 * 2^-24 + 2^-19) * ||q|| ||kbar|| / sqrt(d), at
  most ~2.5e-4 for the planted needles; 3e-4 absolute plus 1e-5 relative is allowed.
Selections and set-differences must match exactly wherever the oracle's k-th and
(k+1)-th keys are not a near-tie; at a near-tie the oracle's selection is fed to the
GPU attention and set-difference so that both sides keep the same state.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from long_context_serving_gb300 import bsattn as B
from long_context_serving_gb300.layer import PagedLayer
from oracle import bsattn_oracle as O

ATT_ABS, ATT_REL, REL_FLOOR = 2e-3, 1e-2, 0.2
LSE_ABS = 2e-3
SUM_ABS = 1e-4
SCORE_ABS, SCORE_REL = 3e-4, 1e-5


# Near-ties may make up at most this share of the compared selections (at least one).
# With thousands of candidates a unit's k-th and (k+1)-th scores often lie within the
# near-tie band (up to about one retrieval unit-step in six at 8,193 candidates), so
# this cap is loose; what keeps a near-tie from hiding a wrong selection is the exact
# check below: every selection the GPU makes, near-tie or not, must be the selection
# rule applied to the GPU's own fp32 scores, and those scores must match the oracle's.
NEAR_TIE_SHARE = 0.25


@dataclass
class Report:
    att_abs: float = 0.0
    att_rel: float = 0.0
    lse_abs: float = 0.0
    sum_abs: float = 0.0
    score_abs: float = 0.0
    compared_units: int = 0        # unit-steps whose attention and set-difference were compared
    selection_checks: int = 0      # unit-steps whose selection was compared (exact or near-tie)
    near_ties: int = 0
    exact_selections: int = 0
    skipped_near_tie: int = 0      # fused mode: near-tie unit-steps whose GPU selection differed
    notes: list = field(default_factory=list)

    def check(self):
        print(f"parity: {self.exact_selections} exact selections, {self.near_ties} near-ties "
              f"(of {self.selection_checks}), {self.compared_units} attention unit-steps, "
              f"{self.skipped_near_tie} skipped; att abs {self.att_abs:.2e} rel {self.att_rel:.2e}, "
              f"lse {self.lse_abs:.2e}, sums {self.sum_abs:.2e}, scores {self.score_abs:.2e}")
        assert self.att_abs <= ATT_ABS, self
        assert self.att_rel <= ATT_REL, self
        assert self.lse_abs <= LSE_ABS, self
        assert self.sum_abs <= SUM_ABS, self
        assert self.score_abs <= SCORE_ABS, self
        assert self.compared_units > 0
        assert self.exact_selections + self.near_ties == self.selection_checks, self
        assert self.near_ties <= max(1, NEAR_TIE_SHARE * self.selection_checks), self
        assert self.skipped_near_tie <= self.near_ties, self


def attention_errors(o_gpu: np.ndarray, o_ref: np.ndarray):
    diff = np.abs(o_gpu.astype(np.float64) - o_ref)
    return float(diff.max()), float((diff / np.maximum(np.abs(o_ref), REL_FLOOR)).max())


def run_parity(wl, units=None, group_reduce="max", steps=None, summary_rows_sample=None, seed=0,
               fused=False, q_fp32=False, attend_units=None, ed_dma=False) -> Report:
    """Drive the GPU path and the oracle through the same steps on ``units`` (default all).

    ``attend_units``: compare the attention output only on these units (the oracle's
    float64 attention is the slow part at full size); summaries, scores, selections,
    alive masks and set-differences are compared on every unit of ``units``.

    ``q_fp32``: queries passed as fp32 (the same values) over the bf16 cache.
    ``ed_dma``: the attention adds each block's eviction logit to its tokens' logits
    (oracle: ed_dma_attention) on both sides.
    ``fused``: run each step through bs_decode_step (one call for all five steps). A
    near-tie unit whose GPU selection differs from the oracle's then cannot be given
    the oracle's selection before attention: its attention and set-difference are not
    compared at that step, and the oracle's selection is written back as the previous
    selection of the next step, so both sides continue from the same state."""
    units = list(range(wl.U)) if units is None else list(units)
    reduce_code = B.BS_GROUP_MAX if group_reduce == "max" else B.BS_GROUP_MEAN
    rng = np.random.default_rng(seed)
    layer = PagedLayer(wl, q_fp32=q_fp32, ed_dma=ed_dma)
    layer.prefill()
    state = O.init_state(wl, units)
    rep = Report()
    G = wl.G
    for step in range(wl.steps if steps is None else steps):
        layer.append(step)
        if fused:
            layer.fused_step(step, reduce_code)         # advances: results sit in 1 - cur
            sel_buf = 1 - layer.cur
        else:
            layer.update_summaries(step)
            layer.score(step, reduce_code)
            layer.select(step)
            sel_buf = layer.cur
        torch.cuda.synchronize()
        alive_before = {u: None if state[u].alive is None else state[u].alive.copy() for u in units}
        res = O.decode_step(wl, step, state, units, group_reduce, attend_units=attend_units, ed_dma=ed_dma)
        gsel = layer.selection(sel_buf)
        scores = layer.scores.cpu().numpy()
        alive = layer.alive.cpu().numpy() if layer.alive is not None else None
        override = {}
        for u in units:
            r = res[u]
            g, s = int(wl.g[u]), int(wl.s[u])
            n_sub = -(-r.T // s)
            # a1: summaries (the updated row plus every row or a sample)
            rows = np.arange(n_sub) if summary_rows_sample is None else np.unique(
                np.concatenate([[n_sub - 1], rng.integers(0, n_sub, size=min(summary_rows_sample, n_sub))]))
            gs = layer.unit_summaries(u, n_sub)
            rep.sum_abs = max(rep.sum_abs, float(np.abs(gs[rows] - state[u].kbar[rows]).max()))
            if wl.cls[u] != O.STREAMING:
                # a2: scores on candidates (-inf elsewhere from the stand-alone call)
                C = O.candidate_blocks(r.T, g, int(wl.sink[u]), int(wl.local[u]))
                if C:
                    err = np.abs(scores[u, C] - r.scores[C]) - SCORE_REL * np.abs(r.scores[C])
                    rep.score_abs = max(rep.score_abs, float(err.max()))
                if not fused:
                    mask = np.ones(layer.max_blocks, bool)
                    mask[C] = False
                    assert np.all(scores[u, mask] == -np.inf), (step, u)
            # a3: the selection kernel is exact on its own inputs: the oracle's rule applied
            # to the GPU's fp32 scores (and the same eviction logits and alive mask) gives
            # the GPU's selection, at every unit, near-tie or not.
            if wl.cls[u] != O.STREAMING:
                ev = None
                if wl.cls[u] == O.DUAL:
                    ev = np.full(layer.max_blocks, -np.inf)
                    n_ev = min(layer.max_blocks, wl.evict.shape[1])
                    ev[:n_ev] = wl.evict[u, :n_ev]
                own = O.select_unit(int(wl.cls[u]), r.T, g, int(wl.sink[u]), int(wl.local[u]), int(wl.k[u]),
                                    int(wl.k_e[u]), scores[u].astype(np.float64), ev, alive_before[u])
                assert gsel[u] == own.sel, (step, u, "selection differs from the rule on the GPU's own scores")
            rep.selection_checks += 1
            if r.sel.near_tie:
                rep.near_ties += 1
                if gsel[u] != r.sel.sel:
                    override[u] = r.sel.sel
            else:
                assert gsel[u] == r.sel.sel, (step, u, gsel[u], r.sel.sel)
                rep.exact_selections += 1
            if wl.cls[u] == O.DUAL:
                n_blk = -(-r.T // g)
                assert np.array_equal(alive[u, :n_blk], r.sel.alive[:n_blk]), (step, u)
        if fused:
            # Only a near-tie unit whose selection differs is left out at this step.
            skip = set(override)
            assert all(res[u].sel.near_tie for u in skip), skip
            rep.skipped_near_tie += len(skip)
            if override:
                layer.set_selection(override, which=sel_buf)
        else:
            skip = set()
            if override:
                layer.set_selection(override)
            layer.attend(step)
            layer.setdiff()
        torch.cuda.synchronize()
        out = layer.out.cpu().numpy()
        lse = layer.lse.cpu().numpy()
        added = layer.added.cpu().numpy()
        added_cnt = layer.added_cnt.cpu().numpy()
        removed = layer.removed.cpu().numpy()
        removed_cnt = layer.removed_cnt.cpu().numpy()
        for u in units:
            r = res[u]
            if u in skip:
                continue
            assert added[u, :added_cnt[u]].tolist() == r.added, (step, u)
            assert removed[u, :removed_cnt[u]].tolist() == r.removed, (step, u)
            assert (added[u, added_cnt[u]:] == -1).all() and (removed[u, removed_cnt[u]:] == -1).all()
            if r.o is None:
                continue
            b, hk = divmod(u, wl.Hkv)
            a_abs, a_rel = attention_errors(out[b, hk * G:(hk + 1) * G], r.o)
            rep.att_abs, rep.att_rel = max(rep.att_abs, a_abs), max(rep.att_rel, a_rel)
            rep.lse_abs = max(rep.lse_abs, float(np.abs(lse[b, hk * G:(hk + 1) * G] - r.lse).max()))
            rep.compared_units += 1
        if not fused:
            layer.advance()
        status = layer.read_status()
        assert status == 0, f"device status {status}: {B.status_string(status)}"
    return rep
