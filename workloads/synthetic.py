"""Seeded synthetic workloads shaped like the pages' long-context decode settings.

The pages evaluate on LongBench, L-Eval, RULER and HELMET with Llama-3.1-8B and
Qwen2.5-7B models (Technische Samenvatting: Fluxion, section "Experimentele
Resultaten"; Technisches Resümee: NOSA, section "Experimentelle Ergebnisse").
None of those suites or weights is used here. These generators stand in for them:
they take only the model shapes (query/KV heads, head_dim) and the 8K-128K context
range, and fill K, V and q with seeded random values plus two planted structures:

* an attention sink at token 0 (its key scaled x8, its value scaled to 0.05 of its
  norm), the phenomenon named in Fluxion, "Kerninzichten" item 1;
* needle blocks whose keys are pushed toward the group-mean query, so that a
  retrieval head has something to retrieve.

Randomness: numpy ``Generator(PCG64)`` with one ``SeedSequence`` child per unit
(one unit = one (sequence, KV head) pair), one per sequence, one for per-head
parameters and one for the page permutation. Values are drawn in float32; bf16
inputs are rounded to nearest-even from those float32 values.

Nothing here computes a summary, a score, a selection or an attention output.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

# Head classes (Fluxion, "Kerninzichten" item 2 and "Systeemcomponenten"; NOSA
# dual selection, "1. Algorithmus: NOSA").
STREAMING = 0
RETRIEVAL = 1
DUAL = 2

PAGE_TOKENS = 16
CONFIG_IDS = (1, 2, 3, 4, 5)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (b + (((b >> 16) & np.uint32(1)) + np.uint32(0x7FFF))) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class Workload:
    """One seeded decode workload on logical (unpaged) arrays.

    Units are ordered u = b * Hkv + h_kv. At decode step i (0-based) the token at
    position ``T_prefill[b] + i`` has just been appended, so the cache holds
    ``T = T_prefill[b] + i + 1`` tokens and the current token sits at T - 1.
    """

    name: str
    cfg_id: int
    seed: int
    B: int
    Hq: int
    Hkv: int
    d: int
    dtype: str                      # "bf16" or "fp32": storage of K, V and q
    steps: int
    T_prefill: np.ndarray           # int64 [B]
    cls: np.ndarray                 # int32 [U]
    g: np.ndarray                   # int32 [U] block size in tokens
    s: np.ndarray                   # int32 [U] sub-block size in tokens
    k: np.ndarray                   # int32 [U] selected blocks outside the forced set
    k_e: np.ndarray                 # int32 [U] of which eviction-selected (dual units)
    sink: np.ndarray                # int32 [U] sink tokens
    local: np.ndarray               # int32 [U] local-window tokens
    K: np.ndarray                   # [U][T_cap][d] uint16 (bf16 bits) or float32
    V: np.ndarray                   # same as K
    q: np.ndarray                   # [steps][B][Hq][d] uint16 (bf16 bits) or float32
    evict: np.ndarray | None        # float32 [U][n_blk_cap] pre-exponential logits
    needles: list                   # per sequence: int64 token positions
    page_table: np.ndarray          # int32 [U][max_pages]; -1 where unused
    n_pages: int                    # physical pages in the pool

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def U(self) -> int:
        return self.B * self.Hkv

    @property
    def T_cap(self) -> int:
        return int(self.K.shape[1])

    def T(self, step: int, b: int) -> int:
        return int(self.T_prefill[b]) + step + 1

    def seq_lens(self, step: int) -> np.ndarray:
        return (self.T_prefill + step + 1).astype(np.int32)

    def unit_seq(self, u: int) -> int:
        return u // self.Hkv

    def _widen(self, a: np.ndarray) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f32(a).astype(np.float64)
        return np.asarray(a, dtype=np.float64)

    def K64(self, u: int) -> np.ndarray:
        """Keys of unit u as float64 (exact widening of the stored values)."""
        return self._widen(self.K[u])

    def V64(self, u: int) -> np.ndarray:
        return self._widen(self.V[u])

    def q64(self, step: int, u: int) -> np.ndarray:
        """The G query heads of unit u at a step, float64 [G][d]."""
        b, h = divmod(u, self.Hkv)
        return self._widen(self.q[step, b, h * self.G:(h + 1) * self.G])


def _budget_k(frac: float, T: int, g: int) -> int:
    # Budget fraction of the context's blocks, at least one block.
    return max(1, int(math.floor(frac * math.ceil(T / g))))


def _base_params(cfg_id: int, B, T, steps, Hq=None, Hkv=None, d=None):
    """Shapes and schedule of each configuration, before any random draw."""
    if cfg_id == 1:
        p = dict(name="tiny-check", B=1, Hq=4, Hkv=1, d=64, dtype="fp32", steps=1, T_first=2048,
                 n_needles=1)
    elif cfg_id == 2:
        p = dict(name="llama8b-32k", B=1, Hq=32, Hkv=8, d=128, dtype="bf16", steps=1,
                 T_first=32768, n_needles=4)
    elif cfg_id == 3:
        p = dict(name="llama8b-128k-mixed", B=4, Hq=32, Hkv=8, d=128, dtype="bf16", steps=8,
                 T_first=131069, n_needles=8)
    elif cfg_id == 4:
        p = dict(name="qwen7b-32k-64k-lowrank", B=8, Hq=28, Hkv=4, d=128, dtype="bf16", steps=1,
                 T_first=None, T_lo=32768, T_hi=65536, n_needles=4)
    elif cfg_id == 5:
        p = dict(name="nosa-dual-16k", B=64, Hq=32, Hkv=8, d=128, dtype="bf16", steps=16,
                 T_first=16377, n_needles=2)
    else:
        raise ValueError(f"unknown config {cfg_id}")
    if B is not None:
        p["B"] = B
    if steps is not None:
        p["steps"] = steps
    if T is not None:
        p["T_first"] = T
        p["T_lo"] = p["T_hi"] = T
    if Hq is not None:
        p["Hq"] = Hq
    if Hkv is not None:
        p["Hkv"] = Hkv
    if d is not None:
        p["d"] = d
    if p["Hq"] % p["Hkv"] != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return p


def make_workload(cfg_id: int, seed: int = 0, *, B: int | None = None, T: int | None = None,
                  steps: int | None = None, T_range: tuple | None = None, Hq: int | None = None,
                  Hkv: int | None = None, d: int | None = None) -> Workload:
    """Build configuration ``cfg_id`` (1..5) from ``seed``.

    Overrides shrink a configuration for tests: ``B`` sequences, ``T`` tokens in the
    cache at the first decode step (all sequences), ``T_range`` = (lo, hi) for the
    per-sequence length draw of configuration 4, ``steps`` decode steps, ``Hq`` and
    ``Hkv`` the query and KV head counts (other GQA group sizes; configuration 2 makes
    its KV heads 0-3 streaming and the rest retrieval), ``d`` the head dimension.
    """
    p = _base_params(cfg_id, B, T, steps, Hq, Hkv, d)
    if T_range is not None:
        p["T_lo"], p["T_hi"] = T_range
    Bn, Hq, Hkv, d, steps_n = p["B"], p["Hq"], p["Hkv"], p["d"], p["steps"]
    G = Hq // Hkv
    U = Bn * Hkv

    root = np.random.SeedSequence([seed, cfg_id])
    params_ss, seqs_ss, units_ss, pages_ss = root.spawn(4)
    prng = np.random.Generator(np.random.PCG64(params_ss))
    seq_rngs = [np.random.Generator(np.random.PCG64(c)) for c in seqs_ss.spawn(Bn)]
    unit_rngs = [np.random.Generator(np.random.PCG64(c)) for c in units_ss.spawn(U)]

    # --- sequence lengths -------------------------------------------------------
    if cfg_id == 4:
        T_first = np.array([int(r.integers(p["T_lo"], p["T_hi"], endpoint=True)) for r in seq_rngs],
                           dtype=np.int64)
    else:
        T_first = np.full(Bn, p["T_first"], dtype=np.int64)
    T_prefill = T_first - 1
    T_last = T_prefill + steps_n                       # tokens at the last step

    # --- per-unit head properties (inputs of the method, not outputs) -----------
    cls = np.empty(U, np.int32)
    g = np.empty(U, np.int32)
    s = np.empty(U, np.int32)
    k = np.zeros(U, np.int32)
    k_e = np.zeros(U, np.int32)
    sink = np.empty(U, np.int32)
    local = np.empty(U, np.int32)
    for u in range(U):
        b, h = divmod(u, Hkv)
        Tf = int(T_first[b])
        if cfg_id == 1:
            cls[u], g[u], s[u], k[u], sink[u], local[u] = RETRIEVAL, 64, 16, 4, 64, 64
        elif cfg_id == 2:
            g[u], s[u] = 32, 8
            if h < 4:
                cls[u], sink[u], local[u] = STREAMING, 128, 2048
            else:
                cls[u], sink[u], local[u] = RETRIEVAL, 32, 32
                k[u] = _budget_k(0.05, Tf, 32)
        elif cfg_id == 3:
            gg = int(prng.choice([16, 32, 64, 128]))
            frac = float(prng.uniform(0.02, 0.10))
            retrieval = bool(prng.random() < 0.5)
            g[u], s[u] = gg, gg // 4
            if retrieval:
                cls[u], sink[u], local[u] = RETRIEVAL, gg, gg
                k[u] = _budget_k(frac, Tf, gg)
            else:
                cls[u], sink[u], local[u] = STREAMING, 128, 2048
        elif cfg_id == 4:
            cls[u], g[u], s[u], sink[u], local[u] = RETRIEVAL, 64, 16, 64, 64
            k[u] = _budget_k(0.05, Tf, 64)
        else:
            cls[u], g[u], s[u], sink[u], local[u] = DUAL, 64, 16, 0, 1
            k[u], k_e[u] = 32, 24

    # --- needle positions, shared by all units of a sequence --------------------
    g_max = int(g.max())
    needles = []
    for b in range(Bn):
        us = range(b * Hkv, (b + 1) * Hkv)
        lo = max(int(math.ceil(sink[u] / g[u])) * int(g[u]) for u in us)
        hi = min(int(max(0, int(T_first[b]) - local[u]) // g[u]) * int(g[u]) for u in us)
        c_lo, c_hi = -(-lo // g_max), hi // g_max
        n = min(p["n_needles"], max(0, c_hi - c_lo))
        picks = seq_rngs[b].choice(np.arange(c_lo, c_hi), size=n, replace=False) if n else []
        needles.append(np.sort(np.asarray(picks, dtype=np.int64) * g_max))

    # --- K, V, q, eviction logits per unit ---------------------------------------
    T_cap = int(T_last.max())
    bf16 = p["dtype"] == "bf16"
    store = np.uint16 if bf16 else np.float32
    K = np.zeros((U, T_cap, d), dtype=store)
    V = np.zeros((U, T_cap, d), dtype=store)
    qf = np.empty((steps_n, Bn, Hq, d), dtype=np.float32)
    dual = bool((cls == DUAL).any())
    n_blk_cap = int(-(-T_cap // int(g.min())))
    evict = np.zeros((U, n_blk_cap), dtype=np.float32) if dual else None

    for u in range(U):
        b, h = divmod(u, Hkv)
        r = unit_rngs[u]
        Tu = int(T_last[b])
        if cfg_id == 4:
            # Low-rank keys and values: rank-32 signal plus N(0, 0.1^2) noise.
            WK = r.standard_normal((32, d), dtype=np.float32) * np.float32(math.sqrt(1.0 / 32))
            WV = r.standard_normal((32, d), dtype=np.float32) * np.float32(math.sqrt(1.0 / 32))
            a = r.standard_normal((G, 32), dtype=np.float32)
            q_base = a @ WK + np.float32(0.1) * r.standard_normal((G, d), dtype=np.float32)
            Ku = r.standard_normal((Tu, 32), dtype=np.float32) @ WK
            Ku += np.float32(0.1) * r.standard_normal((Tu, d), dtype=np.float32)
            Vu = r.standard_normal((Tu, 32), dtype=np.float32) @ WV
            Vu += np.float32(0.1) * r.standard_normal((Tu, d), dtype=np.float32)
        else:
            q_base = r.standard_normal((G, d), dtype=np.float32)
            Ku = r.standard_normal((Tu, d), dtype=np.float32)
            Vu = r.standard_normal((Tu, d), dtype=np.float32)
        # Attention sink at token 0.
        Ku[0] *= np.float32(8.0)
        Vu[0] *= np.float32(0.05)
        # Needle blocks: keys pushed toward the group-mean query direction.
        qbar = q_base.mean(axis=0)
        push = (np.float32(2.0 * math.sqrt(d)) * qbar / np.float32(np.linalg.norm(qbar))).astype(np.float32)
        gu = int(g[u])
        for pos in needles[b]:
            c = int(pos) // gu
            Ku[c * gu:min((c + 1) * gu, Tu)] += push
        if bf16:
            K[u, :Tu] = to_bf16_bits(Ku)
            V[u, :Tu] = to_bf16_bits(Vu)
        else:
            K[u, :Tu] = Ku
            V[u, :Tu] = Vu
        for i in range(steps_n):
            if steps_n > 1:
                qf[i, b, h * G:(h + 1) * G] = q_base + np.float32(0.3) * r.standard_normal((G, d), dtype=np.float32)
            else:
                qf[i, b, h * G:(h + 1) * G] = q_base
        if dual:
            evict[u] = r.standard_normal(n_blk_cap, dtype=np.float32)

    q = to_bf16_bits(qf) if bf16 else qf

    # --- physical page assignment (a seeded permutation of the pool) ------------
    pages_per_unit = np.array([-(-int(T_last[u // Hkv]) // PAGE_TOKENS) for u in range(U)], np.int64)
    n_pages = int(pages_per_unit.sum())
    perm = np.random.Generator(np.random.PCG64(pages_ss)).permutation(n_pages).astype(np.int32)
    max_pages = int(pages_per_unit.max())
    page_table = np.full((U, max_pages), -1, dtype=np.int32)
    off = 0
    for u in range(U):
        n = int(pages_per_unit[u])
        page_table[u, :n] = perm[off:off + n]
        off += n

    return Workload(name=p["name"], cfg_id=cfg_id, seed=seed, B=Bn, Hq=Hq, Hkv=Hkv, d=d,
                    dtype=p["dtype"], steps=steps_n, T_prefill=T_prefill, cls=cls, g=g, s=s, k=k,
                    k_e=k_e, sink=sink, local=local, K=K, V=V, q=q, evict=evict, needles=needles,
                    page_table=page_table, n_pages=n_pages)
