#!/usr/bin/env python
"""Decode-step benchmark of block-sparse decode attention on one GB300 per rank.

Workload (default): the Llama-3.1-8B-shaped 128K decode layer with mixed heads (batch
4, 32 query / 8 KV heads, head_dim 128, T = 131069 growing to 131076 over 8 decode
steps, per KV head a block size in {16, 32, 64, 128} with sub-block g/4, a budget of
2-10% of the context and a streaming or retrieval class drawn from a seed), seeded
synthetic bf16 data. One step = one decode step through 4 layers, each layer with its
own cache, summaries and selection buffers (about 8.6 GB, far above the 129 MB L2,
so no layer's data is cache-resident when its turn comes); the 8 decode steps of the
workload are replayed in order, again and again (one CUDA graph per decode step). Per
layer: sub-block update, block scores, selection, sparse attention, set-difference,
through one bs_decode_step call (two launches); --path calls uses the five separate
calls instead. --config 2|4|5 runs the other workloads the same way.

Reported: microseconds per layer per decode step (lower is better) and the fraction of
the HBM roofline the layer step reaches, an end-to-end figure through pinned host
buffers, the float64 oracle timed on the host cores (one thread and all cores), SM
clocks, and the same layer-step figure for the Llama 32K and Qwen 32-64K workloads.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--config C]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse decode attn µs/layer/step; achieved HBM GB/s vs ~8 TB/s peak"
UNIT = "us/layer/step"
DEFAULT_CFG = 3
# Workloads of the path: description and layer buffers per step (each step's working
# set several times the L2, within a few GB of HBM).
WORKLOADS = {
    2: ("llama3.1-8b decode layer at 32K: B=1, Hq=32, Hkv=8, d=128, T=32768, g=32, s=8; 4 streaming heads "
        "(sink 128 + window 2048), 4 retrieval heads (5% budget = 51 blocks)", 32),
    3: ("llama3.1-8b decode layer at 128K, mixed heads: B=4, Hq=32, Hkv=8, d=128, T=131069..131076 over 8 "
        "decode steps, per KV head g in {16,32,64,128} (s=g/4), budget 2-10%, streaming/retrieval 50/50", 4),
    4: ("qwen2.5-7b decode layer, low-rank K/V: B=8, Hq=28, Hkv=4, d=128, T_b in [32768, 65536], g=64, "
        "s=16, all retrieval, 5% budget", 8),
    5: ("nosa dual selection: B=64, Hq=32, Hkv=8, d=128, T=16377..16392 over 16 decode steps, g=64, s=16, "
        "k=32, k_e=24", 2),
}
# Other workloads measured beside the default one in the same run (layer step only).
EXTRA_CFGS = (2, 4)
FALLBACK_HBM_GBS = 6800.0
PAGE = 16


# ---------------------------------------------------------------------------
# Oracle timing (CPU baseline and the reference arm). A child process without CUDA
# generates the workload and times the oracle's per-step work over every unit of one
# layer, with the units spread over forked worker processes (one BLAS thread each).
# ---------------------------------------------------------------------------
_ORACLE_SNIPPET = r"""
import json, multiprocessing as mp, os, sys, time
sys.path.insert(0, %(root)r)
from workloads import make_workload
from oracle import bsattn_oracle as O

wl = make_workload(%(cfg)d, seed=0)
units = list(range(wl.U))

def worker(conn, mine):
    state = O.init_state(wl, mine)
    conn.send("ready")
    while True:
        i = conn.recv()
        if i is None:
            return
        O.decode_step(wl, i %% wl.steps, state, mine)
        conn.send("done")

def run(n, reps, warm):
    ctx = mp.get_context("fork")
    pipes, procs = [], []
    for w in range(n):
        a, b = ctx.Pipe()
        p = ctx.Process(target=worker, args=(b, units[w::n]))
        p.start()
        pipes.append(a)
        procs.append(p)
    for a in pipes:
        a.recv()
    walls = []
    for i in range(warm + reps):
        t = time.perf_counter()
        for a in pipes:
            a.send(i)
        for a in pipes:
            a.recv()
        if i >= warm:
            walls.append(time.perf_counter() - t)
    for a in pipes:
        a.send(None)
    for p in procs:
        p.join()
    return walls

workers = min(%(workers)d, len(units))
res = {"workers": workers, "U": wl.U, "multi": run(workers, %(reps)d, %(warm)d)}
if %(single_reps)d > 0:
    res["single"] = run(1, %(single_reps)d, 0)
print(json.dumps(res))
"""


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(cfg: int, reps: int, warm: int, single_reps: int = 0, workers: int | None = None) -> dict:
    """The oracle's per-step work (summary update, scores, selection, attention,
    set-difference) over every unit of one layer of workload ``cfg``: ``reps`` timed
    decode steps after ``warm`` untimed ones on ``workers`` processes (default: every
    host core), plus ``single_reps`` steps on one process."""
    workers = workers or host_cores()
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = _ORACLE_SNIPPET % dict(root=ROOT, cfg=cfg, reps=reps, warm=warm, workers=workers,
                                  single_reps=single_reps)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    res = json.loads(r.stdout.strip().splitlines()[-1])
    multi_us = statistics.median(res["multi"]) * 1e6
    out = {"value": round(multi_us, 1), "unit": UNIT, "cores": res["workers"], "kind": "oracle",
           "sample": (f"one layer of the workload ({res['U']} units) per decode step, the workload's decode "
                      f"steps in order; {reps} timed steps (median) after {warm} untimed; float64 numpy, units "
                      f"spread over {res['workers']} processes of one thread; K/V generation and prefill "
                      f"summaries untimed"),
           "mean_step_ms": round(statistics.fmean(res["multi"]) * 1e3, 3)}
    if res.get("single"):
        out["single_thread"] = {"value": round(statistics.median(res["single"]) * 1e6, 1), "unit": UNIT,
                                "cores": 1, "steps": len(res["single"])}
    return out


def run_reference(args) -> None:
    """The reference arm: the oracle (the pages ship no code) on the host cores, on the
    same workload, metric and unit; rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    t0 = time.perf_counter()
    res = time_oracle(args.config, args.steps, args.warmup)
    wall = time.perf_counter() - t0
    line = {"impl": "reference", "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["mean_step_ms"],
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOADS[args.config][0], "layers_per_step": 1, "kv_dtype": "bf16",
                       "q_dtype": "bf16", "note": "one layer per timed step; value is per layer per step"},
            "cpu_baseline": {k: res[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": res["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(wall, 1)}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------
_CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                 "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                 "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    def __init__(self, gpu_index: int, path: str | None):
        self.path = path
        self.proc = None
        try:
            self.out = open(path, "w") if path else subprocess.PIPE
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + ",".join(_CLOCK_FIELDS),
                                          "--format=csv,noheader,nounits", "-lms", "200", "-i", str(gpu_index)],
                                         stdout=self.out, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            text = self.proc.communicate(timeout=5)[0] if self.path is None else None
        except subprocess.TimeoutExpired:
            self.proc.kill()
            text = None
        if self.path:
            self.out.close()
            text = open(self.path).read()
        rows = [[x.strip() for x in ln.split(",")] for ln in (text or "").splitlines() if ln.strip()]
        sm = [float(r[1]) for r in rows if len(r) == len(_CLOCK_FIELDS) and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) == len(_CLOCK_FIELDS) and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows if len(r) == len(_CLOCK_FIELDS)
                          for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sm)}


# ---------------------------------------------------------------------------
# Algorithmic bytes (what the method must move; intermediates a fused kernel could
# avoid -- block scores, split partials -- are not counted)
# ---------------------------------------------------------------------------
def _geom(T, g, sink, local):
    n_blk = -(-T // g)
    n_sink = min(-(-sink // g), n_blk)
    local_lo = max(0, T - local) // g
    return n_blk, n_sink, local_lo, n_sink, max(local_lo, n_sink)


def algorithmic_bytes(wl, sel_lists, prev_lists, step: int = 0):
    """Bytes one decode step of one layer must move at decode step ``step``, per step of
    the path, given each unit's selection and the previous step's."""
    d, G = wl.d, wl.G
    out = {"score": 0, "attn": 0, "select": 0, "setdiff": 0, "summary_update": 0}
    for u in range(wl.U):
        T = wl.T(step, u // wl.Hkv)
        g, s = int(wl.g[u]), int(wl.s[u])
        n_blk, _, _, c_lo, c_hi = _geom(T, g, int(wl.sink[u]), int(wl.local[u]))
        n_cand = c_hi - c_lo
        # a1: the touched sub-block's tokens read, one summary row written
        out["summary_update"] += (((T - 1) % s) + 1) * d * 2 + d * 4
        if wl.cls[u] != 0:
            # dual units need no scores of their Gamma_e blocks
            n_scored = n_cand - (min(int(wl.k_e[u]), n_cand) if wl.cls[u] == 2 else 0)
            out["score"] += n_scored * (g // s) * d * 4 + G * d * 2 + n_scored * 4
            out["select"] += n_cand * 4 + len(sel_lists[u]) * 4 + (n_blk * 5 if wl.cls[u] == 2 else 0)
        sel = sel_lists[u]
        tokens = sum(min(g, T - c * g) for c in sel)
        pages = sum(-(-min(g, T - c * g) // PAGE) for c in sel)
        out["attn"] += tokens * d * 2 * 2 + G * d * 2 + pages * 4 + len(sel) * 4 + G * (d + 1) * 4
        out["setdiff"] += (len(sel) + len(prev_lists[u])) * 4 * 2
    out["layer_step"] = sum(out.values())
    return out


def _json_default(o):
    """numpy scalars in the JSON line become plain numbers."""
    if hasattr(o, "item"):
        return o.item()
    raise TypeError(f"not JSON serializable: {type(o).__name__}")


def csrc_sha() -> str:
    """Hash of every CUDA source and header of the library (any change invalidates counters)."""
    d = os.path.join(ROOT, "long_context_serving_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh")):
            h.update(name.encode())
            h.update(open(os.path.join(d, name), "rb").read())
    return h.hexdigest()[:16]


def _measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if no kernel source changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel, {}).get(workload)
    if not rec or rec.get("csrc_sha") != csrc_sha():
        return None
    return rec["bytes_per_launch"]


def _peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm"):
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k]), "of measured"
        except (ValueError, OSError):
            pass
    return FALLBACK_HBM_GBS, "of fallback"


# ---------------------------------------------------------------------------
# Block swap from host memory (the offload path): bandwidth of a full cache refill,
# beside a plain pinned-host copy of the same bytes as the host link's reference
# ---------------------------------------------------------------------------
def measure_block_swap(layer, wl, B, torch, reps: int = 20) -> dict:
    """Time bs_block_swap filling an empty GPU block cache with one layer's whole
    selection from pinned host memory (every selected page, K and V, crosses the host
    link once per call), alternating with a call that empties it; and one pinned-host
    to device copy of the same number of bytes."""
    dev = layer.device
    U, MS = wl.U, layer.max_sel
    slots, pps = MS, int(wl.g.max()) // 16
    n = U * slots * pps
    ck = torch.empty((n, 16, wl.d), dtype=layer.k_pool.dtype, device=dev)
    cv = torch.empty_like(ck)
    cpt = torch.full_like(layer.page_table, -1)
    sb = torch.full((U, slots), -1, dtype=torch.int32, device=dev)
    bsl = torch.full((U, layer.max_blocks), -1, dtype=torch.int32, device=dev)
    cache = B.BlockCache(k_pool=ck.data_ptr(), v_pool=cv.data_ptr(), page_table=cpt.data_ptr(),
                         slot_block=sb.data_ptr(), block_slot=bsl.data_ptr(), slots_per_unit=slots, pages_per_slot=pps)
    hk = layer.k_pool.cpu().pin_memory()
    hv = layer.v_pool.cpu().pin_memory()
    host = B.HostKV(k_pool=hk.data_ptr(), v_pool=hv.data_ptr(), page_table=layer.page_table.data_ptr(),
                    n_pages=int(wl.n_pages))
    sel, cnt = layer.sel[0], layer.cnt[0]
    zero = torch.zeros_like(cnt)
    T = layer.seq_lens[0]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    lists = layer.selection(0)
    Tn = [int(wl.T(0, u // wl.Hkv)) for u in range(U)]
    pages = sum(-(-min(int(wl.g[u]), Tn[u] - int(c) * int(wl.g[u])) // PAGE) for u in range(U) for c in lists[u])
    nbytes = int(pages) * 2 * PAGE * int(wl.d) * (2 if wl.dtype == "bf16" else 4)

    def fill():
        B.block_swap(layer.dims, layer.cfg, T, host, cache, sel, cnt, sel, zero, status)

    def empty():
        B.block_swap(layer.dims, layer.cfg, T, host, cache, sel, zero, sel, cnt, status)

    for _ in range(3):
        fill()
        empty()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    total_ms = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fill()
        e1.record(stream)
        empty()
        torch.cuda.synchronize()
        total_ms += e0.elapsed_time(e1)
    assert int(status.item()) == 0, "device status set during the block swap"
    us = total_ms * 1000.0 / reps
    # The host link's reference: one pinned-host -> device copy (cudaMemcpyAsync) of the
    # same byte count.
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    for _ in range(3):
        dst.copy_(src, non_blocking=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        dst.copy_(src, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    copy_us = e0.elapsed_time(e1) * 1000.0 / reps
    del hk, hv, src, dst
    gbs = nbytes / (us * 1e-6) / 1e9
    copy_gbs = nbytes / (copy_us * 1e-6) / 1e9
    return {"workload": "one layer's whole selection (every unit) copied into an empty GPU block cache",
            "bytes_per_call": nbytes, "us_per_call": round(us, 3), "gbs": round(gbs, 1),
            "source": "pinned host memory read by the kernel over the host link (unified addressing)",
            "host_link_copy": {"what": "one pinned-host to device cudaMemcpyAsync of the same byte count",
                               "us": round(copy_us, 3), "gbs": round(copy_gbs, 1)},
            "frac_of_host_link_copy": round(gbs / copy_gbs, 3)}


# ---------------------------------------------------------------------------
# CPU/GPU split attention: the host cores' share and the GPU merge
# ---------------------------------------------------------------------------
def measure_cpu_split(layer, wl, B, torch, reps: int = 10) -> dict:
    """Time bs_cpu_sparse_attn on every other selected block of every unit (about half
    the layer's selected KV, read from host memory by all host cores) and bs_lse_merge
    combining its result with a GPU partial result."""
    import numpy as np
    dev = layer.device
    lists = layer.selection(0)
    MS = layer.max_sel
    idx = np.full((wl.U, MS), -1, np.int32)
    cnt = np.zeros(wl.U, np.int32)
    for u, lst in enumerate(lists):
        part = lst[1::2]
        idx[u, :len(part)] = part
        cnt[u] = len(part)
    hk, hv = layer.k_pool.cpu(), layer.v_pool.cpu()
    pt, seq, gs = layer.page_table.cpu(), layer.seq_lens[0].cpu(), layer.cfg_arrays["block_tokens"].cpu()
    qh = layer.q[0].cpu()
    out = np.zeros((wl.B, wl.Hq, wl.d), np.float32)
    lse = np.zeros((wl.B, wl.Hq), np.float32)
    host = B.HostKV(k_pool=hk.data_ptr(), v_pool=hv.data_ptr(), page_table=0, n_pages=int(wl.n_pages))
    tables = B.HostTables(page_table=pt.data_ptr(), seq_lens=seq.data_ptr(), block_tokens=gs.data_ptr())
    threads = host_cores()
    Tn = [int(wl.T(0, u // wl.Hkv)) for u in range(wl.U)]
    tokens = sum(min(int(wl.g[u]), Tn[u] - int(c) * int(wl.g[u])) for u in range(wl.U) for c in idx[u, :cnt[u]])
    nbytes = int(tokens) * 2 * int(wl.d) * (2 if wl.dtype == "bf16" else 4)
    B.cpu_sparse_attn(layer.dims, qh, host, tables, idx, cnt, out, lse, threads)
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        B.cpu_sparse_attn(layer.dims, qh, host, tables, idx, cnt, out, lse, threads)
        times.append(time.perf_counter() - t0)
    cpu_us = statistics.median(times) * 1e6
    ob, lb = torch.as_tensor(out, device=dev), torch.as_tensor(lse, device=dev)
    oa, la = layer.out.clone(), layer.lse.clone()
    stream = torch.cuda.current_stream()
    for _ in range(3):
        B.lse_merge(layer.dims, oa, la, ob, lb, oa, la)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(100):
        B.lse_merge(layer.dims, oa, la, ob, lb, oa, la)
    e1.record(stream)
    torch.cuda.synchronize()
    return {"cpu_share": "every other selected block of every unit", "cpu_bytes": nbytes, "cpu_threads": threads,
            "cpu_us": round(cpu_us, 1), "cpu_gbs": round(nbytes / (cpu_us * 1e-6) / 1e9, 2),
            "merge_us": round(e0.elapsed_time(e1) * 10.0, 3)}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
_IO_OUTPUTS = ("out", "lse", "added", "added_cnt", "removed", "removed_cnt")


def _pack_io(layers, torch, dev):
    """Rebind every layer's queries and step outputs to views of contiguous device
    buffers: q_all[step] holds that decode step's queries of every layer (one copy per
    step), o_all every layer's outputs (regions 256-byte aligned)."""
    steps = layers[0].q.shape[0]
    q_all = torch.empty((steps, len(layers)) + tuple(layers[0].q.shape[1:]), dtype=layers[0].q.dtype, device=dev)
    for i, layer in enumerate(layers):
        q_all[:, i].copy_(layer.q)
        layer.q = q_all[:, i]
    al = lambda n: (n + 255) // 256 * 256  # noqa: E731
    per = sum(al(getattr(layers[0], n).numel() * getattr(layers[0], n).element_size()) for n in _IO_OUTPUTS)
    o_all = torch.zeros(len(layers) * per, dtype=torch.uint8, device=dev)
    for i, layer in enumerate(layers):
        off = i * per
        for n in _IO_OUTPUTS:
            t = getattr(layer, n)
            nb = t.numel() * t.element_size()
            v = o_all[off:off + nb].view(t.dtype).view(t.shape)
            v.copy_(t)
            setattr(layer, n, v)
            off += al(nb)
    return q_all, o_all


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (a time); x itself on a single process."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class Bench:
    """The layers of one workload on one GPU, their per-step CUDA graphs and timers."""

    def __init__(self, cfg: int, n_layers: int, path: str, rank: int, dev, torch, B):
        from long_context_serving_gb300.layer import PagedLayer
        from workloads import make_workload
        self.torch, self.B, self.dev = torch, B, dev
        self.cfg, self.path = cfg, path
        # Each rank serves its own batch (weak scaling): independent units, no exchange.
        self.wl = make_workload(cfg, seed=rank)
        self.layers = []
        for _ in range(n_layers):
            layer = PagedLayer(self.wl, device=dev, preload_all=True)
            layer._K = layer._V = None                  # logical copies are not needed any more
            self.layers.append(layer)
        torch.cuda.empty_cache()
        for layer in self.layers:
            layer.prefill()
        torch.cuda.synchronize()
        # Queries of each decode step and the outputs of every layer in contiguous device
        # buffers: the end-to-end step moves its inputs and results with one copy each way.
        self.q_all, self.o_all = _pack_io(self.layers, torch, dev)
        # One graph per decode step of the workload; step i writes selection buffer i % 2
        # (an even number of graphs, so replaying them in order keeps alternating).
        self.n_graph = self.wl.steps if self.wl.steps % 2 == 0 else 2 * self.wl.steps
        for i in range(self.n_graph):                   # eager warm-up, also the first selections
            self._set_parity(i)
            for layer in self.layers:
                self.layer_calls(layer, i % self.wl.steps)
        torch.cuda.synchronize()
        codes = [layer.read_status() for layer in self.layers]
        assert not any(codes), f"device status set during warm-up: {codes}"
        self.cap = torch.cuda.Stream(device=dev)
        self.graphs = []
        for i in range(self.n_graph):
            g = torch.cuda.CUDAGraph()
            self._set_parity(i)
            with torch.cuda.graph(g, stream=self.cap):
                for layer in self.layers:
                    self.layer_calls(layer, i % self.wl.steps)
            self.graphs.append(g)
        self.launches_per_layer = bn_launches(path, self.layers[0], B)
        self.launches_per_step = self.launches_per_layer * n_layers

    def _set_parity(self, i):
        for layer in self.layers:
            layer.cur = i % 2

    def layer_calls(self, layer, step):
        if self.path == "fused":
            self.B.decode_step(layer.dims, layer.kv_at(layer.seq_lens[step]), layer.cfg, layer.step_io(step))
        else:
            layer.update_summaries(step)
            layer.score(step)
            layer.select(step)
            layer.attend(step)
            layer.setdiff()

    def timed(self, graph_list, n, barrier, start_at=0):
        torch = self.torch
        stream = torch.cuda.current_stream()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(n):
            graph_list[(start_at + i) % len(graph_list)].replay()
        end.record(stream)
        torch.cuda.synchronize()
        barrier()
        return start.elapsed_time(end)

    def step_bytes(self):
        """Algorithmic bytes of one layer step, averaged over the workload's decode steps
        (each step's selection read back after replaying that step's graph)."""
        per = []
        for i in range(self.n_graph):
            self.graphs[i].replay()
            self.torch.cuda.synchronize()
            cur = self.layers[0].selection(i % 2)
            prev = self.layers[0].selection(1 - i % 2)
            per.append(algorithmic_bytes(self.wl, cur, prev, i % self.wl.steps))
        keys = per[0].keys()
        return {k: int(round(statistics.fmean(p[k] for p in per))) for k in keys}

    def free(self):
        self.graphs = []
        self.layers = []
        self.q_all = self.o_all = None
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    from long_context_serving_gb300 import bsattn as B
    from long_context_serving_gb300.build import build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
    B.lib()

    def barrier():
        if world > 1:
            dist.barrier()

    n_layers = args.layers or WORKLOADS[args.config][1]
    bn = Bench(args.config, n_layers, args.path, rank, dev, torch, B)
    wl, layers = bn.wl, bn.layers

    # Clock samples cover warm-up, the timed region and, when the timed region is
    # shorter than a second, a soak of further replays so that the sampler sees load.
    sampler = ClockSampler(local, f"{args.clocks_csv}.rank{rank}" if args.clocks_csv else None)
    for i in range(args.warmup):
        bn.graphs[i % bn.n_graph].replay()
    ms = bn.timed(bn.graphs, args.steps, barrier, start_at=args.warmup % bn.n_graph)
    ms = max_over_ranks(ms, dev)
    soak_s = 0.0
    while soak_s < 1.0 - ms / 1000:
        t0 = time.perf_counter()
        for i in range(max(20, 200 // n_layers)):
            bn.graphs[i % bn.n_graph].replay()
        torch.cuda.synchronize()
        soak_s += time.perf_counter() - t0
    clocks = sampler.stop()
    ms_per_step = ms / args.steps
    value = ms_per_step * 1000.0 / n_layers
    assert all(layer.read_status() == 0 for layer in layers), "device status set during the timed region"

    nbytes = bn.step_bytes()
    peak, peak_note = _peak_hbm()
    layer_gbs = nbytes["layer_step"] / (value * 1e-6) / 1e9

    # Stand-alone per-call launch times (graphs of one call type over the layers, decode
    # step 0): context for the layer step, not its roofline.
    def kernel_graph(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=bn.cap):
            for layer in layers:
                fn(layer)
        return g

    # Buffer 0 must hold decode step 0's selection for the stand-alone calls at step 0.
    bn._set_parity(0)
    bn.graphs[0].replay()
    torch.cuda.synchronize()
    per_kernel = {}
    for name, fn in (("attn", lambda l: l.attend(0)), ("score", lambda l: l.score(0)),
                     ("select", lambda l: l.select(0)), ("summary_update", lambda l: l.update_summaries(0)),
                     ("setdiff", lambda l: l.setdiff())):
        g = kernel_graph(fn)
        for _ in range(3):
            g.replay()
        reps = max(20, args.steps)
        per_kernel[name] = bn.timed([g], reps, barrier) * 1000.0 / (reps * n_layers)    # us per launch
    assert all(layer.read_status() == 0 for layer in layers), "device status set by the stand-alone calls"
    b0 = algorithmic_bytes(wl, layers[0].selection(0), layers[0].selection(1), 0)
    standalone = {k: {"us": round(per_kernel[k], 3),
                      "gbs": round(b0[k] / (per_kernel[k] * 1e-6) / 1e9, 1) if k in ("attn", "score") else None}
                  for k in per_kernel}
    # The roofline of the timed path: one layer step is the launches of bs_decode_step,
    # each a programmatic dependent of the one before (overlapping), timed as one.
    # traffic: DRAM bytes of one layer step's kernels (one ncu capture of each on a
    # small case of this workload, profiles/), only while no library source changed.
    traffic = _measured_traffic("layer_step", wl.name) if args.path == "fused" else None
    roofline = {"bound": "hbm", "achieved": round(layer_gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(layer_gbs / peak, 4), "traffic": traffic,
                "kernel": (f"bs_decode_step = {step_kernels(wl, bn.launches_per_layer)} (one layer step; "
                           "the launches overlap through programmatic dependent launch)" if args.path == "fused"
                           else "the five calls of one layer step"),
                "peak_source": peak_note, "algorithmic_bytes_per_launch": nbytes["layer_step"],
                "launch_us": round(value, 3),
                "timed_as": "CUDA events around the replayed decode-step graphs, per layer per step"}

    # End to end: every step copies that decode step's queries of all layers from pinned
    # host memory (one copy), replays the step and reads back out, lse and the
    # set-difference lists of all layers into pinned host memory (one copy).
    q_host = torch.empty_like(bn.q_all, device="cpu").pin_memory()
    q_host.copy_(bn.q_all.cpu())
    o_host = torch.empty_like(bn.o_all, device="cpu").pin_memory()
    h2d = q_host[0].numel() * q_host.element_size()
    d2h = o_host.numel() * o_host.element_size()

    def e2e_step(i):
        k = i % bn.n_graph
        bn.q_all[k % wl.steps].copy_(q_host[k % wl.steps], non_blocking=True)
        bn.graphs[k].replay()
        o_host.copy_(bn.o_all, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for i in range(args.warmup):
        e2e_step(i)
    barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(args.warmup + i)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, dev)
    e2e_value = e2e_s / args.steps * 1e6 / n_layers

    swap = measure_block_swap(layers[0], wl, B, torch) if rank == 0 and not args.no_extras else None
    split = measure_cpu_split(layers[0], wl, B, torch) if rank == 0 and not args.no_extras else None
    launches_per_layer, launches_per_step = bn.launches_per_layer, bn.launches_per_step
    bn.free()
    del bn, layers

    # The same layer-step measurement on the other 32K-128K workloads.
    extras = {}
    if not args.no_extras:
        for c in EXTRA_CFGS:
            if c == args.config:
                continue
            eb = Bench(c, WORKLOADS[c][1], args.path, rank, dev, torch, B)
            for i in range(3):
                eb.graphs[i % eb.n_graph].replay()
            n = max(20, args.steps)
            ems = max_over_ranks(eb.timed(eb.graphs, n, barrier), dev)
            ev = ems / n * 1000.0 / WORKLOADS[c][1]
            assert all(layer.read_status() == 0 for layer in eb.layers), f"device status set (config {c})"
            eby = eb.step_bytes()["layer_step"]
            extras[f"config{c}"] = {"workload": WORKLOADS[c][0], "layers_per_step": WORKLOADS[c][1],
                                    "value": round(ev, 3), "unit": UNIT, "steps": n,
                                    "algorithmic_bytes_per_layer_step": eby,
                                    "gbs": round(eby / (ev * 1e-6) / 1e9, 1),
                                    "frac": round(eby / (ev * 1e-6) / 1e9 / peak, 4)}
            eb.free()
            del eb

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = time_oracle(args.config, reps=args.cpu_reps, warm=1, single_reps=args.cpu_single_reps)
        cpu.pop("mean_step_ms", None)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": WORKLOADS[args.config][0], "layers_per_step": n_layers,
                           "decode_steps_cycled": wl.steps, "kv_dtype": wl.dtype, "q_dtype": wl.dtype,
                           "l2": f"inputs larger than L2: {n_layers} distinct layer buffers per step",
                           "graph": (f"one CUDA graph per decode step, {n_layers} layers x "
                                     f"{launches_per_layer} launches each"),
                           "ranks": world, "parallelism": f"replicas x{world}, units independent",
                           "path": args.path},
                "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h},
                "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
                "algorithmic_bytes_per_layer": nbytes,
                "standalone_calls_us_per_launch": standalone,
                "other_workloads": extras or None,
                "block_swap": swap,
                "cpu_gpu_split": split}
        print(json.dumps(line, default=_json_default), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bn_launches(path: str, layer, B) -> int:
    """Kernel launches of one layer step: those of one bs_decode_step call (the library
    says how many for the layer's dims), or five for the separate calls."""
    if path != "fused":
        return 5
    n = B.decode_step_launches(layer.dims)
    assert n > 0, "bad dims"
    return n


def step_kernels(wl, launches: int) -> str:
    """The kernels of one bs_decode_step call, in launch order."""
    front = "step_score_balanced + step_select_kernel" if launches == 3 else "step_front_kernel"
    return f"{front} + {'attn_mma_kernel' if wl.dtype == 'bf16' else 'attn_ffma_kernel'}"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-reps", type=int, default=5, help="timed oracle steps on all host cores")
    ap.add_argument("--cpu-single-reps", type=int, default=2, help="timed oracle steps on one core")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads, the block swap and the CPU/GPU split measurements")
    ap.add_argument("--path", choices=["fused", "calls"], default="fused",
                    help="fused: bs_decode_step per layer; calls: the five separate calls per layer")
    ap.add_argument("--clocks-csv", default=None,
                    help="also keep the raw nvidia-smi clock samples in this file (one per rank)")
    ap.add_argument("--layers", type=int, default=None,
                    help="layer buffers per step (fewer only for profiling small cases)")
    ap.add_argument("--config", type=int, choices=sorted(WORKLOADS), default=DEFAULT_CFG,
                    help="workload (3, the default: Llama-3.1-8B shape at 128K with mixed heads)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
