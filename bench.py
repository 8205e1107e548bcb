#!/usr/bin/env python
"""Decode-step benchmark of block-sparse decode attention on one GB300 per rank.

Workload: the Llama-3.1-8B-shaped 32K decode layer (batch 1, 32 query / 8 KV heads,
head_dim 128, T = 32768, block 32 / sub-block 8, KV heads 0-3 streaming with a
128-token sink and a 2048-token window, heads 4-7 retrieval with a 5% budget), seeded
synthetic bf16 data. One step = one decode step through 32 layers, each layer with
its own cache, summaries and selection buffers (about 0.5 GB touched per step, well
above the 129 MB L2, so no layer's data is cache-resident when its turn comes). Per
layer: sub-block update, block scores, selection, sparse attention, set-difference.
The 32 layers are captured in CUDA graphs (one per parity of the previous/current
selection buffers) and replayed. By default each layer is one bs_decode_step call (two
launches); --path calls uses the five separate calls instead.

Reported: microseconds per layer per decode step (lower is better), the roofline
of the dominant kernel against HBM bandwidth, an end-to-end figure through pinned
host buffers, the float64 oracle timed on the host cores, and SM clocks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
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
CFG_ID = 2
LAYERS = 32
WORKLOAD = ("llama3.1-8b decode layer: B=1, Hq=32, Hkv=8, d=128, T=32768, g=32, s=8; "
            "4 streaming heads (sink 128 + window 2048), 4 retrieval heads (5% budget = 51 blocks)")
# Other workloads of the same path (--config), measured beside the headline one; layer
# counts keep each step's working set several times the L2 within a few GB of HBM.
WORKLOADS = {
    2: (WORKLOAD, 32),
    3: ("llama3.1-8b decode layer at 128K, mixed heads: B=4, Hq=32, Hkv=8, d=128, T=131069, per-unit "
        "g in {16,32,64,128} (s=g/4), budget 2-10%, streaming/retrieval 50/50", 4),
    4: ("qwen2.5-7b decode layer, low-rank K/V: B=8, Hq=28, Hkv=4, d=128, T_b in [32768, 65536], g=64, "
        "s=16, all retrieval, 5% budget", 8),
    5: ("nosa dual selection: B=64, Hq=32, Hkv=8, d=128, T=16377, g=64, s=16, k=32, k_e=24", 2),
}
FALLBACK_HBM_GBS = 6800.0
PAGE = 16


def _config(extra=None):
    c = {"workload": WORKLOAD, "layers_per_step": LAYERS, "kv_dtype": "bf16", "q_dtype": "bf16",
         "l2": f"inputs larger than L2: {LAYERS} distinct layer buffers per step",
         "graph": f"CUDA graph of {LAYERS} layers"}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------------------
# Oracle timing (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
_ORACLE_SNIPPET = r"""
import json, sys, time
sys.path.insert(0, %r)
from workloads import make_workload
from oracle import bsattn_oracle as O
wl = make_workload(%d, seed=0)
state = O.init_state(wl)
reps, warm = %d, %d
for _ in range(warm):
    O.decode_step(wl, 0, state)
times = []
for _ in range(reps):
    t = time.perf_counter()
    O.decode_step(wl, 0, state)
    times.append(time.perf_counter() - t)
print(json.dumps({"times": times}))
"""


def time_oracle(reps: int, warm: int) -> dict:
    """Time the oracle's per-step work (summary update, scores, selection, attention,
    set-difference) on one layer of the workload, single-threaded, in a child process."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _ORACLE_SNIPPET % (ROOT, CFG_ID, reps, warm)], env=env,
                       capture_output=True, text=True, check=True)
    times = json.loads(r.stdout.strip().splitlines()[-1])["times"]
    us = statistics.median(times) * 1e6
    return {"value": round(us, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"one of the 32 layers, {reps} timed decode steps (median) after {warm} warm-up, "
                      f"float64 numpy, 1 thread; K/V generation and prefill summaries untimed",
            "times_s": [round(t, 4) for t in times]}


def run_reference(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    t0 = time.perf_counter()
    res = time_oracle(args.steps, args.warmup)
    wall = time.perf_counter() - t0
    line = {"impl": "reference", "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["value"] * LAYERS / 1000, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config({"layers_per_step": 1, "graph": None,
                                                    "note": "oracle timed on one layer; value per layer"}),
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


def algorithmic_bytes(wl, sel_lists, prev_lists):
    d, G = wl.d, wl.G
    out = {"score": 0, "attn": 0, "select": 0, "setdiff": 0, "summary_update": 0}
    for u in range(wl.U):
        T = wl.T(0, u // wl.Hkv)
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
# Block swap from host memory (the offload path): bandwidth of a full cache refill
# ---------------------------------------------------------------------------
def measure_block_swap(layer, wl, B, torch, reps: int = 20) -> dict:
    """Time bs_block_swap filling an empty GPU block cache with one layer's whole
    selection from pinned host memory (every selected page, K and V, crosses the host
    link once per call), alternating with a call that empties it."""
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
    del hk, hv
    return {"workload": "one layer's whole selection (every unit) copied into an empty GPU block cache",
            "bytes_per_call": nbytes, "us_per_call": round(us, 3), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "source": "pinned host memory read by the kernel over the host link (unified addressing)"}


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
    threads = os.cpu_count() or 1
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
    """Rebind every layer's q and its step outputs to views of two contiguous device
    buffers (regions 256-byte aligned); returns (q_all, o_all)."""
    q_all = torch.empty((len(layers),) + tuple(layers[0].q.shape), dtype=layers[0].q.dtype, device=dev)
    for i, layer in enumerate(layers):
        q_all[i].copy_(layer.q)
        layer.q = q_all[i]
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


def run_ours(args) -> None:
    import numpy as np
    import torch
    import torch.distributed as dist

    from long_context_serving_gb300 import bsattn as B
    from long_context_serving_gb300.build import build
    from long_context_serving_gb300.layer import PagedLayer
    from workloads import make_workload

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

    # Each rank serves its own batch (weak scaling): independent units, no exchange.
    wl = make_workload(CFG_ID, seed=rank)
    layers = []
    for _ in range(LAYERS):
        layer = PagedLayer(wl, device=dev, preload_all=True)
        layer._K = layer._V = None                      # logical copies are not needed any more
        layers.append(layer)
    torch.cuda.empty_cache()
    for layer in layers:
        layer.prefill()
    torch.cuda.synchronize()
    # Every layer's queries and outputs live in two contiguous device buffers, so the
    # end-to-end step moves its inputs and results with one copy each way.
    q_all, o_all = _pack_io(layers, torch, dev)

    def layer_calls(layer):
        if args.path == "fused":
            B.decode_step(layer.dims, layer.kv_at(layer.seq_lens[0]), layer.cfg, layer.step_io(0))
        else:
            layer.update_summaries(0)
            layer.score(0)
            layer.select(0)
            layer.attend(0)
            layer.setdiff()

    # Eager warm-up of both buffer parities (also the first selection / set-difference).
    for parity in (0, 1):
        for layer in layers:
            layer.cur = parity
            layer_calls(layer)
    torch.cuda.synchronize()
    assert all(layer.read_status() == 0 for layer in layers), "device status set during warm-up"

    graphs = []
    cap = torch.cuda.Stream(device=dev)
    for parity in (0, 1):
        g = torch.cuda.CUDAGraph()
        for layer in layers:
            layer.cur = parity
        with torch.cuda.graph(g, stream=cap):
            for layer in layers:
                layer_calls(layer)
        graphs.append(g)
    launches_per_step = (2 if args.path == "fused" else 5) * LAYERS

    def timed_replays(graph_list, n):
        stream = torch.cuda.current_stream()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(n):
            graph_list[i % len(graph_list)].replay()
        end.record(stream)
        torch.cuda.synchronize()
        barrier()
        return start.elapsed_time(end)

    # Clock samples cover warm-up, the timed region and, when the timed region is
    # shorter than a second, a soak of further replays so that the sampler sees load.
    sampler = ClockSampler(local, f"{args.clocks_csv}.rank{rank}" if args.clocks_csv else None)
    for i in range(args.warmup):
        graphs[i % 2].replay()
    ms = timed_replays(graphs, args.steps)
    ms = max_over_ranks(ms, dev)
    soak_s = 0.0
    while soak_s < 1.0 - ms / 1000:
        t0 = time.perf_counter()
        for i in range(200):
            graphs[i % 2].replay()
        torch.cuda.synchronize()
        soak_s += time.perf_counter() - t0
    clocks = sampler.stop()
    ms_per_step = ms / args.steps
    value = ms_per_step * 1000.0 / LAYERS
    assert all(layer.read_status() == 0 for layer in layers), "device status set during the timed region"

    # Per-kernel launch time (graphs of one call type over the 32 layers).
    def kernel_graph(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for layer in layers:
                fn(layer)
        return g

    for layer in layers:
        layer.cur = 0
    per_kernel = {}
    for name, fn in (("attn", lambda l: l.attend(0)), ("score", lambda l: l.score(0)),
                     ("select", lambda l: l.select(0)), ("summary_update", lambda l: l.update_summaries(0)),
                     ("setdiff", lambda l: l.setdiff())):
        g = kernel_graph(fn)
        for _ in range(3):
            g.replay()
        reps = max(20, args.steps)
        per_kernel[name] = timed_replays([g], reps) * 1000.0 / (reps * LAYERS)    # us per launch

    sel_now = layers[0].selection(0)
    prev_now = layers[0].selection(1)
    nbytes = algorithmic_bytes(wl, sel_now, prev_now)
    dominant = max(("attn", "score"), key=lambda k: per_kernel[k])
    peak, peak_note = _peak_hbm()
    achieved = nbytes[dominant] / (per_kernel[dominant] * 1e-6) / 1e9
    attn_kernel = "attn_mma_kernel" if wl.dtype == "bf16" else "attn_ffma_kernel"
    kernel_name = {"attn": attn_kernel, "score": "score_kernel"}[dominant]
    traffic = _measured_traffic(kernel_name, wl.name)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": kernel_name,
                "peak_source": peak_note, "algorithmic_bytes_per_launch": nbytes[dominant],
                "launch_us": round(per_kernel[dominant], 3),
                "timed_as": "graph of this call over the 32 layers, us per launch"}

    # End to end: every step copies the queries of all layers from pinned host memory
    # (one copy), replays, and reads back out, lse and the set-difference lists of all
    # layers into pinned host memory (one copy).
    q_host = torch.empty_like(q_all, device="cpu").pin_memory()
    q_host.copy_(q_all.cpu())
    o_host = torch.empty_like(o_all, device="cpu").pin_memory()
    h2d = q_host.numel() * q_host.element_size()
    d2h = o_host.numel() * o_host.element_size()

    def e2e_step(i):
        q_all.copy_(q_host, non_blocking=True)
        graphs[i % 2].replay()
        o_host.copy_(o_all, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for i in range(args.warmup):
        e2e_step(i)
    barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, dev)
    e2e_value = e2e_s / args.steps * 1e6 / LAYERS

    swap = measure_block_swap(layers[0], wl, B, torch) if rank == 0 else None
    split = measure_cpu_split(layers[0], wl, B, torch) if rank == 0 else None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = time_oracle(reps=args.cpu_reps, warm=1)
        cpu.pop("times_s", None)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": _config({"ranks": world, "parallelism": f"replicas x{world}, units independent",
                                   "path": args.path,
                                   "graph": f"CUDA graph of {LAYERS} layers x {launches_per_step // LAYERS} launches"}),
                "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h},
                "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
                "kernels_us_per_launch": {k: round(v, 3) for k, v in per_kernel.items()},
                "block_swap": swap,
                "cpu_gpu_split": split,
                "algorithmic_bytes_per_layer": nbytes,
                "layer_step_gbs": round(nbytes["layer_step"] / (value * 1e-6) / 1e9, 1),
                "layer_step_frac": round(nbytes["layer_step"] / (value * 1e-6) / 1e9 / peak, 4)}
        print(json.dumps(line, default=_json_default), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-reps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", choices=["fused", "calls"], default="fused",
                    help="fused: bs_decode_step per layer; calls: the five separate calls per layer")
    ap.add_argument("--clocks-csv", default=None,
                    help="also keep the raw nvidia-smi clock samples in this file (one per rank)")
    ap.add_argument("--layers", type=int, default=None,
                    help="layer buffers per step (fewer only for profiling small cases)")
    ap.add_argument("--config", type=int, choices=sorted(WORKLOADS), default=CFG_ID,
                    help="workload (2, the default, is the headline one)")
    args = ap.parse_args()
    globals()["CFG_ID"] = args.config
    globals()["WORKLOAD"], default_layers = WORKLOADS[args.config]
    globals()["LAYERS"] = args.layers if args.layers else default_layers
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
