#!/usr/bin/env python
"""Benchmark of the L³ layer on B300: one JSON line on stdout (rank 0).

Workload (default): the large bf16 prefill batch — vocab 128256, v 4194304 table rows
(a 17 GB key table and a 4 GB value table), d 2048, d_v 512, T 65536 tokens (16 x 4096)
with Zipf(1.1) ids, rows per id from the Zipf^0.7 rule capped at k = 512. A step is one
l3_forward over the batch (route, gather-attend, GEMM-up + LayerNorm statistics,
GEMM-mix), replayed as one CUDA graph captured from l3_forward; inputs are resident in
HBM and L2 is flushed (a 256 MB write, then a 256 MB read) before every timed step,
outside its events. `e2e` times the same forward through l3_forward_host from pinned host
buffers, copies included. Beside the headline the line carries, measured the same way,
the decode batch (`decode`: vocab 128256, v 1048576, d 2048, d_v 512, T 64) and the
prefill batch (`prefill`: vocab 32768, v 262144, d 1024, d_v 256, T 8192), and a forward
+ backward rate (`fwd_bwd`).

Multi-GPU (torchrun): every rank runs an independent batch (its own token seed) on its
own GPU with no collective on the data path; the timed region is bracketed by barriers,
the time is the max over ranks, and value = all ranks' tokens / that time (weak scaling).

`--impl reference` times the CPU fp64 oracle on bounded samples of the same workload
(rank 0 only), the reference arm for this library.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import l3_workloads as W  # noqa: E402

METRIC = "L^3 layer tokens/sec (fwd, fwd+bwd) on 1 B300; HBM GB/s vs ~8 TB/s roofline"
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0}


# ---- host-side workload accounting ---------------------------------------------------------------

def workload_bytes(p, ids: np.ndarray, offs: np.ndarray) -> dict:
    """Algorithmic bytes and FLOPs of one forward over the batch (per kernel stage).

    A distinct id's table rows are read once, each token's x row once and its a row
    written once. Ids held by at least ``long_th`` tokens of the batch go to the
    tensor-core kernel ("attend_long"), the rest to the split-row kernel ("attend");
    ``long_th`` is 8 for bf16 batches of at least 1024 tokens and 0 (no split) otherwise,
    the same rule the library applies.
    """
    b = 2 if p.dtype == "bf16" else 4
    T = len(ids)
    long_th = 8 if (p.dtype == "bf16" and T >= 1024 and p.d % 64 == 0
                    and p.d_v % 128 == 0 and p.d_v <= 512) else 0
    uniq, cnt = np.unique(ids, return_counts=True)
    n = np.diff(offs.astype(np.int64))
    is_long = cnt >= long_th if long_th > 0 else np.zeros(len(uniq), bool)

    def part(mask):
        rows = int(n[uniq[mask]].sum())
        tok = int(cnt[mask].sum())
        return rows * (p.d + p.d_v) * b + tok * (p.d + p.d_v) * b

    uniq_rows = int(n[uniq].sum())
    logical = int(n[ids].sum()) * (p.d + p.d_v) * b + 2 * T * p.d * b
    return {
        "unique_rows": uniq_rows,
        "distinct_ids": int(len(uniq)),
        "long_threshold": long_th,
        "long_ids": int(is_long.sum()),
        "attend_bytes": part(np.ones(len(uniq), bool)),
        "attend_short_bytes": part(~is_long),
        "attend_long_bytes": part(is_long),
        "route_bytes": T * 4 * 3 + 2 * len(uniq) * 8,
        "logical_bytes": logical,
        "up_flops": 2 * T * p.d * p.d_v,
        "mix_flops": 4 * T * p.d * p.d,
    }


# fp32 FMA throughput of the part: 148 SMs x 128 lanes x 2 FLOP per FMA x 2.032 GHz (TFLOP/s)
FP32_FMA_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of a stage's main
# kernel, from one ncu capture of the current kernel code on that workload (cold cache);
# an entry is removed when its kernel changes, and the roofline then reports null.
NCU_TRAFFIC = {
    ("prefill-bf16", "attend"): 206.20e6 + 1.13e6,     # attend_mma_kernel<16,8,2>
    ("prefill-bf16", "attend_long"): 98.56e6 + 0.26e6,  # attend_tc_kernel
    ("prefill-bf16", "mix"): 38.34e6 + 0.01e6,         # tc_gemm_kernel<256,2,4,0,0,0>
    ("prefill-bf16", "up"): 6.87e6,                    # tc_gemm_kernel<256,1,4,0,0,0>
    ("decode-bf16", "attend"): 85.23e6 + 0.12e6,       # attend_mma_kernel<8,16,4>
}
# Captures too large for ncu's replay at full size, taken on a reduced batch of the same
# shapes: (DRAM bytes of the launch, algorithmic bytes of the launch on that batch, the
# batch). The full-size traffic is the captured bytes scaled by the ratio of algorithmic
# bytes (the rows read grow with the distinct ids the batch touches).
NCU_TRAFFIC_SCALED = {
    ("large-prefill-bf16", "attend"): (1167.82e6 + 6.12e6, 1109.75488e6,
                                       "table rows 1048576, T 16384"),
}


def max_over_ranks(ms: float, device) -> float:
    """The largest of the ranks' times (the job is as slow as its slowest rank)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, T: int, steps: int, total_ms: float) -> float:
    """Whole-job tokens/s: every rank processes its own T-token batch per step (weak scaling)."""
    return world * T * steps / (total_ms / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


class L2Flush:
    """Empties L2 before a timed step: writes a 256 MB buffer (twice L2), then reads
    another 256 MB one, so the dirty lines of the write are written back to HBM here and
    not while the timed step runs."""

    def __init__(self, dev):
        import torch

        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


# ---- clocks --------------------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples (every 50 ms) for the whole run; ``window(t0, t1)`` summarises
    the samples taken while a timed region ran."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="l3clk", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        deadline = time.time() + 5.0
        while time.time() < deadline and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def _rows(self):
        import datetime

        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [s.strip() for s in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except ValueError:
                    continue
        return rows

    def window(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)  # the sample after the region's end
        rows = self._rows()
        win = [r for r in rows if t0 - 0.1 <= r[0] <= t1 + 0.1]
        if not win and rows:  # timed region shorter than the sampling interval: nearest sample
            mid = 0.5 * (t0 + t1)
            win = [min(rows, key=lambda r: abs(r[0] - mid))]
        reasons = sorted({nm for r in win for nm, val in zip(self.REASONS, r[3])
                          if val.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in win) if win else None,
                "sm_max_mhz": max(r[2] for r in win) if win else None, "reasons": reasons,
                "samples": len(win)}

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        os.unlink(self.path)


# ---- the CPU oracle as a baseline ------------------------------------------------------------------

class _Rows:
    """Host copy of the table rows of a set of ids, sliced like the full table."""

    def __init__(self, table, offs, ids):
        ranges = sorted({(int(offs[t]), int(offs[t + 1])) for t in set(int(i) for i in ids)})
        rows = np.concatenate([np.arange(a, c) for a, c in ranges])
        self.host = W.table_rows_to_numpy(table, rows)
        self.pos, k = {}, 0
        for a, c in ranges:
            self.pos[(a, c)] = k
            k += c - a

    def __getitem__(self, sl):
        k = self.pos[(sl.start, sl.stop)]
        return self.host[k:k + sl.stop - sl.start]


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def time_oracle(wl, offs_np, K, V, tokens) -> float:
    """Seconds the oracle takes for the given tokens (tables rows copied to host first)."""
    import oracle

    Kh = _Rows(K, offs_np, wl.ids[tokens])
    Vh = _Rows(V, offs_np, wl.ids[tokens])
    t0 = time.perf_counter()
    oracle.forward(offs_np, Kh, Vh, wl.W_up, wl.W_mix, wl.ids, wl.x, tokens=tokens)
    return time.perf_counter() - t0


def cpu_baseline(wl, offs_np, K, V, budget_s: float = 15.0) -> dict:
    probe = list(range(min(16, wl.T)))
    dt = time_oracle(wl, offs_np, K, V, probe)
    S = int(min(wl.T, max(len(probe), budget_s * len(probe) / max(dt, 1e-6))))
    toks = list(range(S))
    sec = time_oracle(wl, offs_np, K, V, toks)
    return {"value": S / sec, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"first {S} of {wl.T} tokens of the batch, fp64 numpy, one token at a time "
                      f"({sec:.1f} s)"}


# ---- runs -----------------------------------------------------------------------------------------

def config_block(p, T, extra=None):
    c = {"workload": f"{p.name}: vocab {p.vocab}, v {p.v}, d {p.d}, d_v {p.d_v}, T {T}, "
                     f"k {p.k_max}, Zipf(1.1) ids, rows per id from freq^{p.power}",
         "vocab": p.vocab, "v": p.v, "d": p.d, "d_v": p.d_v, "T": T, "k_max": p.k_max,
         "l2": "flushed before every timed step (256 MB write, then 256 MB read, outside the timed events)"}
    if extra:
        c.update(extra)
    return c


def run_reference(args, rank):
    if rank != 0:
        return 0
    import torch

    p = W.PRESETS[args.config]
    wl = W.make(args.config)
    import oracle

    offs_np = oracle.allocate(wl.freq, p.v, 1, p.k_max, p.power).offs
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    K, V = W.tables(wl, dev)
    # a bounded sample per step: the whole run stays near 4096 oracle tokens (tens of s)
    per_step = max(1, min(args.ref_tokens, 4096 // max(1, args.steps)))
    for w in range(args.warmup):
        time_oracle(wl, offs_np, K, V, [w % wl.T])
    total, toks = 0.0, 0
    for k in range(args.steps):
        sel = [(k * per_step + j) % wl.T for j in range(per_step)]
        total += time_oracle(wl, offs_np, K, V, sel)
        toks += per_step
    value = toks / total
    cores = blas_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(p, wl.T, {"sample_tokens_per_step": per_step}),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle",
                             "sample": f"{per_step} tokens per step of the {wl.T}-token batch"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


class Layer:
    """Device inputs of one preset (tables, weights, batch) and its forward workspace."""

    def __init__(self, l3, cid, args, dev, shard=0, v=None, vocab=None, T=None):
        import torch

        self.wl = wl = W.make(cid, T=T, shard=shard, v=v, vocab=vocab)
        self.p = p = wl.p
        self.T = wl.T
        self.offs_np = l3.l3_alloc_offsets(wl.freq, p.v, 1, p.k_max, p.power)
        self.dt = dt = W.torch_dtype(p)
        self.K, self.V = W.tables(wl, dev)
        self.offs = torch.as_tensor(self.offs_np, device=dev)
        self.W_up = torch.as_tensor(wl.W_up, device=dev).to(dt)
        self.W_mix = torch.as_tensor(wl.W_mix, device=dev).to(dt)
        self.ids = torch.as_tensor(wl.ids, device=dev)
        self.x = torch.as_tensor(wl.x, device=dev).to(dt)
        self.y = torch.empty((self.T, p.d), dtype=dt, device=dev)
        self.L = l3.make_layer(self.offs, self.K, self.V, self.W_up, self.W_mix, p.k_max)
        self.ws = torch.empty(l3.l3_workspace_size(self.L, self.T, l3.L3_PASS_FORWARD),
                              dtype=torch.uint8, device=dev)
        l3.l3_check_layer(self.L, self.ws)


def graph_forward(l3, lay, args, flush, clk, world, window):
    """Times ``args.steps`` replays of a CUDA graph of l3_forward (L2 flushed before each,
    outside the events), then replays a second graph with events between the stages.

    Returns (per-step ms list, per-stage mean ms list, launches per step, clock summary).
    """
    import torch
    import torch.distributed as dist

    nst = l3.L3_FWD_STAGES

    def new_events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)]
        for e in evs:
            e.record()
        return evs

    # Warm-up (eager): first calls set up kernel attributes and tensor-map entry points.
    warm = new_events()
    for _ in range(args.warmup):
        flush()
        l3.l3_forward_timed(lay.L, lay.ids, lay.x, lay.y, lay.ws, warm)
    torch.cuda.synchronize()
    if l3.l3_get_error(lay.ws) != 0:
        raise RuntimeError("device-side error during warm-up")
    # The timed step is one replay of a CUDA graph that holds the whole forward, so host-side
    # enqueue gaps are not timed. The per-stage breakdown comes from a second graph with
    # event-record nodes between the stages, replayed after the timed steps: the events
    # would keep each kernel from being set up while the previous one drains.
    stage_ev = new_events()
    cap = torch.cuda.Stream()

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
            fn()
        torch.cuda.synchronize()
        return g

    n_cap0 = l3.l3_launch_count()
    graph = capture(lambda: l3.l3_forward(lay.L, lay.ids, lay.x, lay.y, lay.ws))
    launches_per_step = l3.l3_launch_count() - n_cap0
    graph_st = capture(lambda: l3.l3_forward_timed(lay.L, lay.ids, lay.x, lay.y, lay.ws, stage_ev))
    for g in (graph, graph_st):
        g.replay()
    torch.cuda.synchronize()
    if l3.l3_get_error(lay.ws) != 0:
        raise RuntimeError("device-side error in the captured forward")
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    t0 = time.time()
    for k in range(args.steps):
        flush()
        step_ev[k][0].record()
        graph.replay()
        step_ev[k][1].record()
    barrier()
    t1 = time.time()
    stage_samples = []
    for k in range(args.steps):
        flush()
        graph_st.replay()
        torch.cuda.synchronize()
        stage_samples.append([stage_ev[s].elapsed_time(stage_ev[s + 1]) for s in range(nst)])
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    stage_ms = [statistics.mean(smp[s] for smp in stage_samples) for s in range(nst)]
    if l3.l3_get_error(lay.ws) != 0:
        raise RuntimeError("device-side error in the timed steps")
    return step_ms, stage_ms, launches_per_step, clk.window(t0, t1) if window else None


def attend_summary(lay, stage_ms, names, peaks):
    acct = workload_bytes(lay.p, lay.wl.ids, lay.offs_np)
    att_ms = stage_ms[names.index("attend")]
    long_ms = stage_ms[names.index("attend_long")]
    attend_s = (att_ms + long_ms) / 1e3
    return acct, {
        "unique_gbs": acct["attend_bytes"] / attend_s / 1e9,
        "logical_gbs": acct["logical_bytes"] / attend_s / 1e9,
        "frac_of_8tbs": acct["attend_bytes"] / attend_s / 8e12,
        "frac_of_measured": acct["attend_bytes"] / attend_s / 1e9 / peaks["hbm_gbs"],
        "unique_rows": acct["unique_rows"], "distinct_ids": acct["distinct_ids"],
        "long_threshold": acct["long_threshold"], "long_ids": acct["long_ids"],
        "short_gbs": acct["attend_short_bytes"] / (att_ms / 1e3) / 1e9,
        "short_frac_of_measured": acct["attend_short_bytes"] / (att_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
        "long_gbs": (acct["attend_long_bytes"] / (long_ms / 1e3) / 1e9 if long_ms > 0 else None)}


def gemm_summary(acct, stage_ms, names, peaks):
    out = {}
    for st, key in (("up", "up_flops"), ("mix", "mix_flops")):
        ms = stage_ms[names.index(st)]
        tf = acct[key] / (ms / 1e3) / 1e12
        out[st] = {"tflops": tf, "frac_of_measured": tf / peaks["bf16_tflops"]}
    return out


def sub_workload(l3, cid, args, dev, flush, clk, peaks) -> dict:
    """A second workload measured beside the headline (same protocol, own clock window)."""
    import torch

    lay = Layer(l3, cid, args, dev)
    step_ms, stage_ms, launches, clocks = graph_forward(l3, lay, args, flush, clk, 1, True)
    names = l3.STAGE_NAMES
    ms = statistics.mean(step_ms)
    acct, att = attend_summary(lay, stage_ms, names, peaks)
    p = lay.p
    esz = 2 if p.dtype == "bf16" else 4
    weights = (p.d * p.d_v + 2 * p.d * p.d) * esz
    step_bytes = acct["attend_bytes"] + lay.T * p.d * esz + weights  # + U/x re-reads not counted
    out = {"workload": config_block(p, lay.T)["workload"],
           "value": lay.T / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
           "stage_ms": dict(zip(names, stage_ms)), "attend_hbm": att,
           "gemm": gemm_summary(acct, stage_ms, names, peaks),
           "step_unique_bytes": step_bytes,
           "step_frac_of_measured_hbm": step_bytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
           "gpu_launches_per_step": launches, "clocks": clocks}
    del lay
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local_rank):
    import torch

    import static_token_routed_csr_b300 as l3

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lay = Layer(l3, args.config, args, dev, shard=rank, v=args.rows, vocab=args.vocab,
                T=args.tokens)
    p, T = lay.p, lay.T
    flush = L2Flush(dev)
    clk = ClockSampler(local_rank)
    clk.start()
    step_ms, stage_ms, launches_per_step, clocks = graph_forward(l3, lay, args, flush, clk,
                                                                 world, True)
    launches = launches_per_step * args.steps
    total_ms = max_over_ranks(sum(step_ms), dev)
    value = job_rate(world, T, args.steps, total_ms)
    names = l3.STAGE_NAMES
    peaks = load_peaks()

    if args.profile_bwd:
        # profiler captures of the backward: a few forward + row-gradient backward steps
        acct = workload_bytes(p, lay.wl.ids, lay.offs_np)
        args.bwd_steps, args.warmup = 3, 1
        fb = fwd_bwd_rows_rate(l3, lay, args, flush, acct, world)
        clk.stop()
        if rank == 0:
            print(json.dumps({"metric": METRIC, "fwd_bwd": fb, "config": config_block(p, T),
                              "note": "forward + backward (profiling run)"}), flush=True)
        return 0
    if args.fwd_only:
        clk.stop()
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": "tokens/s",
                              "config": config_block(p, T),
                              "stage_ms": dict(zip(names, stage_ms)),
                              "note": "forward only (profiling run)"}), flush=True)
        return 0
    # end to end through the host-buffer entry point
    import torch.distributed as dist

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    ws_h = torch.empty(l3.l3_workspace_size(lay.L, T, l3.L3_PASS_FORWARD_HOST), dtype=torch.uint8,
                       device=dev)
    ids_h = lay.ids.cpu().pin_memory()
    x_h = lay.x.cpu().pin_memory()
    y_h = torch.empty((T, p.d), dtype=lay.dt).pin_memory()
    for _ in range(max(1, args.warmup)):
        l3.l3_forward_host(lay.L, ids_h, x_h, y_h, ws_h)
    torch.cuda.synchronize()
    e2e_steps = min(args.steps, args.e2e_steps)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(e2e_steps)]
    barrier()
    for k in range(e2e_steps):
        flush()
        e2e_ev[k][0].record()
        l3.l3_forward_host(lay.L, ids_h, x_h, y_h, ws_h)
        e2e_ev[k][1].record()
    barrier()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev), dev)
    if not torch.equal(y_h.to(dev), lay.y):
        raise RuntimeError("host-buffer forward disagrees with the device forward")
    del ws_h
    esz = 2 if p.dtype == "bf16" else 4

    acct, att = attend_summary(lay, stage_ms, names, peaks)
    fb_rows = None
    if p.dtype == "bf16" and not args.no_bwd:
        fb_rows = fwd_bwd_rows_rate(l3, lay, args, flush, acct, world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(lay.wl, lay.offs_np, lay.K, lay.V)
    del lay
    torch.cuda.empty_cache()

    # beside the headline: forward + backward, the decode batch and the prefill batch
    fb = fwd_bwd_rate(l3, dev, args)
    subs = {}
    if not args.no_sub:
        for key, cid in (("decode", 3), ("prefill", 2)):
            if cid != args.config:
                subs[key] = sub_workload(l3, cid, args, dev, flush, clk, peaks)
        subs["offload"] = offload_leg(l3, 3, args, dev, flush, peaks)
    clk.stop()
    if rank != 0:
        return 0
    dom = int(np.argmax(stage_ms))
    dom_s = stage_ms[dom] / 1e3
    hbm_bytes = {"route": acct["route_bytes"], "attend": acct["attend_short_bytes"],
                 "attend_long": acct["attend_long_bytes"]}
    if names[dom] in hbm_bytes:
        achieved = hbm_bytes[names[dom]] / dom_s / 1e9
        kern = {"route": "route", "attend": "gather-attend (split-row)",
                "attend_long": "gather-attend (tensor-core)"}[names[dom]]
        roof = {"kernel": kern, "bound": "hbm", "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": None, "bytes_per_launch": hbm_bytes[names[dom]]}
    else:
        flops = acct["up_flops"] if names[dom] == "up" else acct["mix_flops"]
        achieved = flops / dom_s / 1e12
        if p.dtype == "bf16":
            roof = {"kernel": "gemm-" + names[dom], "bound": "tensor", "achieved": achieved,
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": achieved / peaks["bf16_tflops"], "traffic": None}
        else:  # fp32 layers: CUDA-core GEMMs against the fp32 FMA rate
            roof = {"kernel": "gemm-" + names[dom] + " (fp32 CUDA cores)", "bound": "alu",
                    "achieved": achieved, "peak": FP32_FMA_TFLOPS, "unit": "TFLOP/s",
                    "frac": achieved / FP32_FMA_TFLOPS, "traffic": None}
    full_size = args.rows is None and args.tokens is None and args.vocab is None
    roof["traffic"] = NCU_TRAFFIC.get((p.name, names[dom])) if full_size else None
    sc = NCU_TRAFFIC_SCALED.get((p.name, names[dom]))
    if full_size and sc is not None and roof.get("bytes_per_launch"):
        roof["traffic"] = sc[0] * roof["bytes_per_launch"] / sc[1]
        roof["traffic_note"] = ("scaled from an ncu capture on a reduced batch (" + sc[2] +
                                ") by the ratio of algorithmic bytes")
    roof["peak_source"] = peaks["source"] if roof["bound"] != "alu" else (
        "derived: 148 SMs x 128 fp32 lanes x 2 FLOP x 2.032 GHz")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": p.dtype,
        "data": "synthetic (seeded Zipf ids, N(0,1) x, N(0,0.02^2) tables, N(0,1/fan_in) weights)",
        "config": config_block(p, T),
        "stage_ms": dict(zip(names, stage_ms)),
        "attend_hbm": att,
        "gemm": gemm_summary(acct, stage_ms, names, peaks) if p.dtype == "bf16" else None,
        "roofline": roof,
        "e2e": {"value": job_rate(world, T, e2e_steps, e2e_ms), "unit": "tokens/s",
                "steps": e2e_steps,
                "h2d_bytes_per_step": T * 4 + T * p.d * esz, "d2h_bytes_per_step": T * p.d * esz},
        "fwd_bwd": fb_rows if fb_rows is not None else fb,
        "fwd_bwd_small": fb,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    line.update(subs)
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    return 0


def fwd_bwd_rows_rate(l3, lay, args, flush, acct, world) -> dict:
    """Forward (keeping the saved state) + row-gradient backward over the headline batch,
    one CUDA graph per step, L2 flushed before each step (outside the events)."""
    import torch

    p, T, dev = lay.p, lay.T, lay.x.device
    g = torch.Generator(device=dev)
    g.manual_seed(7000 + p.cid)
    dy = torch.randn((T, p.d), generator=g, device=dev).to(torch.bfloat16)
    rows = acct["unique_rows"]
    sv = torch.empty(l3.l3_saved_size(lay.L, T), dtype=torch.uint8, device=dev)
    wsb = torch.empty(l3.l3_workspace_size(lay.L, T, l3.L3_PASS_BACKWARD_ROWS), dtype=torch.uint8,
                      device=dev)
    dx = torch.empty((T, p.d), device=dev)
    row_index = torch.empty(rows, dtype=torch.int32, device=dev)
    dK = torch.empty((rows, p.d), device=dev)
    dV = torch.empty((rows, p.d_v), device=dev)
    n_rows = torch.zeros(1, dtype=torch.int32, device=dev)
    dWu = torch.empty((p.d, p.d_v), device=dev)
    dWm = torch.empty((p.d, 2 * p.d), device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def step(timed):
        if timed:
            ev[0].record()
        l3.l3_forward(lay.L, lay.ids, lay.x, lay.y, lay.ws, saved=sv)
        if timed:
            ev[1].record()
        l3.l3_backward_rows(lay.L, lay.ids, lay.x, dy, sv, dx, row_index, dK, dV, n_rows, dWu, dWm,
                            wsb)
        if timed:
            ev[2].record()

    for _ in range(args.warmup):
        flush()
        step(False)
    torch.cuda.synchronize()
    if l3.l3_get_error(wsb) != 0 or int(n_rows.item()) != rows:
        raise RuntimeError("row-gradient backward reported an error")
    cap = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=cap, capture_error_mode="thread_local"):
        step(False)
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, args.bwd_steps))
    tot = 0.0
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(steps)]
    for k in range(steps):
        flush()
        pairs[k][0].record()
        graph.replay()
        pairs[k][1].record()
    torch.cuda.synchronize()
    tot = sum(a.elapsed_time(b) for a, b in pairs)
    total_ms = max_over_ranks(tot, dev)
    # the split between forward and backward, from one eager step with events
    flush()
    step(True)
    torch.cuda.synchronize()
    return {"workload": config_block(p, T)["workload"] + ", dy ~ N(0,1) bf16",
            "value": job_rate(world, T, steps, total_ms), "unit": "tokens/s",
            "ms_per_step": total_ms / steps, "steps": steps,
            "fwd_ms": ev[0].elapsed_time(ev[1]), "bwd_ms": ev[1].elapsed_time(ev[2]),
            "touched_rows": rows,
            "row_grad_bytes": rows * (p.d + p.d_v) * 4,
            "l2": "flushed before every timed step (outside the timed events)"}


def offload_leg(l3, cid, args, dev, flush, peaks) -> dict:
    """Tables in pinned host memory: per step the batch's rows are staged into device memory
    (l3_stage_rows) and the forward runs over the staged layer. Reported serially (stage, then
    forward) and pipelined (the next batch's rows staged on a second stream while the current
    forward runs, double-buffered staging), the way a model would prefetch during earlier
    layers."""
    import torch

    lay = Layer(l3, cid, args, dev)
    p, T = lay.p, lay.T
    K_h, V_h = lay.K.cpu().pin_memory(), lay.V.cpu().pin_memory()
    del lay.K, lay.V
    torch.cuda.empty_cache()
    L_h = l3.make_layer(lay.offs, K_h, V_h, lay.W_up, lay.W_mix, p.k_max)
    acct = workload_bytes(p, lay.wl.ids, lay.offs_np)
    U = acct["unique_rows"]
    cap = U + T
    bufs = []
    for _ in range(2):
        K_s = torch.empty((cap, p.d), dtype=lay.dt, device=dev)
        V_s = torch.empty((cap, p.d_v), dtype=lay.dt, device=dev)
        offs_s = torch.empty(T + 1, dtype=torch.int32, device=dev)
        ids_s = torch.empty(T, dtype=torch.int32, device=dev)
        n_rows = torch.zeros(1, dtype=torch.int32, device=dev)
        ws_s = torch.empty(l3.l3_workspace_size(L_h, T, l3.L3_PASS_STAGE), dtype=torch.uint8,
                           device=dev)
        y = torch.empty((T, p.d), dtype=lay.dt, device=dev)
        bufs.append(dict(K=K_s, V=V_s, offs=offs_s, ids=ids_s, n=n_rows, ws=ws_s, y=y))
    s_main = torch.cuda.current_stream()
    s_copy = torch.cuda.Stream()

    def stage(b, stream):
        with torch.cuda.stream(stream):
            b["L"] = l3.l3_stage_rows(L_h, lay.ids, b["K"], b["V"], b["offs"], b["ids"], b["n"],
                                      b["ws"], stream=stream)

    def fwd(b):
        wsf = b.setdefault("wsf", torch.empty(l3.l3_workspace_size(b["L"], T, l3.L3_PASS_FORWARD),
                                              dtype=torch.uint8, device=dev))
        l3.l3_forward(b["L"], b["ids"], lay.x, b["y"], wsf)

    for k in range(max(2, args.warmup)):
        stage(bufs[k % 2], s_main)
        fwd(bufs[k % 2])
    torch.cuda.synchronize()
    if l3.l3_get_error(bufs[0]["ws"]) != 0 or int(bufs[0]["n"].item()) != U:
        raise RuntimeError("staging reported an error")
    steps = max(3, min(args.steps, 50))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    st_ms, fw_ms = [], []
    for _ in range(steps):
        flush()
        ev[0].record()
        stage(bufs[0], s_main)
        ev[1].record()
        fwd(bufs[0])
        ev[2].record()
        torch.cuda.synchronize()
        st_ms.append(ev[0].elapsed_time(ev[1]))
        fw_ms.append(ev[1].elapsed_time(ev[2]))
    # pipelined: stage batch k + 1 on the copy stream while batch k's forward runs
    done = [torch.cuda.Event() for _ in range(2)]
    staged = [torch.cuda.Event() for _ in range(2)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stage(bufs[0], s_copy)
    staged[0].record(s_copy)
    torch.cuda.synchronize()
    a.record()
    for k in range(steps):
        cur, nxt = bufs[k % 2], bufs[(k + 1) % 2]
        s_copy.wait_event(done[(k + 1) % 2]) if k > 0 else None
        stage(nxt, s_copy)
        staged[(k + 1) % 2].record(s_copy)
        s_main.wait_event(staged[k % 2])
        fwd(cur)
        done[k % 2].record(s_main)
    b.record()
    torch.cuda.synchronize()
    pipe_ms = a.elapsed_time(b) / steps
    staged_bytes = U * (p.d + p.d_v) * (2 if p.dtype == "bf16" else 4)
    st = statistics.median(st_ms)
    out = {"workload": config_block(p, T)["workload"] + ", tables in pinned host memory",
           "stage_ms": st, "forward_ms": statistics.median(fw_ms),
           "serial_ms_per_step": st + statistics.median(fw_ms),
           "pipelined_ms_per_step": pipe_ms, "value": T / (pipe_ms / 1e3), "unit": "tokens/s",
           "staged_bytes": staged_bytes, "host_link_gbs": staged_bytes / (st / 1e3) / 1e9,
           "l2": "serial steps flushed before each step; pipelined steps back to back"}
    del K_h, V_h, bufs, lay
    torch.cuda.empty_cache()
    return out


def fwd_bwd_rate(l3, dev, args) -> dict:
    import torch

    wl = W.make(5)
    p = wl.p
    offs_np = l3.l3_alloc_offsets(wl.freq, p.v, 1, p.k_max, p.power)
    K, V = W.tables(wl, dev)
    dt = torch.bfloat16
    offs = torch.as_tensor(offs_np, device=dev)
    Wu = torch.as_tensor(wl.W_up, device=dev).to(dt)
    Wm = torch.as_tensor(wl.W_mix, device=dev).to(dt)
    ids = torch.as_tensor(wl.ids, device=dev)
    x = torch.as_tensor(wl.x, device=dev).to(dt)
    dy = torch.as_tensor(wl.dy, device=dev).to(dt)
    L = l3.make_layer(offs, K, V, Wu, Wm, p.k_max)
    T = wl.T
    ws = torch.empty(l3.l3_workspace_size(L, T, 0), dtype=torch.uint8, device=dev)
    wsb = torch.empty(l3.l3_workspace_size(L, T, 1), dtype=torch.uint8, device=dev)
    sv = torch.empty(l3.l3_saved_size(L, T), dtype=torch.uint8, device=dev)
    y = torch.empty((T, p.d), dtype=dt, device=dev)
    g = [torch.empty(s, device=dev) for s in ((T, p.d), (p.v, p.d), (p.v, p.d_v), (p.d, p.d_v), (p.d, 2 * p.d))]

    def step():
        l3.l3_forward(L, ids, x, y, ws, saved=sv)
        l3.l3_backward(L, ids, x, dy, sv, *g, wsb)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        step()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    return {"workload": f"{p.name}: vocab {p.vocab}, v {p.v}, d {p.d}, d_v {p.d_v}, T {T}, k {p.k_max}",
            "value": T / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "l2": "not flushed (whole working set is under 2 MB)"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)  # ~0.2 s timed: clock samples fall inside
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", type=int, default=4, choices=sorted(W.PRESETS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fwd-only", action="store_true",
                    help="skip the e2e, fwd+bwd and side-workload legs (for profiler captures)")
    ap.add_argument("--no-sub", action="store_true",
                    help="skip the decode and prefill workloads measured beside the headline")
    ap.add_argument("--e2e-steps", type=int, default=50,
                    help="timed steps of the host-buffer (end-to-end) leg")
    ap.add_argument("--bwd-steps", type=int, default=20,
                    help="timed steps of the forward + row-gradient backward leg")
    ap.add_argument("--no-bwd", action="store_true", help="skip the forward + backward leg")
    ap.add_argument("--profile-bwd", action="store_true",
                    help="only a few forward + backward steps (for profiler captures)")
    ap.add_argument("--rows", type=int, default=None,
                    help="profiling: table rows v of a smaller table with the preset's shapes")
    ap.add_argument("--vocab", type=int, default=None, help="profiling: vocabulary size")
    ap.add_argument("--tokens", type=int, default=None, help="profiling: tokens T per batch")
    ap.add_argument("--ref-tokens", type=int, default=128,
                    help="tokens per reference-arm step")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed steps before timing
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank)
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
