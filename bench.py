#!/usr/bin/env python
"""Benchmark of paged GQA decode attention on GB300.

Workload (default): the ragged eight-request decode of lucebox PR #555
(Benchmark results, its ragged-workload table): sequence lengths 131072 and
7 x 8192 (188,416 live tokens), 16-token pages handed out round-robin as if the
requests arrived together, Q4_0 K/V from N(0,1) sources, D=256, 24 query heads
on 4 KV heads, one query token.  Synthetic, seeded inputs.

One step = one pa_decode (split-K pass + merge pass) over the whole batch,
replayed from a CUDA graph.  Metric: K/V GB/s = algorithmic K+V bytes read per
step (every live row of every KV head once) / step time, and us/step.  Between
timed steps L2 is flushed outside the timed region: a buffer of twice the L2
is written and then read back, so that neither the inputs nor dirty lines of
the flush are left in L2 when a step starts.  The same steps without the flush
("warm") are reported beside them.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun): the global batch is N copies of the workload's sequences,
partitioned across the ranks by sequence with the K/V bytes balanced
(partition.py), with no data-path communication (the (sequence, KV head)
segments are independent); the value is the bytes all ranks processed over the
slowest rank's time.  --impl reference times the float64 CPU oracle on the
host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attention K/V GB/s (fraction of GB300 HBM peak) and us/step"
FALLBACK_HBM_GBS = 6800.0
# RTX 3090, paged, same workload: 4.095 ms per step (lucebox PR #555, ragged
# table) = 217,055,232 B / 4.095 ms = 53.0 GB/s.  Another machine: context.
PAGES_PAGED_3090_MS = 4.095
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
DECODE_SOURCES = ["paged_kv_gqa_11_gb300/csrc/pa_decode.cu", "paged_kv_gqa_11_gb300/csrc/pa_decode_impl.cuh",
                  "paged_kv_gqa_11_gb300/csrc/pa_decode_kern.cu", "paged_kv_gqa_11_gb300/csrc/pa_device.cuh",
                  "paged_kv_gqa_11_gb300/csrc/pa_layout.cuh", "paged_kv_gqa_11_gb300/csrc/pa_rows_impl.cuh",
                  "paged_kv_gqa_11_gb300/csrc/pa_rows_tc.cuh"]


def workload_for(name: str) -> W.Workload:
    if name == "ragged":
        return W.config(3)
    if name == "ragged-contiguous":
        return W.config(3, variant="contiguous")
    if name == "uniform":
        return W.config(2)
    if name.startswith("verify"):
        return W.config(4, n_qtok=int(name[-1]) if name[-1].isdigit() else 4)
    if name == "long":
        return W.config(5, variant="a")
    if name == "many":
        return W.config(5, variant="b")
    if name == "shared-prefix":  # 8 sequences forked from a 32K-token prompt, 1K own rows each
        return W.shared_prefix()
    if name.startswith("rows-"):  # rows-<4k|16k|64k>-<17|65|96>: row tiles, Q8_0 K / Q4_0 V, one sequence
        _, size, nq = name.split("-")
        return W.rows_workload({"4k": 4096, "16k": 16384, "64k": 65536}[size], int(nq))
    if name.startswith("percall-"):  # percall-<32k|131k|262k>-<1|3|4>: Q8_0 K / Q4_0 V, one sequence
        _, size, nq = name.split("-")
        return W.percall({"32k": 32768, "131k": 131072, "262k": 262144}[size], int(nq))
    raise SystemExit(f"unknown workload {name}")


def describe(w: W.Workload) -> str:
    lens = w.seq_lens
    if len(set(lens.tolist())) == 1:
        shape = f"{len(lens)}x{int(lens[0])}"
    elif len(lens) <= 8:
        shape = "+".join(str(int(x)) for x in lens)
    else:
        shape = f"{len(lens)} seqs, sum {int(lens.sum())}, max {int(lens.max())}"
    kt = W.TYPE_NAMES[w.k_type]
    vt = W.TYPE_NAMES[w.v_type]
    return (f"{w.name}: paged GQA decode, lengths {shape}, page size {w.page_size}, K {kt} / V {vt}, "
            f"D=256, Hq=24, Hkv=4, {w.n_qtok} query token(s)")


def source_hash() -> str:
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profile_traffic(workload: str):
    """DRAM bytes per launch of the split kernel (dram__bytes_read.sum +
    dram__bytes_write.sum from one ncu capture), from profiles/traffic.json,
    if it was taken on this workload with the current kernel sources."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            entries = json.load(f)
    except (OSError, ValueError):
        return None
    for e in entries if isinstance(entries, list) else []:
        if e.get("workload") == workload and e.get("source") == source_hash():
            try:
                return int(e["dram_bytes_per_launch"])
            except (KeyError, TypeError, ValueError):
                return None
    return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples over the GPU phase of the run.

    The window opens before the warm-up and closes after the last GPU leg, so
    that a short run still holds samples under load; the samples inside the
    headline timed region are counted separately."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 10):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []
        self.t_begin = self.t_end = None
        self.timed = []  # (begin, end) of the headline timed regions

    @staticmethod
    def _now():
        from datetime import datetime
        return datetime.now()

    def begin(self):
        self.t_begin = self._now()

    def end(self):
        self.t_end = self._now()
        time.sleep(3 * self.period / 1000.0)

    def mark_timed(self, t0, t1):
        self.timed.append((t0, t1))

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)  # let the first samples arrive
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        from datetime import datetime
        sm, mx, reasons, in_timed = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in list(self.lines):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                continue
            if self.t_begin and ts < self.t_begin or self.t_end and ts > self.t_end:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            in_timed += any(a <= ts <= b for a, b in self.timed)
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_in_timed_region": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "sm_mhz_min": min(sm),
                "reasons": sorted(reasons), "samples": len(sm), "samples_in_timed_region": in_timed,
                "window": "warm-up to the last GPU leg, every 10 ms"}


def rank_max(dist, x: float, device) -> float:
    """The largest of one float over all ranks (the slowest rank's time)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(n_ranks: int, bytes_per_rank_step: int, slowest_step_ms: float) -> float:
    """Whole-job K/V GB/s: every rank decodes its own batch (weak scaling)."""
    return n_ranks * bytes_per_rank_step / (slowest_step_ms * 1e-3) / 1e9


def _select(w: W.Workload, pairs):
    sel = np.zeros((w.n_seq, W.HQ), bool)
    for s, g in pairs:
        sel[s, g * W.GQA:(g + 1) * W.GQA] = True
    return sel


def oracle_segments(w: W.Workload, cache, budget_s: float, threads: int):
    """A bounded sample of the workload for the float64 oracle: whole
    (sequence, KV head) segments, shortest first, added until one run of the
    sample is estimated to take about budget_s on `threads` host threads."""
    import oracle
    segs = sorted((int(w.seq_lens[s]), s, g) for s in range(w.n_seq) for g in range(W.HKV))
    L0, s0, g0 = segs[0]
    t0 = time.perf_counter()
    oracle.decode(cache, w.q, w.scale, _select(w, [(s0, g0)]), n_threads=threads)
    per_row = max(time.perf_counter() - t0, 1e-5) / L0
    chosen, est = [], 0.0
    for L, s, g in segs:
        if chosen and est + L * per_row > budget_s:
            break
        chosen.append((s, g))
        est += L * per_row
    return chosen


def oracle_time(w: W.Workload, cache, pairs, threads: int) -> float:
    import oracle
    t0 = time.perf_counter()
    oracle.decode(cache, w.q, w.scale, _select(w, pairs), n_threads=threads)
    return time.perf_counter() - t0


def sample_bytes(w: W.Workload, pairs) -> int:
    rb = W.row_bytes(w.k_type) + W.row_bytes(w.v_type)
    return sum(int(w.seq_lens[s]) for s, _ in pairs) * rb


def sample_desc(w: W.Workload, pairs) -> str:
    rows = sum(int(w.seq_lens[s]) for s, _ in pairs)
    return (f"{len(pairs)} of {w.n_seq * W.HKV} (sequence, KV head) segments, shortest first, "
            f"{rows} K/V rows, all {W.GQA * w.n_qtok} query rows of each")


def oracle_cache(w: W.Workload):
    import oracle
    oracle.build()
    return oracle.Cache.from_workload(w)


def run_reference(args, w: W.Workload):
    """The float64 oracle on the host cores, each step a bounded sample."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    threads = os.cpu_count() or 1
    cache = oracle_cache(w)
    per_step = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    pairs = oracle_segments(w, cache, per_step, threads)
    times = []
    for i in range(args.warmup + args.steps):
        dt = oracle_time(w, cache, pairs, threads)
        if i >= args.warmup:
            times.append(dt)
    step = statistics.mean(times)
    value = sample_bytes(w, pairs) / step / 1e9
    desc = sample_desc(w, pairs)
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(w), "sample": desc, "l2": "n/a (CPU)"},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_append(args, w: W.Workload):
    """Quantise-on-append throughput: every row of the workload, given as
    binary16, quantised into the workload's K/V formats and scattered through
    its table, per call; bytes = fp16 rows read + pool bytes written."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_gqa_11_gb300.cache import PagedKVCache
    dev = torch.device("cuda", 0)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    c = PagedKVCache(w.n_blocks, w.page_size, w.k_type, w.v_type, device=dev)
    n = int(w.row_seq.shape[0])
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    hk = torch.randn((n, W.HKV, W.D), generator=g, device=dev).half()
    hv = torch.randn((n, W.HKV, W.D), generator=g, device=dev).half()
    rs, rp, tab = t(w.row_seq), t(w.row_pos), t(w.table)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        c.append_f16(hk, hv, rs, rp, tab, stream=stream.cuda_stream)
    torch.cuda.synchronize()
    if c.check() != 0:
        raise SystemExit("append reported a device error")
    K = min(args.steps, 200)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush.fill_(1.0)
        ev[i][0].record(stream)
        c.append_f16(hk, hv, rs, rp, tab, stream=stream.cuda_stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    nbytes = n * W.HKV * (2 * W.D * 2 + W.row_bytes(w.k_type) + W.row_bytes(w.v_type))
    peaks = measured_peaks()
    peak = float(peaks["hbm_gbs"]) if peaks and "hbm_gbs" in peaks else FALLBACK_HBM_GBS
    gbps = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "quantise-on-append GB/s (binary16 rows read + pool bytes written)", "value": round(gbps, 2),
        "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "dtype": "f32", "data": "synthetic",
        "config": {"workload": describe(w) + f"; {n} rows appended per call", "bytes_per_step": nbytes},
        "roofline": {"bound": "hbm", "achieved": round(gbps, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(gbps / peak, 4), "traffic": None}}))


def percentiles(ms):
    a = np.sort(np.asarray(ms, dtype=np.float64))
    return {"mean_us": round(float(a.mean()) * 1e3, 2), "median_us": round(float(np.median(a)) * 1e3, 2),
            "p10_us": round(float(np.percentile(a, 10)) * 1e3, 2), "p90_us": round(float(np.percentile(a, 90)) * 1e3, 2)}


def rank_workload(w: W.Workload, world: int, rank: int) -> W.Workload:
    """This rank's share of a global batch of `world` copies of w's
    sequences, partitioned by sequence with the K/V bytes balanced."""
    from paged_kv_gqa_11_gb300 import partition
    n = w.n_seq
    lens = np.tile(w.seq_lens, world)
    parts = partition.balance_by_sequence(partition.kv_bytes_per_sequence(lens, w.k_type, w.v_type, W.HKV), world)
    return w.subset([i % n for i in parts[rank]])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ragged")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", choices=["decode", "append"], default="decode",
                    help="append: time quantise-on-append (pa_append_rows_f16) instead of decode")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    w = workload_for(args.workload)
    if args.impl == "reference":
        run_reference(args, w)
        return
    if args.mode == "append":
        run_append(args, w)
        return

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        w = rank_workload(w, world, rank)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_gqa_11_gb300 as pa
    from paged_kv_gqa_11_gb300.cache import PagedKVCache

    def barrier():
        if dist is not None:
            dist.barrier()

    clocks = ClockSampler(local).__enter__()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    cache = PagedKVCache(w.n_blocks, w.page_size, w.k_type, w.v_type, device=dev)
    table = t(w.table)
    cache.append(t(w.k_rows), t(w.v_rows), t(w.row_seq), t(w.row_pos), table)
    sl_dev = t(w.seq_lens)
    sl_host = np.ascontiguousarray(w.seq_lens, np.int32)
    ws = cache.workspace(w.n_seq, w.n_qtok)
    if cache.check() != pa.PA_OK:
        raise SystemExit("append reported a device error")
    kv_bytes = w.kv_bytes()
    plan = pa.pa_decode_plan(cache.pool, sl_host, w.n_qtok, local)
    # our kernels per step: one split kernel per sub-batch of up to 128
    # sequences, plus a merge kernel where a segment is split into pieces
    launches_per_step = 0
    for c0 in range(0, w.n_seq, 128):
        sub = sl_host[c0:c0 + 128]
        pl = pa.pa_decode_plan(cache.pool, sub, w.n_qtok, local)
        segs = len(sub) * (1 if w.n_qtok == 1 else W.HKV)
        launches_per_step += 1 + (pl["partials"] > segs)

    # Step inputs (query + one new K/V row per sequence + its index) packed in
    # one buffer, outputs (out + lse) in another: one H2D and one D2H per step
    # in the end-to-end leg.
    new_idx = np.array([int(w.seq_offsets[s + 1]) - 1 for s in range(w.n_seq)])  # last row of each sequence
    parts_in = [np.ascontiguousarray(w.q).view(np.uint8).ravel(),
                np.ascontiguousarray(w.k_rows[new_idx]).view(np.uint8).ravel(),
                np.ascontiguousarray(w.v_rows[new_idx]).view(np.uint8).ravel(),
                np.ascontiguousarray(w.row_seq[new_idx]).view(np.uint8).ravel(),
                np.ascontiguousarray(w.row_pos[new_idx]).view(np.uint8).ravel()]
    offs, o = [], 0
    for a in parts_in:
        offs.append(o)
        o += (a.nbytes + 255) // 256 * 256
    h_in = torch.zeros(o, dtype=torch.uint8).pin_memory()
    for a, off in zip(parts_in, offs):
        h_in[off:off + a.nbytes] = torch.from_numpy(a)
    d_in = h_in.to(dev)
    view = lambda buf, i, dtype, shape: buf[offs[i]:offs[i] + parts_in[i].nbytes].view(dtype).view(shape)
    q = view(d_in, 0, torch.float32, w.q.shape)
    d_k = view(d_in, 1, torch.uint8, (w.n_seq,) + w.k_rows.shape[1:])
    d_v = view(d_in, 2, torch.uint8, (w.n_seq,) + w.v_rows.shape[1:])
    d_seq = view(d_in, 3, torch.int32, (w.n_seq,))
    d_pos = view(d_in, 4, torch.int32, (w.n_seq,))
    n_out = w.n_seq * w.n_qtok * W.HQ * W.D
    d_outbuf = torch.empty(n_out + w.n_seq * w.n_qtok * W.HQ, dtype=torch.float32, device=dev)
    h_outbuf = torch.empty(d_outbuf.shape, dtype=torch.float32).pin_memory()
    out = d_outbuf[:n_out].view(w.n_seq, w.n_qtok, W.HQ, W.D)
    lse = d_outbuf[n_out:].view(w.n_seq, w.n_qtok, W.HQ)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    flush_acc = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush():
        # write 2 x L2, then read it back: the write evicts the inputs, the
        # read evicts the flush's own dirty lines (their write-back happens
        # here, not inside the next timed step)
        flush_buf.fill_(1.0)
        torch.sum(flush_buf, dim=0, out=flush_acc)

    def decode(passes, s):
        pa.pa_decode(cache.pool, q, cache.k_pool, cache.v_pool, table, table.shape[1], sl_dev, sl_host, w.n_seq,
                     w.n_qtok, W.HQ, w.scale, out, lse, ws, ws.numel(), cache.err, s, passes=passes)

    def capture(passes):
        """pa_decode (or one pass) captured once into a CUDA graph."""
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            decode(passes, side.cuda_stream)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            decode(passes, side.cuda_stream)
        torch.cuda.synchronize()
        return g

    g_all, g_split, g_merge = capture("all"), capture("split"), capture("merge")

    def capture_chain(n):
        """n pa_decode calls back to back in one CUDA graph: each step's split
        kernel is a programmatic dependent of the previous step's merge."""
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(n):
                decode("all", side.cuda_stream)
        torch.cuda.synchronize()
        return g
    clock_hz = 2.0e9

    def prime(n_steps):
        # a bounded device sleep ahead of the timed steps, so that the host
        # queues them all before the GPU reaches the first one
        torch.cuda._sleep(int(clock_hz * min(0.1, 1e-3 + 40e-6 * n_steps)))

    def timed(n, body, pre=None, headline=False):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        barrier()
        torch.cuda.synchronize()
        t0 = ClockSampler._now()
        prime(n)
        for i in range(n):
            if pre:
                pre()
            ev[i][0].record(stream)
            body()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier()
        if headline:
            clocks.mark_timed(t0, ClockSampler._now())
        return [ev[i][0].elapsed_time(ev[i][1]) for i in range(n)]

    clocks.begin()
    for _ in range(args.warmup):
        flush()
        g_all.replay()
    torch.cuda.synchronize()
    if cache.check() != pa.PA_OK:
        raise SystemExit("decode reported a device error")

    K = args.steps
    # ---- K steps back to back (the decode loop of a server), in graphs of up
    # to 20 chained steps, one event pair per graph.  Only where the step's
    # K/V bytes exceed the L2: no step can then find its inputs in L2.
    pipelined = kv_bytes > l2
    chain = min(K, 20)
    g_chain = capture_chain(chain)
    rest = K % chain
    g_rest = capture_chain(rest) if rest else None
    for _ in range(2):
        g_chain.replay()
    torch.cuda.synchronize()
    pipe_ms = None
    if pipelined:
        wall0 = time.perf_counter()
        chunks = timed(K // chain, g_chain.replay, headline=True)
        if g_rest is not None:
            chunks += timed(1, g_rest.replay)
        wall = time.perf_counter() - wall0
        pipe_ms = [sum(chunks) / K]
    # ---- each step alone: one graph replay between events, L2 flushed between
    wall0 = time.perf_counter()
    step_ms = timed(K, g_all.replay, flush, headline=not pipelined)
    if not pipelined:
        wall = time.perf_counter() - wall0
    if cache.check() != pa.PA_OK:
        raise SystemExit("decode reported a device error")
    # ---- the same steps, one replay each, no flush (warm)
    warm_ms = timed(K, g_all.replay)
    # ---- the split kernel alone (the roofline's kernel), merge replayed after it
    KS = max(3, min(K, 1000))
    split_ms = timed(KS, g_split.replay, lambda: (g_merge.replay(), flush()))

    # ---- end to end through the public API: packed host inputs in, host outputs back
    h2d = h_in.numel()
    d2h = h_outbuf.numel() * 4

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        cache.append(d_k, d_v, d_seq, d_pos, table, stream=stream.cuda_stream)
        decode("all", stream.cuda_stream)
        h_outbuf.copy_(d_outbuf, non_blocking=True)

    for _ in range(3):
        flush()
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = timed(args.e2e_steps, e2e_step, flush)
    clocks.end()
    clocks.__exit__()
    if cache.check() != pa.PA_OK:
        raise SystemExit("end-to-end step reported a device error")
    if not np.isfinite(h_outbuf.numpy()).all():
        raise SystemExit("non-finite output")

    # ---- max over ranks
    # algorithmic flops of a step: QK^T and PV over every visible key of every
    # query row (2 x 2 x 256 per key and row)
    flops = sum(sum(int(L) - w.n_qtok + t + 1 for t in range(w.n_qtok)) for L in w.seq_lens) * W.HQ * W.D * 4
    tensor_bound = w.n_qtok > 8  # row tiles: flop/B far above the HBM ridge
    my_iso, my_split, my_e2e, my_warm = (statistics.mean(x) for x in (step_ms, split_ms, e2e_ms, warm_ms))
    my_step = pipe_ms[0] if pipelined else my_iso
    step = rank_max(dist, my_step, dev)
    iso = rank_max(dist, my_iso, dev)
    split = rank_max(dist, my_split, dev)
    e2e = rank_max(dist, my_e2e, dev)
    warm = rank_max(dist, my_warm, dev)
    n = world
    value = job_gbps(n, kv_bytes, step)
    achieved = kv_bytes / (split * 1e-3) / 1e9
    peaks = measured_peaks()
    peak = float(peaks["hbm_gbs"]) if peaks and "hbm_gbs" in peaks else FALLBACK_HBM_GBS
    peak_src = "measured (MEASURED_PEAKS.json hbm_gbs, copy)" if peaks else "fallback"
    # binary16 MMA runs at the bf16 rate; a kernel timed alone takes the burst figure
    tpeak = float(peaks["bf16_tflops"]) if peaks and "bf16_tflops" in peaks else 1900.0
    tpeak_src = ("measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst; fp16 MMA at the bf16 rate)" if peaks
                 else "fallback 1.9 PFLOP/s")

    cpu = None
    if rank == 0 and n == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        ocache = oracle_cache(w)
        pairs = oracle_segments(w, ocache, args.cpu_budget, threads)
        secs = oracle_time(w, ocache, pairs, threads)
        pairs1 = oracle_segments(w, ocache, max(1.0, args.cpu_budget / 3), 1)
        secs1 = oracle_time(w, ocache, pairs1, 1)
        cpu = {"value": round(sample_bytes(w, pairs) / secs / 1e9, 4), "unit": "GB/s", "cores": threads,
               "kind": "oracle", "sample": sample_desc(w, pairs) + f"; {secs:.1f} s wall on {threads} threads",
               "single_thread": {"value": round(sample_bytes(w, pairs1) / secs1 / 1e9, 4), "unit": "GB/s",
                                 "cores": 1, "sample": sample_desc(w, pairs1) + f"; {secs1:.1f} s wall"}}

    if dist is not None:
        dist.destroy_process_group()
    if rank != 0:
        return
    wl = args.workload
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": n,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step, 5),
        "us_per_step": round(step * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(value / (kv_bytes / (PAGES_PAGED_3090_MS * 1e-3) / 1e9), 2) if wl == "ragged" else None,
        "vs_baseline_note": "vs RTX 3090 paged 4.095 ms/step on the same workload (lucebox PR #555); context only"
        if wl == "ragged" else None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {
            "workload": describe(w),
            "kv_bytes_per_step": kv_bytes,
            "kv_storage": f"K {W.TYPE_NAMES[w.k_type]} / V {W.TYPE_NAMES[w.v_type]}",
            "arithmetic": "fp16 tensor-core products, fp32 accumulation and softmax",
            "l2": (f"inputs larger than L2 ({kv_bytes / 1e6:.0f} MB of K/V against {l2 / 1e6:.0f} MB): steps back "
                   "to back, no flush" if pipelined else
                   "flushed between timed steps outside the timed region (2 x L2 written, then read back)"),
            "plan": plan,
            "timing": ((f"K pa_decode steps back to back in CUDA graphs of {chain} chained steps (each split "
                        "kernel a programmatic dependent of the previous merge), CUDA events on the launching "
                        "stream around each graph; value = bytes x K / total") if pipelined else
                       "CUDA events on the launching stream around each CUDA-graph replay of pa_decode "
                       "(split + merge), L2 flushed between; value from the mean over the steps"),
            "multi_gpu": f"global batch of {n} copies, partitioned by sequence, K/V bytes balanced" if n > 1 else None,
            "wall_s": round(wall, 3),
        },
        "timing": {"pipelined_us_per_step": round(step * 1e3, 2) if pipelined else None,
                   "isolated_flushed": percentiles(step_ms),
                   "isolated_flushed_gbps": round(job_gbps(n, kv_bytes, iso), 2),
                   "isolated_warm": percentiles(warm_ms), "isolated_warm_gbps": round(job_gbps(n, kv_bytes, warm), 2),
                   "split_kernel_flushed": percentiles(split_ms)},
        "frac_of_hbm_peak": round(value / n / peak, 4),
        "roofline": ({
            "bound": "hbm",
            "kernel": "pa_split_decode_kernel",
            "achieved": round(achieved, 2),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": profile_traffic(wl),
            "peak_source": peak_src,
            "split_us": round(split * 1e3, 2),
        } if not tensor_bound else {
            "bound": "tensor",
            "kernel": "pa_rows_tc_kernel",
            "achieved": round(flops / (split * 1e-3) / 1e12, 2),
            "peak": tpeak,
            "unit": "TFLOP/s",
            "frac": round(flops / (split * 1e-3) / 1e12 / tpeak, 4),
            "traffic": profile_traffic(wl),
            "peak_source": tpeak_src,
            "split_us": round(split * 1e3, 2),
            "flops_per_step": flops,
            "hbm_gbps_of_split": round(achieved, 2),
        }),
        "e2e": {"value": round(n * kv_bytes / (e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(e2e * 1e3, 2), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "pa_append_rows + pa_decode through the C ABI, pinned host buffers, no graph"},
        "gpu_launches": launches_per_step * K,  # split (+ merge) kernels per sub-batch, per timed step
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
