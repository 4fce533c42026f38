"""Benchmark: one hybrid decode step at 128K tokens (history GB/s and us/step).

Workload: 1 request, 4 KV heads x 8 query rows, head size 256, 131,072-token
history = 1,984 8-bit pages + 4,096 recent BF16 tokens, keys with 4 outlier
channels per head at 20x std, values and q ~ N(0, 1), seed 2; the 8-bit pages
are converted on the GPU before timing.  A step is one call of
tpk_decode_hybrid_batched (both tiers split over the thread blocks of one decode
launch, their partials folded by a second small launch).

value  = algorithmic history bytes / device time per step, inputs resident in
         HBM, L2 flushed between timed steps (256 MB written, then 256 MB read).
roofline = the decode kernel alone (CUDA events around its launch in the step's
         graph) against the measured copy peak; read_ceiling beside it is the
         fastest plain read of HBM measured in the same run.
e2e    = the same metric through the library's host-resident path: the step's
         history image (8-bit records, recent BF16 pages, q, page tables) sits in
         pinned host memory; each step stages it into a device slot through the
         stager (tpk_stager_*), runs the decode call on the slot and reads o and
         lse back.
tiers_128k = each tier alone over a 131,072-token history (all BF16: 536.9 MB; all
         8-bit: 287.3 MB), same call and timing, for the exact and the 8-bit
         kernel paths separately; kernel_* = the decode kernel alone, timed as
         the roofline's.
batched_16 = the 16-request batched hybrid decode (8K-64K tokens each, 1.35 GB),
         one multi-request call per step, same timing.
host_resident = 16 layers of such history images in pinned host memory through
         two device slots, each layer staged while the previous one decodes;
         link GB/s against a plain pinned copy measured in the same run.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {tpk,reference}]
Under torchrun (N > 1) every rank runs an independent replica on its GPU.
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

METRIC = "decode-attn history GB/s (% of HBM peak) and µs/step at 128K hybrid, 1 GB300"
WORKLOAD = ("hybrid 128K: 1 request, 4 KV heads x 8 q rows, head_dim 256, 131072 tokens = "
            "1984 8-bit pages + 4096 BF16 tokens, 4 outlier key channels at 20x std, seed 2")
KERNEL_SOURCES = ["tiered_paged_kv_gb300/csrc/common.cuh", "tiered_paged_kv_gb300/csrc/decode_common.cuh",
                  "tiered_paged_kv_gb300/csrc/decode_simt.cu", "tiered_paged_kv_gb300/csrc/decode_mma.cu",
                  "tiered_paged_kv_gb300/csrc/api.cu"]
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, the vendor's figure
kPageTokensBench = 64


def kernel_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        p = os.path.join(ROOT, f)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def sm_max_mhz():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return float(json.load(open(p))["sm_max_mhz"])
        except Exception:
            pass
    return 2070.0


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return float(json.load(open(p))["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def read_ceiling(dev, stream):
    """The fastest plain read of HBM found on this GPU, measured in the same run: a
    library integer maximum over 2 GiB (best of 10 after warm-up, CUDA events on the
    stream).  Context for the decode kernel, which only reads its history: a copy,
    the roofline's peak, reads and writes."""
    import torch

    with torch.cuda.stream(stream):
        x = torch.ones(1 << 29, dtype=torch.int32, device=dev)
        best = 0.0
        for i in range(13):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            torch.max(x)
            b.record(stream)
            b.synchronize()
            if i >= 3:
                best = max(best, x.numel() * 4 / (a.elapsed_time(b) * 1e-3) / 1e9)
        del x
    return best


def measured_traffic(impl_name):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "decode_hybrid_128k_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(impl_name)
        if e and e.get("kernel_hash") == kernel_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return dist, dist.get_rank(), ws
    return None, 0, 1


def max_over_ranks(dist, x):
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def host_cores():
    """The cores this process may run on (its affinity set)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def barrier(dist):
    if dist is not None:
        dist.barrier()


def build_workload():
    from tiered_paged_kv_gb300 import synth
    return synth.hybrid_128k(seed=2)


# --------------------------------------------------------------------- oracle
def oracle_time(w, rec_host, n_threads, sample_heads=None):
    """Time the oracle's hybrid step (as it stands) on host cores."""
    import oracle
    if sample_heads is not None:
        w = head_slice(w, sample_heads, rec_host)
        rec_host = w.meta["rec"]
    t0 = time.perf_counter()
    oracle.hybrid_workload(w, rec_host, n_threads=n_threads)
    dt = time.perf_counter() - t0
    return dt, w.history_bytes(), min(n_threads, w.B * w.H * w.G)


def oracle_quant_time(w, n_threads):
    """Time the oracle's page conversion (as it stands) on host cores: every 8-bit
    page of the workload on one thread, then the same pages split over n_threads
    threads (the C oracle releases the GIL).  Returns GB/s of BF16 read + records
    written, as the GPU conversion figure counts them, and the oracle's records."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    s8 = w.int8_slots()
    per_ph = 65536 + oracle.REC_BYTES
    rec = np.empty(w.n_slots * w.H * oracle.REC_BYTES, np.uint8)
    rec.fill(0)                                              # fault the pages in before timing
    oracle.quantize_pages(w.H, w.k_pool, w.v_pool, s8[:1], s8[:1], rec)   # load the library
    t0 = time.perf_counter()
    oracle.quantize_pages(w.H, w.k_pool, w.v_pool, s8, s8, rec)
    dt1 = time.perf_counter() - t0
    n = max(1, min(n_threads, len(s8)))
    parts = np.array_split(s8, n)
    t0 = time.perf_counter()
    with ThreadPoolExecutor(n) as ex:
        list(ex.map(lambda sl: oracle.quantize_pages(w.H, w.k_pool, w.v_pool, sl, sl, rec), parts))
    dt = time.perf_counter() - t0
    nb = len(s8) * w.H * per_ph
    return {"value": round(nb / dt / 1e9, 4), "unit": "GB/s", "cores": n, "value_1_thread": round(nb / dt1 / 1e9, 4),
            "sample": f"all {len(s8)} 8-bit pages x {w.H} heads of the workload ({dt1:.1f} s on one thread, "
                      f"{dt:.2f} s on {n})", "kind": "oracle"}, rec


def head_slice(w, heads, rec_host):
    """The same history restricted to the first `heads` KV heads (a sample)."""
    from tiered_paged_kv_gb300 import synth
    H = w.H
    rec = rec_host.reshape(w.n_slots, H, -1)[:, :heads].copy().reshape(-1)
    w2 = synth.Workload(H=heads, G=w.G, d=w.d, seed=w.seed, n_tokens=w.n_tokens, n8=w.n8, n_ex=w.n_ex,
                        pages=w.pages, n_slots=w.n_slots, q=w.q[:, :heads * w.G].copy(),
                        k_pool=w.k_pool[:, :heads].copy(), v_pool=w.v_pool[:, :heads].copy())
    w2.meta["rec"] = rec
    return w2


# ------------------------------------------------------------------ GPU arm
def graph_times(step, steps, warmup, stream, flush, flush_r):
    """Device times (ms) of `steps` CUDA-graph replays of step(), L2 flushed
    before each (256 MB written, then 256 MB read)."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            step()
        stream.synchronize()
        for _ in range(warmup):
            graph.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i, (a, b) in enumerate(ev):
            flush.fill_(float(i))
            flush_r.max()
            a.record(stream)
            graph.replay()
            b.record(stream)
        stream.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def loop_graph(step_fns, n_steps, stream):
    """One CUDA graph holding n_steps decode steps back to back, step i running
    step_fns[i % len(step_fns)].  With two resident copies of a history the steps
    alternate between them, so no step reads bytes that the step before it left
    in L2 (each copy's bytes are read again only after the other copy's)."""
    import torch
    with torch.cuda.stream(stream):
        for f in step_fns:
            f()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            for i in range(n_steps):
                step_fns[i % len(step_fns)]()
        stream.synchronize()
        graph.replay()  # the first replay uploads the graph
        stream.synchronize()
    return graph


def loop_times(step_fns, n_steps, stream, reps=3):
    """Per-step device time (ms) of n_steps steps in one graph (loop_graph), the
    median of `reps` replays timed by events around each replay."""
    import torch
    graph = loop_graph(step_fns, n_steps, stream)
    out = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            stream.synchronize()
            out.append(a.elapsed_time(b) / n_steps)
    return statistics.median(out)


def decode_kernel_loop_times(step_fns, n_steps, stream):
    """Mean device time (ms) of the decode kernel inside a graph of n_steps steps
    back to back (alternating as in loop_graph): every step's decode launch is
    captured between its own pair of CUDA events (tpk_set_decode_timing_events),
    and the graph is replayed twice (the first replay uploads it); the second
    replay's n_steps durations are averaged."""
    import torch

    import tiered_paged_kv_gb300 as tpk

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_steps)]
    with torch.cuda.stream(stream):
        for a, b in evs:   # the events exist from their first record on
            a.record(stream)
            b.record(stream)
        for f in step_fns:
            f()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            for i in range(n_steps):
                tpk.set_decode_timing_events(*evs[i])
                try:
                    step_fns[i % len(step_fns)]()
                finally:
                    tpk.set_decode_timing_events()
        for _ in range(2):
            graph.replay()
            stream.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / n_steps


def step_fields(hist_bytes, ms_loop, ms_iso, n_iso, peak):
    """A workload's step figures: timed as the headline is (steps back to back in
    one graph over two resident copies), and each step alone beside it (one graph
    replay between events, L2 flushed before it)."""
    out = {"us_per_step": round(ms_loop * 1e3, 2)}
    if hist_bytes is not None:
        gbs = hist_bytes / (ms_loop * 1e-3) / 1e9
        out.update({"GBps": round(gbs, 1), "hbm_frac": round(gbs / peak, 4)})
    iso = {"us_per_step_median": round(ms_iso * 1e3, 2), "steps": n_iso}
    if hist_bytes is not None:
        g = hist_bytes / (ms_iso * 1e-3) / 1e9
        iso.update({"GBps": round(g, 1), "hbm_frac": round(g / peak, 4)})
    out["isolated"] = iso
    return out


def decode_kernel_times(step, steps, stream, flush, flush_r):
    """Mean device time (ms) of the decode kernel alone: a graph of step() captured
    while the library records two events around its decode launch, replayed after
    an L2 flush, each replay read back before the next."""
    import torch

    import tiered_paged_kv_gb300 as tpk

    before = torch.cuda.Event(enable_timing=True)
    after = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        before.record(stream)   # the events exist from their first record on
        after.record(stream)
        stream.synchronize()
        tpk.set_decode_timing_events(before, after)
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
                step()
        finally:
            tpk.set_decode_timing_events()
        out = []
        for i in range(3 + steps):
            flush.fill_(float(i))
            flush_r.max()
            graph.replay()
            stream.synchronize()
            if i >= 3:
                out.append(before.elapsed_time(after))
    return sum(out) / len(out)


def run_batched(impl, args, stream, dev, flush, flush_r, peak, int_query=0, keep=None):
    """The 16-request batched hybrid decode (lengths uniform in [8K, 64K], 2048
    recent BF16 tokens each, 4 KV heads x 8 q rows, outlier keys, seed 3): one
    multi-request call per step, each request with its own page tables.  With
    keep (a dict), the workload and the step's output are stored in it."""
    import torch

    import tiered_paged_kv_gb300 as tpk
    from tiered_paged_kv_gb300 import synth

    w = synth.batched_hybrid(seed=3)
    H, G, B = w.H, w.G, w.B
    shape = tpk.Shape(H, impl=impl, kv_slots=w.n_slots, rec_slots=w.n_slots, int_query=int_query)
    with torch.cuda.stream(stream):
        kp = torch.from_numpy(w.k_pool.view(np.int16)).to(dev)
        vp = torch.from_numpy(w.v_pool.view(np.int16)).to(dev)
        q = torch.from_numpy(w.q.view(np.int16)).to(dev)
        rec = torch.zeros(w.n_slots * H * tpk.RECORD_BYTES, dtype=torch.uint8, device=dev)
        slots = torch.from_numpy(w.int8_slots()).to(dev)
        tpk.kv_quantize_pages(shape, kp, vp, slots, slots, len(slots), rec, stream)
        pt, off = w.exact_page_table()
        pt8, off8 = w.int8_page_table()
        pt_d = torch.from_numpy(pt).to(dev)
        pt8_d = torch.from_numpy(pt8).to(dev)
        o = torch.empty(B, H * G, 256, dtype=torch.float32, device=dev)
        lse = torch.empty(B, H * G, dtype=torch.float32, device=dev)
        nbytes = tpk.hybrid_workspace_bytes(shape, B)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def step():
        tpk.decode_hybrid_batched(shape, B, q, kp, vp, rec, pt_d, off, w.n_ex, pt8_d, off8, w.n8, o, lse, ws,
                                  nbytes, stream)

    with torch.cuda.stream(stream):
        kp2, vp2, rec2 = kp.clone(), vp.clone(), rec.clone()

    def step2():
        tpk.decode_hybrid_batched(shape, B, q, kp2, vp2, rec2, pt_d, off, w.n_ex, pt8_d, off8, w.n8, o, lse, ws,
                                  nbytes, stream)

    times = graph_times(step, args.tier_steps, 3, stream, flush, flush_r)
    lms = loop_times([step, step2], max(10, args.tier_steps), stream)
    st, flags = tpk.get_device_status(reset=True, stream=stream)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags} (batched)")
    kms = decode_kernel_loop_times([step, step2], max(10, args.tier_steps), stream)
    if keep is not None:
        stream.synchronize()
        keep["w"], keep["o"] = w, o.cpu().numpy()
    ms = statistics.median(times)
    kgbs = w.history_bytes() / (kms * 1e-3) / 1e9
    return {"history_bytes": w.history_bytes(), "requests": B, "tokens": int(w.n_tokens.sum()),
            **step_fields(w.history_bytes(), lms, ms, len(times), peak),
            "kernel_us_mean": round(kms * 1e3, 2), "kernel_GBps": round(kgbs, 1),
            "kernel_hbm_frac": round(kgbs / peak, 4),
            "workload": "16 requests, lengths uniform in [8192, 65536] (seed 3), 2048 BF16 recent each, "
                        "4 KV heads x 8 q rows, head_dim 256, outlier keys"}


def run_tier(which, impl, args, stream, dev, flush, flush_r, peak, int_query=0):
    """One tier alone over a 131,072-token history of the main workload's shape
    (4 KV heads x 8 q rows, head_dim 256, 4 outlier key channels at 20x std):
    'exact' = all BF16, 'int8' = all 8-bit (2048 pages, converted on the GPU
    first), through the same multi-request call."""
    import torch

    import tiered_paged_kv_gb300 as tpk
    from tiered_paged_kv_gb300 import synth

    w = synth.make_workload([131072], None if which == "exact" else 0, H=4, seed=12,
                            key_sigma="outliers")
    H, G = w.H, w.G
    shape = tpk.Shape(H, impl=impl, kv_slots=w.n_slots, rec_slots=w.n_slots, int_query=int_query)
    with torch.cuda.stream(stream):
        kp = torch.from_numpy(w.k_pool.view(np.int16)).to(dev)
        vp = torch.from_numpy(w.v_pool.view(np.int16)).to(dev)
        q = torch.from_numpy(w.q.view(np.int16)).to(dev)
        rec = torch.zeros(w.n_slots * H * tpk.RECORD_BYTES if which == "int8" else 16, dtype=torch.uint8,
                          device=dev)
        if which == "int8":
            slots = torch.from_numpy(w.int8_slots()).to(dev)
            tpk.kv_quantize_pages(shape, kp, vp, slots, slots, len(slots), rec, stream)
        pt, off = w.exact_page_table()
        pt8, off8 = w.int8_page_table()
        pt_d = torch.from_numpy(np.concatenate([pt, np.zeros(1, np.int32)])).to(dev)
        pt8_d = torch.from_numpy(np.concatenate([pt8, np.zeros(1, np.int32)])).to(dev)
        o = torch.empty(1, H * G, 256, dtype=torch.float32, device=dev)
        lse = torch.empty(1, H * G, dtype=torch.float32, device=dev)
        nbytes = tpk.hybrid_workspace_bytes(shape, 1)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def step():
        tpk.decode_hybrid_batched(shape, 1, q, kp, vp, rec, pt_d, off, w.n_ex, pt8_d, off8, w.n8, o, lse, ws,
                                  nbytes, stream)

    with torch.cuda.stream(stream):
        kp2, vp2, rec2 = kp.clone(), vp.clone(), rec.clone()

    def step2():
        tpk.decode_hybrid_batched(shape, 1, q, kp2, vp2, rec2, pt_d, off, w.n_ex, pt8_d, off8, w.n8, o, lse, ws,
                                  nbytes, stream)

    times = graph_times(step, args.tier_steps, 3, stream, flush, flush_r)
    lms = loop_times([step, step2], max(10, args.tier_steps), stream)
    st, flags = tpk.get_device_status(reset=True, stream=stream)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags} ({which} tier)")
    kms = decode_kernel_loop_times([step, step2], max(10, args.tier_steps), stream)
    ms = statistics.median(times)
    kgbs = w.history_bytes() / (kms * 1e-3) / 1e9
    return {"history_bytes": w.history_bytes(), **step_fields(w.history_bytes(), lms, ms, len(times), peak),
            "kernel_us_mean": round(kms * 1e3, 2), "kernel_GBps": round(kgbs, 1),
            "kernel_hbm_frac": round(kgbs / peak, 4),
            "workload": f"131072 tokens {'all BF16' if which == 'exact' else 'all 8-bit (2048 pages)'}, "
                        "4 KV heads x 8 q rows, head_dim 256, outlier keys, seed 12"}


def run_exact_32k(impl, args, stream, dev, flush, flush_r, peak):
    """The exact tier alone: a 32,768-token BF16 history of one request (4 KV heads x
    8 q rows, head_dim 256, K, V, q ~ N(0, 1)) at a seeded permutation of page slots
    (seed 1).  Timed: the multi-request call per step (graph replays, L2 flushed),
    and the decode kernel alone.  Beside it, the same history cut at the seeded
    token index into two primitive exact calls whose partials one merge folds:
    its step time and its largest difference from the unsplit result."""
    import torch

    import tiered_paged_kv_gb300 as tpk
    from tiered_paged_kv_gb300 import synth

    w = synth.exact_32k(seed=1)
    H, G, N = w.H, w.G, int(w.n_tokens[0])
    cut = int(w.meta["split_at"])
    shape = tpk.Shape(H, impl=impl, kv_slots=w.n_slots, rec_slots=1)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    s1 = max(1, min(sms // H - 1, round(sms // H * cut / N)))
    s2 = max(1, sms // H - s1)
    with torch.cuda.stream(stream):
        kp = torch.from_numpy(w.k_pool.view(np.int16)).to(dev)
        vp = torch.from_numpy(w.v_pool.view(np.int16)).to(dev)
        q = torch.from_numpy(w.q.view(np.int16)).to(dev)
        rec = torch.zeros(16, dtype=torch.uint8, device=dev)
        pt, off = w.exact_page_table()
        pt_d = torch.from_numpy(np.concatenate([pt, np.zeros(1, np.int32)])).to(dev)
        pt8_d = torch.zeros(1, dtype=torch.int32, device=dev)
        off8 = np.zeros(2, np.int32)
        o = torch.empty(1, H * G, 256, dtype=torch.float32, device=dev)
        lse = torch.empty(1, H * G, dtype=torch.float32, device=dev)
        nbytes = tpk.hybrid_workspace_bytes(shape, 1)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        o_part = torch.empty(s1 + s2, H * G, 256, dtype=torch.float32, device=dev)
        lse_part = torch.empty(s1 + s2, H * G, dtype=torch.float32, device=dev)
        o_acc = torch.empty(H * G, 256, dtype=torch.float32, device=dev)
        lse_acc = torch.empty(H * G, dtype=torch.float32, device=dev)

    def step():
        tpk.decode_hybrid_batched(shape, 1, q, kp, vp, rec, pt_d, off, w.n_ex, pt8_d, off8, w.n8, o, lse, ws,
                                  nbytes, stream)

    with torch.cuda.stream(stream):
        kp2, vp2 = kp.clone(), vp.clone()

    def step2():
        tpk.decode_hybrid_batched(shape, 1, q, kp2, vp2, rec, pt_d, off, w.n_ex, pt8_d, off8, w.n8, o, lse, ws,
                                  nbytes, stream)

    def step_split():
        o_acc.zero_()
        lse_acc.fill_(float("-inf"))
        tpk.decode_attn_exact(shape, q, kp, vp, pt_d, 0, cut, s1, o_part[:s1], lse_part[:s1], stream)
        tpk.decode_attn_exact(shape, q, kp, vp, pt_d, cut, N, s2, o_part[s1:], lse_part[s1:], stream)
        tpk.merge_lse(s1 + s2, H * G, 256, o_part, lse_part, o_acc, lse_acc, stream)

    times = graph_times(step, args.tier_steps, 3, stream, flush, flush_r)
    kms = decode_kernel_loop_times([step, step2], max(10, args.tier_steps), stream)
    times_split = graph_times(step_split, args.tier_steps, 3, stream, flush, flush_r)
    lms = loop_times([step, step2], max(10, args.tier_steps), stream)
    stream.synchronize()
    st, flags = tpk.get_device_status(reset=True, stream=stream)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags} (exact 32K)")
    o_u, l_u = o[0].cpu().numpy(), lse[0].cpu().numpy()
    o_s, l_s = o_acc.cpu().numpy(), lse_acc.cpu().numpy()
    ms, ms_split = statistics.median(times), statistics.median(times_split)
    hb = w.history_bytes()
    kgbs = hb / (kms * 1e-3) / 1e9
    return {"history_bytes": hb, **step_fields(hb, lms, ms, len(times), peak), "kernel_us_mean": round(kms * 1e3, 2),
            "kernel_GBps": round(kgbs, 1), "kernel_hbm_frac": round(kgbs / peak, 4),
            "split_merge": {"split_at": cut, "splits": [s1, s2],
                            "us_per_step_median": round(ms_split * 1e3, 2),
                            "max_abs_do_over_max_o": float(np.abs(o_s - o_u).max() / np.abs(o_u).max()),
                            "max_abs_dlse": float(np.abs(l_s - l_u).max()),
                            "how": "two tpk_decode_attn_exact calls ([0, cut), [cut, N)) + one tpk_merge_lse "
                                   "into a fresh accumulator, against the unsplit call"},
            "workload": "32768 tokens all BF16, 1 request, 4 KV heads x 8 q rows, head_dim 256, K, V, q ~ N(0, 1), "
                        "page slots at a seeded permutation (seed 1)"}


def run_tiny(impl, args, stream, dev, flush, flush_r, peak, keep=None):
    """The tiny hybrid decode (1 request, 1 KV head x 8 query rows, 1024 tokens =
    12 8-bit pages + 256 BF16 tokens, per-channel std log-uniform in [0.1, 10],
    seed 0): a launch this small is timed for its fixed cost, not its bandwidth."""
    import torch

    import tiered_paged_kv_gb300 as tpk
    from tiered_paged_kv_gb300 import synth

    w = synth.tiny_hybrid(seed=0)
    H, G = w.H, w.G
    shape = tpk.Shape(H, impl=impl, kv_slots=w.n_slots, rec_slots=w.n_slots)
    with torch.cuda.stream(stream):
        kp = torch.from_numpy(w.k_pool.view(np.int16)).to(dev)
        vp = torch.from_numpy(w.v_pool.view(np.int16)).to(dev)
        q = torch.from_numpy(w.q.view(np.int16)).to(dev)
        rec = torch.zeros(w.n_slots * H * tpk.RECORD_BYTES, dtype=torch.uint8, device=dev)
        slots = torch.from_numpy(w.int8_slots()).to(dev)
        tpk.kv_quantize_pages(shape, kp, vp, slots, slots, len(slots), rec, stream)
        pt, off = w.exact_page_table()
        pt8, off8 = w.int8_page_table()
        pt_d = torch.from_numpy(pt).to(dev)
        pt8_d = torch.from_numpy(pt8).to(dev)
        o = torch.empty(1, H * G, 256, dtype=torch.float32, device=dev)
        lse = torch.empty(1, H * G, dtype=torch.float32, device=dev)
        nbytes = tpk.hybrid_workspace_bytes(shape, 1)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def step():
        tpk.decode_hybrid_batched(shape, 1, q, kp, vp, rec, pt_d, off, w.n_ex, pt8_d, off8, w.n8, o, lse, ws,
                                  nbytes, stream)

    times = graph_times(step, args.tier_steps, 3, stream, flush, flush_r)
    lms = loop_times([step], max(10, args.tier_steps), stream)
    stream.synchronize()
    st, flags = tpk.get_device_status(reset=True, stream=stream)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags} (tiny)")
    if keep is not None:
        keep["w"], keep["o"] = w, o.cpu().numpy()
    ms = statistics.median(times)
    return {"history_bytes": w.history_bytes(), **step_fields(None, lms, ms, len(times), peak),
            "workload": "1 request, 1 KV head x 8 q rows, head_dim 256, 1024 tokens = 12 8-bit pages + 256 BF16, "
                        "K, V with per-channel std log-uniform in [0.1, 10], seed 0 (launch-bound: a parity "
                        "config)"}


def hybrid_error(w, o_gpu, rec_host, n_thr):
    """Worst merged error of the hybrid result against attention over the original
    BF16 history (no quantisation), for the oracle's hybrid step on its own records
    and for the GPU's result: max |o - o_fp| over rows and channels (the pages'
    bound is 0.005), also over max |o_fp| and as an RMS ratio."""
    import oracle
    of, _ = oracle.full_precision_workload(w, n_threads=n_thr)
    oo, _ = oracle.hybrid_workload(w, rec_host, n_threads=n_thr)
    out = {"bound": 0.005, "max_abs_o_fp": float(np.abs(of).max())}
    for name, o in (("oracle", oo), ("gpu", np.asarray(o_gpu, np.float64).reshape(of.shape))):
        e = np.abs(o - of)
        out[name] = {"max_abs": round(float(e.max()), 6), "max_abs_over_max_o": round(float(e.max() / np.abs(of).max()), 6),
                     "rms_rel": round(float(np.sqrt((e ** 2).mean() / (of ** 2).mean())), 6),
                     "bound_met": bool(e.max() <= 0.005)}
    return out


def run_gpu(args, dist, rank, world):
    import torch

    import tiered_paged_kv_gb300 as tpk
    from tiered_paged_kv_gb300 import build as tbuild

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    tbuild.build()
    impl = {"simt": tpk.IMPL_SIMT, "tensor": tpk.IMPL_TENSOR, "default": tpk.IMPL_DEFAULT}[args.kernel]
    w = build_workload()
    H, G = w.H, w.G
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(dev)
    if args.int_query and impl == tpk.IMPL_SIMT:
        raise SystemExit("--int-query runs on the tensor-core kernel only")
    shape = tpk.Shape(H, impl=impl, kv_slots=w.n_slots, rec_slots=w.n_slots, int_query=int(args.int_query))
    with torch.cuda.stream(stream):
        kp = torch.from_numpy(w.k_pool.view(np.int16)).to(dev)
        vp = torch.from_numpy(w.v_pool.view(np.int16)).to(dev)
        q = torch.from_numpy(w.q.view(np.int16)).to(dev)
        rec = torch.zeros(w.n_slots * H * tpk.RECORD_BYTES, dtype=torch.uint8, device=dev)
        slots = torch.from_numpy(w.int8_slots()).to(dev)
        pt, off = w.exact_page_table()
        pt8, off8 = w.int8_page_table()
        pt_d = torch.from_numpy(pt).to(dev)
        pt8_d = torch.from_numpy(pt8).to(dev)
        o = torch.empty(1, H * G, 256, dtype=torch.float32, device=dev)
        lse = torch.empty(1, H * G, dtype=torch.float32, device=dev)
        nbytes = tpk.hybrid_workspace_bytes(shape, 1)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        tpk.workspace_init(ws, nbytes, stream)
        # fresh page conversion of every 8-bit page (timed separately: the median of
        # five conversions of all 7,936 page-heads, each rewriting the same records)
        q_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(6)]
        for a, b in q_ev:
            a.record(stream)
            tpk.kv_quantize_pages(shape, kp, vp, slots, slots, len(slots), rec, stream)
            b.record(stream)
        flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        flush_r = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream.synchronize()
    quant_ms = statistics.median([a.elapsed_time(b) for a, b in q_ev[1:]])
    st, flags = tpk.get_device_status(reset=True, stream=stream)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags}")

    def step():
        tpk.decode_hybrid_batched(shape, 1, q, kp, vp, rec, pt_d, off, w.n_ex, pt8_d, off8, w.n8, o, lse, ws,
                                  nbytes, stream)

    # a second resident copy of the history: the timed steps alternate between the
    # two (2 x 295 MB, more than twice L2), so no step reads what the one before left in L2
    with torch.cuda.stream(stream):
        kp2, vp2, rec2 = kp.clone(), vp.clone(), rec.clone()

    def step2():
        tpk.decode_hybrid_batched(shape, 1, q, kp2, vp2, rec2, pt_d, off, w.n_ex, pt8_d, off8, w.n8, o, lse, ws,
                                  nbytes, stream)

    hist_bytes = w.history_bytes()
    launches_per_step = 2  # the decode kernel, then the fold kernel (heads split over several blocks)
    # a step is captured in a CUDA graph (the split plan and tensor maps are kernel
    # parameters); the timed region is one graph of K steps back to back, and every
    # step is also timed alone (one replay each, L2 flushed before it)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()                          # first calls resolve and cache device attributes
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            step()
        stream.synchronize()
    loop = loop_graph([step, step2], args.steps, stream)
    with torch.cuda.stream(stream), ClockSampler(local) as clk:
        for _ in range(args.warmup):
            graph.replay()
        # soak: back-to-back steps for about a second so the clock sampler sees
        # the GPU under this load; the sampler keeps running through the timed steps
        t_end = time.perf_counter() + args.soak
        while time.perf_counter() < t_end:
            loop.replay()
            stream.synchronize()
        barrier(dist)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        loop.replay()                       # exactly K steps
        t1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        barrier(dist)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            # each step alone: evict the previous step's lines from L2 (write 256 MB,
            # then read another 256 MB so that the dirty lines are written back before it)
            flush.fill_(float(i))
            flush_r.max()
            starts[i].record(stream)
            graph.replay()
            ends[i].record(stream)
        stream.synchronize()
    ms_loop = t0.elapsed_time(t1) / args.steps
    ms_max = max_over_ranks(dist, ms_loop)
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_mean = sum(times) / len(times)
    st, flags = tpk.get_device_status(reset=True, stream=stream)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags} after timing")
    kernel_ms = decode_kernel_loop_times([step, step2], args.steps, stream)
    kernel_iso_ms = decode_kernel_times(step, args.steps, stream, flush, flush_r)
    read_gbs = read_ceiling(dev, stream)

    # ---- each tier alone at 128K (the exact and the 8-bit kernel paths)
    peak, peak_kind = hbm_peak()
    stream.synchronize()
    o_step = o.cpu().numpy()  # the timed step's result (for the hybrid error below)
    tiers = batched = int_query = exact32 = tiny = None
    batch_keep, tiny_keep = {}, {}
    if args.tier_steps > 0:
        tiny = run_tiny(impl, args, stream, dev, flush, flush_r, peak, keep=tiny_keep)
        tiers = {k: run_tier(k, impl, args, stream, dev, flush, flush_r, peak) for k in ("exact", "int8")}
        exact32 = run_exact_32k(impl, args, stream, dev, flush, flush_r, peak)
        batched = run_batched(impl, args, stream, dev, flush, flush_r, peak, keep=batch_keep)
        if impl != tpk.IMPL_SIMT and not args.int_query:
            int_query = run_int_query(w, shape, step, args, stream, dev, flush, flush_r, peak, impl,
                                      (q, kp, vp, rec, pt_d, off, pt8_d, off8, o, lse, ws, nbytes))

    # ---- the economic gate at 32K, 64K and 128K (link model from measured stager copies)
    gate_obj = None
    if args.gate:
        gate_obj = run_gate(args, stream, dev, flush, flush_r, [32768, 65536, 131072],
                            layers_measured=args.gate_layers)

    # ---- end to end from pinned host memory (packed history, identity page tables)
    e2e = run_e2e(args, w, rec, shape, stream, dev, dist)
    host_res = run_host_resident(args, w, rec, shape, stream, dev, dist) if args.layers > 0 else None

    # ---- CPU oracle baseline (rank 0, N = 1)
    cpu = herr = None
    if rank == 0 and world == 1 and not args.no_cpu:
        n_thr = host_cores()
        # the oracle's own page conversion (timed), whose records its decode then reads
        quant_cpu, rec_host = oracle_quant_time(w, n_thr)
        # repeat whole oracle steps until about 10 s of CPU work has been timed
        reps, dt = 0, 0.0
        while reps == 0 or dt * cores < 10.0:
            d, nb, cores = oracle_time(w, rec_host, n_thr)
            reps, dt = reps + 1, dt + d
        reps1, dt1 = 0, 0.0
        while reps1 == 0 or dt1 < 5.0:
            d, nb1, _ = oracle_time(w, rec_host, 1, sample_heads=1)
            reps1, dt1 = reps1 + 1, dt1 + d
        cpu = {"value": round(reps * nb / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"the full 128K hybrid step (all 4 KV heads) {reps} times, {dt:.1f} s on {cores} threads "
                         f"(threads over (request, KV head, query row))",
               "value_1_thread": round(reps1 * nb1 / dt1 / 1e9, 4),
               "sample_1_thread": f"one KV head of the same step on one thread, {reps1} times, {dt1:.1f} s",
               "host_cores_available": n_thr,
               "page_conversion": quant_cpu}
        # worst merged error against unquantised attention (the oracle's and the GPU's)
        herr = {"hybrid_128k": hybrid_error(w, o_step, rec_host, n_thr)}
        if tiny_keep:
            import oracle
            wt = tiny_keep["w"]
            rec_t = np.zeros(wt.n_slots * wt.H * oracle.REC_BYTES, np.uint8)
            st8 = wt.int8_slots()
            oracle.quantize_pages(wt.H, wt.k_pool, wt.v_pool, st8, st8, rec_t)
            herr["tiny_hybrid"] = hybrid_error(wt, tiny_keep["o"], rec_t, n_thr)
        if batch_keep:
            import oracle
            wb = batch_keep["w"]
            rec_b = np.zeros(wb.n_slots * wb.H * oracle.REC_BYTES, np.uint8)
            sb = wb.int8_slots()
            from concurrent.futures import ThreadPoolExecutor
            with ThreadPoolExecutor(n_thr) as ex:
                list(ex.map(lambda sl: oracle.quantize_pages(wb.H, wb.k_pool, wb.v_pool, sl, sl, rec_b),
                            np.array_split(sb, n_thr)))
            herr["batched_16"] = hybrid_error(wb, batch_keep["o"], rec_b, n_thr)
    achieved = hist_bytes / (kernel_ms * 1e-3) / 1e9  # the decode kernel alone
    # secondary ceiling: the step's multiply-adds (QK and PV: 2 G d per token and KV
    # head) on the CUDA cores alone (128 FP32 lanes per SM at the maximum SM clock)
    n_tok = int(np.sum(w.n_ex)) + kPageTokensBench * int(np.sum(w.n8))
    fma_step = n_tok * w.H * 2 * w.G * 256
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz = sm_max_mhz()
    fma_peak = sms * 128 * sm_mhz * 1e6
    value = world * hist_bytes / (ms_max * 1e-3) / 1e9
    traffic = measured_traffic(args.kernel + ("_int_query" if args.int_query else ""))
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max, 5), "us_per_step": round(ms_max * 1e3, 2),
        "hbm_frac": round(hist_bytes / (ms_loop * 1e-3) / 1e9 / peak, 4),  # the whole step, as `value`
        "isolated_step": {"us_mean": round(ms_mean * 1e3, 2), "us_median": round(statistics.median(times) * 1e3, 2),
                          "us_p10_p90": [round(np.percentile(times, 10) * 1e3, 2),
                                         round(np.percentile(times, 90) * 1e3, 2)],
                          "GBps": round(hist_bytes / (ms_mean * 1e-3) / 1e9, 1),
                          "hbm_frac": round(hist_bytes / (ms_mean * 1e-3) / 1e9 / peak, 4), "steps": len(times),
                          "how": "each step alone: one graph replay between CUDA events, L2 flushed before it; "
                                 "includes the graph's launch and the events' own cost (a graph of two tiny "
                                 "kernels timed this way takes about 6.6 us)"},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "dtype_detail": ("BF16 and 8-bit history in; tensor-core products with f32 accumulation: 8-bit tier on "
                         "f16 inputs (codes exact, the folded query as high + low planes, probabilities as one "
                         "plane), exact tier on bf16 inputs (query and history exact, probabilities as high + low "
                         "planes); softmax, rescales and the merge in f32"
                         if args.kernel != "simt" else "BF16 and 8-bit history in; f32 arithmetic throughout"),
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "history_bytes_per_step": hist_bytes, "kernel": args.kernel,
                   "query": "8-bit integer query on the 8-bit tier" if args.int_query else "float",
                   "l2": "inputs larger than L2: the timed steps alternate between two resident copies of the "
                         "history (2 x 295 MB against 129 MB of L2), so each step reads its bytes from HBM; the "
                         "isolated-step figures flush L2 before every step instead (256 MB written, then 256 MB read)",
                   "clocks_sampled": "nvidia-smi every 100 ms over a soak of back-to-back steps and the timed steps",
                   "launch": "timed region: one CUDA graph of K steps (decode + fold kernels each) back to back, "
                             "replayed once between CUDA events; e2e calls the C ABI directly",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "page_conversion_us": round(quant_ms * 1e3, 1),
                   "page_conversion_GBps": round((w.H * int(w.n8.sum()) * (65536 + 35072)) / (quant_ms * 1e-3) / 1e9, 1)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "kernel": "decode_mma_kernel",
                     "kernel_us_mean": round(kernel_ms * 1e3, 2),
                     "timing": "CUDA events recorded around every step's decode launch inside a graph of K "
                               "steps back to back that alternate between the two resident copies as the timed "
                               "region does (tpk_set_decode_timing_events, one event pair per step); the fold "
                               "launch that follows each is outside it",
                     "isolated_kernel_us_mean": round(kernel_iso_ms * 1e3, 2),
                     "isolated_frac": round(hist_bytes / (kernel_iso_ms * 1e-3) / 1e9 / peak, 4),
                     "step_frac": round(hist_bytes / (ms_loop * 1e-3) / 1e9 / peak, 4),
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "read_ceiling": {"GBps": round(read_gbs, 1), "frac": round(achieved / read_gbs, 4),
                                      "step_frac": round(hist_bytes / (ms_loop * 1e-3) / 1e9 / read_gbs, 4),
                                      "how": "library int32 maximum over 2 GiB in the same run, best of 10: "
                                             "the fastest plain read found (the peak above is a copy)"},
                     "secondary": {"bound": "cuda-core fma", "fma_per_step": fma_step,
                                   "peak_tfma_per_s": round(fma_peak / 1e12, 2),
                                   "floor_us": round(fma_step / fma_peak * 1e6, 2),
                                   "peak_source": f"{sms} SMs x 128 FP32 lanes x {sm_mhz:.0f} MHz; QK and PV run "
                                                  "on the tensor cores, so the kernel is not held to it"},
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s"},
        "e2e": e2e,
        "host_resident": host_res,
        "tiny_hybrid": tiny,
        "tiers_128k": tiers,
        "exact_32k": exact32,
        "batched_16": batched,
        "hybrid_error": herr,
        "gate": gate_obj,
        "int_query_variant": int_query,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_int_query(w, shape, step_float, args, stream, dev, flush, flush_r, peak, impl, bufs):
    """The integer-query variant of the 8-bit tier (its QK on the integer tensor
    path) beside the float query, same protocol (graph replays, L2 flushed): the
    128K hybrid step, the 8-bit tier alone and the 16-request batch."""
    import tiered_paged_kv_gb300 as tpk

    q, kp, vp, rec, pt_d, off, pt8_d, off8, o, lse, ws, nbytes = bufs
    shape_iq = tpk.Shape(shape.kv_heads, impl=shape.impl, kv_slots=shape.kv_slots, rec_slots=shape.rec_slots,
                         int_query=1)

    def step_iq():
        tpk.decode_hybrid_batched(shape_iq, 1, q, kp, vp, rec, pt_d, off, w.n_ex, pt8_d, off8, w.n8, o, lse, ws,
                                  nbytes, stream)

    out = {}
    for name, fn in (("float_query", step_float), ("int_query", step_iq)):
        times = graph_times(fn, args.tier_steps, 3, stream, flush, flush_r)
        st, flags = tpk.get_device_status(reset=True, stream=stream)
        if st != 0:
            raise RuntimeError(f"device status {st} flags {flags} ({name})")
        ms = statistics.median(times)
        gbs = w.history_bytes() / (ms * 1e-3) / 1e9
        out[f"hybrid_128k_{name}"] = {"us_per_step_median": round(ms * 1e3, 2), "GBps": round(gbs, 1),
                                      "hbm_frac": round(gbs / peak, 4), "steps": len(times)}
    out["int8_128k_int_query"] = run_tier("int8", impl, args, stream, dev, flush, flush_r, peak, int_query=1)
    out["batched_16_int_query"] = run_batched(impl, args, stream, dev, flush, flush_r, peak, int_query=1)
    return out


def run_e2e(args, w, rec_dev, shape, stream, dev, dist):
    """The step end to end through the library's host-resident path: the step's
    history image (8-bit records, recent BF16 pages, q, page tables) sits in pinned
    host memory; each step stages it into a device slot (tpk_stager_*), decodes
    from the slot and reads o and lse back."""
    import torch

    import tiered_paged_kv_gb300 as tpk

    H, G = w.H, w.G
    img, off = w.packed_image(rec_dev.cpu().numpy())
    img_h = torch.from_numpy(img).pin_memory()
    slots = [torch.empty(off["nbytes"], dtype=torch.uint8, device=dev) for _ in range(2)]
    o_d = torch.empty(1, H * G, 256, dtype=torch.float32, device=dev)
    lse_d = torch.empty(1, H * G, dtype=torch.float32, device=dev)
    o_h = torch.empty(1, H * G, 256, dtype=torch.float32).pin_memory()
    lse_h = torch.empty(1, H * G, dtype=torch.float32).pin_memory()
    shape2 = tpk.Shape(H, impl=shape.impl, kv_slots=off["n_exact_pages"], rec_slots=off["n_int8_pages"],
                       int_query=shape.int_query)
    nbytes = tpk.hybrid_workspace_bytes(shape2, 1)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    views = [slot_views(s, off, w) for s in slots]
    d2h_bytes = o_h.numel() * 4 + lse_h.numel() * 4
    st = tpk.Stager(slots, off["nbytes"])

    def stage():
        slot, _ = st.stage([(img_h, 0, off["nbytes"])])
        return slot

    def consume(slot):
        st.acquire(slot, stream)
        rec, k, v, q, pt, pt8 = views[slot]
        tpk.decode_hybrid_batched(shape2, 1, q, k, v, rec, pt, off["req_page_off"], w.n_ex, pt8,
                                  off["req_page_off8"], w.n8, o_d, lse_d, ws, nbytes, stream)
        st.release(slot, stream)
        o_h.copy_(o_d, non_blocking=True)
        lse_h.copy_(lse_d, non_blocking=True)

    def run(n):
        # n steps, each with its own staging copy and read-back.  Step i + 1's copy is
        # queued before step i's decode and read-back (two slots), so the large
        # host->device copies follow one another instead of each waiting behind the
        # previous step's small device->host read.
        nxt = stage()
        for i in range(n):
            cur = nxt
            nxt = stage() if i + 1 < n else None
            consume(cur)

    try:
        with torch.cuda.stream(stream):
            tpk.workspace_init(ws, nbytes, stream)
            run(max(1, args.warmup))
            stream.synchronize()
            barrier(dist)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            steps = max(3, args.steps // 2)
            ev[0].record(stream)
            ev[0].synchronize()             # the first staging copy starts after the start event
            run(steps)
            ev[1].record(stream)
            stream.synchronize()
            barrier(dist)
    finally:
        st.close()
    ms = ev[0].elapsed_time(ev[1]) / steps
    ms = max_over_ranks(dist, ms)
    world = dist.get_world_size() if dist is not None else 1
    return {"value": round(world * w.history_bytes() / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "us_per_step": round(ms * 1e3, 1), "h2d_bytes_per_step": int(off["nbytes"]),
            "d2h_bytes_per_step": int(d2h_bytes), "steps": steps,
            "path": "tpk_stager_stage/acquire/release + tpk_decode_hybrid_batched from pinned host memory",
            "pipelining": "two device slots; each step's staging copy is queued one step ahead of its decode"}


def slot_views(s, off, w):
    """Typed device views of one staged history image (a uint8 tensor)."""
    H, G = w.H, w.G
    n8, ne = off["n_int8_pages"], off["n_exact_pages"]
    return (s[off["rec"]:off["rec"] + n8 * H * 35072],
            s[off["k"]:off["k"] + ne * H * 64 * 256 * 2],
            s[off["v"]:off["v"] + ne * H * 64 * 256 * 2],
            s[off["q"]:off["q"] + w.B * H * G * 256 * 2],
            s[off["pt"]:off["pt"] + max(ne, 1) * 4],
            s[off["pt8"]:off["pt8"] + max(n8, 1) * 4])


def host_mem_available():
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def run_host_resident(args, w, rec_dev, shape, stream, dev, dist, layers=None, steps=None, label=None,
                      pack13_dev=None):
    """Many layers of the same-sized history in pinned host memory (one image per
    layer; the content of every layer is this workload's), two device slots: per
    step every layer is staged while the previous layer decodes.  Bound by the
    host->device link; the link peak is a plain 1 GiB pinned copy in the same run.
    With pack13_dev (the exact pages' 13-bit records) the exact tier travels as
    compacted 13-bit records and is unpacked into a BF16 scratch pool before each
    layer's decode."""
    import torch

    import tiered_paged_kv_gb300 as tpk

    H, G = w.H, w.G
    img, off = w.packed_image(rec_dev.cpu().numpy(),
                              None if pack13_dev is None else pack13_dev.cpu().numpy())
    lossless = pack13_dev is not None
    layers = args.layers if layers is None else layers
    steps = args.host_steps if steps is None else steps
    avail = host_mem_available()
    if avail and layers * off["nbytes"] * 2 > avail:  # keep well inside the host's memory
        layers = max(2, int(avail // (2 * off["nbytes"])))
    host = []
    for _ in range(layers):
        h = torch.empty(off["nbytes"], dtype=torch.uint8).pin_memory()
        h.copy_(torch.from_numpy(img))
        host.append(h)
    slots = [torch.empty(off["nbytes"], dtype=torch.uint8, device=dev) for _ in range(2)]
    shape2 = tpk.Shape(H, impl=shape.impl, kv_slots=off["n_exact_pages"], rec_slots=off["n_int8_pages"],
                       int_query=shape.int_query)
    nbytes = tpk.hybrid_workspace_bytes(shape2, 1)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    outs = [(torch.empty(1, H * G, 256, dtype=torch.float32, device=dev),
             torch.empty(1, H * G, dtype=torch.float32, device=dev)) for _ in range(layers)]
    views = [slot_views(s, off, w) for s in slots]
    ne = off["n_exact_pages"]
    if lossless:  # BF16 scratch pool the staged records are unpacked into, reused layer after layer
        k13 = torch.empty(max(ne, 1) * H * 64 * 256, dtype=torch.int16, device=dev)
        v13 = torch.empty_like(k13)
        p13 = [(sl[off["p13"]:off["p13"] + off["p13_bytes"]], sl[off["p13off"]:off["p13off"] + 8 * ne * H])
               for sl in slots]
    st = tpk.Stager(slots, off["nbytes"])

    def one_step():
        pending = st.stage([(host[0], 0, off["nbytes"])])
        for l in range(layers):
            nxt = st.stage([(host[l + 1], 0, off["nbytes"])]) if l + 1 < layers else None
            slot, _ = pending
            st.acquire(slot, stream)
            rec, k, v, q, pt, pt8 = views[slot]
            if lossless:
                tpk.kv_unpack13_pages(shape2, p13[slot][0], off["p13_bytes"], p13[slot][1], pt, ne, k13, v13,
                                      stream)
                k, v = k13, v13
            tpk.decode_hybrid_batched(shape2, 1, q, k, v, rec, pt, off["req_page_off"], w.n_ex, pt8,
                                      off["req_page_off8"], w.n8, outs[l][0], outs[l][1], ws, nbytes, stream)
            st.release(slot, stream)
            pending = nxt

    try:
        with torch.cuda.stream(stream):
            one_step()
            stream.synchronize()
            times = []
            for _ in range(steps):
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                ev[0].record(stream)
                ev[0].synchronize()
                one_step()
                ev[1].record(stream)
                stream.synchronize()
                times.append(ev[0].elapsed_time(ev[1]))
            # link peak: one plain pinned host->device copy of 1 GiB
            big_h = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
            big_d = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
            best = 0.0
            for _ in range(3):
                e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                e[0].record(stream)
                big_d.copy_(big_h, non_blocking=True)
                e[1].record(stream)
                stream.synchronize()
                best = max(best, (1 << 30) / (e[0].elapsed_time(e[1]) * 1e-3) / 1e9)
            del big_h, big_d
    finally:
        st.close()
    status, flags = tpk.get_device_status(reset=True, stream=stream)
    if status != 0:
        raise RuntimeError(f"device status {status} flags {flags} (host-resident)")
    ms = statistics.median(times)
    ms = max_over_ranks(dist, ms)
    link = layers * off["nbytes"] / (ms * 1e-3) / 1e9
    return {"layers": layers, "ms_per_step": round(ms, 3), "steps": len(times),
            "h2d_bytes_per_step": int(layers * off["nbytes"]),
            "link_GBps": round(link, 1), "link_peak_GBps": round(best, 1), "link_frac": round(link / best, 4),
            "history_GBps": round(layers * w.history_bytes() / (ms * 1e-3) / 1e9, 1),
            "slots": 2, "slot_bytes": int(off["nbytes"]),
            "workload": label or f"{layers} layers x the 128K hybrid history (one pinned host image per layer)"}


def measure_link(stream, dev, sizes_mb=(1, 4, 16, 64, 256), reps=3):
    """Copies through the stager (pinned host -> device slot), timed on the device
    between the stager's own events around each staging: (bytes, us) samples and
    the fitted transfer model latency + bytes / rate."""
    import torch

    import tiered_paged_kv_gb300 as tpk
    from tiered_paged_kv_gb300 import gate

    top = max(sizes_mb) << 20
    host = torch.empty(top, dtype=torch.uint8).pin_memory()
    host.fill_(1)
    slots = [torch.empty(top, dtype=torch.uint8, device=dev) for _ in range(2)]
    samples = []
    with tpk.Stager(slots, top) as st:
        for mb in sizes_mb:
            for r in range(reps + 1):
                slot, _ = st.stage([(host, 0, mb << 20)])
                ms = st.copy_ms(slot)
                st.acquire(slot, stream)
                st.release(slot, stream)
                if r > 0:  # the first copy of each size warms up
                    samples.append((mb << 20, ms * 1e3))
        st.sync()
    stream.synchronize()
    del host, slots
    return gate.fit_link(samples), samples


def run_gate(args, stream, dev, flush, flush_r, sizes, layers_measured=4, layers_model=16):
    """The economic gate at each history size: three candidate formats of one
    request's history (4 KV heads x 8 q rows, outlier keys, seed 20) -- exact (all
    BF16), the 8-bit hybrid (4096 recent BF16 tokens, older pages 8-bit) and the
    lossless 13-bit tier (all pages 13-bit, unpacked on the device each step) --
    each described by the bytes its history image moves over the host link per
    layer and step and by its device time (kernels per step, graph replays with L2
    flushed, plus its page conversion amortised over a page's 64 tokens).  Verdict:
    accept when the transfer time saved per token (at layers_model layers, with
    the link model fitted to measured stager copies) exceeds the GPU time added.
    The model's host-resident step (layers_measured layers staged through two
    slots) is printed beside the measured one."""
    import dataclasses

    import torch

    import tiered_paged_kv_gb300 as tpk
    from tiered_paged_kv_gb300 import gate
    from tiered_paged_kv_gb300 import synth

    link, samples = measure_link(stream, dev)
    R = tpk.PACK13_RECORD_BYTES
    rows = []
    for n in sizes:
        w = synth.make_workload([n], 4096, H=4, seed=20, key_sigma="outliers")
        we = dataclasses.replace(w, n8=np.zeros_like(w.n8), n_ex=w.n_tokens.copy())
        H, G = w.H, w.G
        shape = tpk.Shape(H, kv_slots=w.n_slots, rec_slots=w.n_slots)
        ex_all, off_all = we.exact_page_table()
        ne_all = len(ex_all)
        with torch.cuda.stream(stream):
            kp = torch.from_numpy(w.k_pool.view(np.int16)).to(dev)
            vp = torch.from_numpy(w.v_pool.view(np.int16)).to(dev)
            q = torch.from_numpy(w.q.view(np.int16)).to(dev)
            rec = torch.zeros(w.n_slots * H * tpk.RECORD_BYTES, dtype=torch.uint8, device=dev)
            s8 = torch.from_numpy(w.int8_slots()).to(dev)
            n8 = len(w.int8_slots())
            pool13 = torch.zeros(w.n_slots * H * R, dtype=torch.uint8, device=dev)
            ex_d = torch.from_numpy(ex_all.astype(np.int32)).to(dev)
            offs = (np.repeat(ex_all.astype(np.int64), H) * H + np.tile(np.arange(H), ne_all)) * R
            offs_d = torch.from_numpy(offs).to(dev)
            k2, v2 = torch.zeros_like(kp), torch.zeros_like(vp)
            o = torch.empty(1, H * G, 256, dtype=torch.float32, device=dev)
            lse = torch.empty(1, H * G, dtype=torch.float32, device=dev)
            nbytes = tpk.hybrid_workspace_bytes(shape, 1)
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            pt_e = torch.from_numpy(np.concatenate([ex_all.astype(np.int32), np.zeros(1, np.int32)])).to(dev)
            pth, offh = w.exact_page_table()
            pt8h, off8h = w.int8_page_table()
            pt_h = torch.from_numpy(np.concatenate([pth, np.zeros(1, np.int32)])).to(dev)
            pt8_h = torch.from_numpy(np.concatenate([pt8h, np.zeros(1, np.int32)])).to(dev)
            zeros8 = np.zeros(2, np.int32)
            pt8_none = torch.zeros(1, dtype=torch.int32, device=dev)

        def timed_once(fn, reps=5):
            ev = []
            with torch.cuda.stream(stream):
                fn()
                for i in range(reps):
                    flush.fill_(float(i))
                    flush_r.max()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    fn()
                    b.record(stream)
                    ev.append((a, b))
                stream.synchronize()
            return statistics.median([a.elapsed_time(b) for a, b in ev]) * 1e3

        conv_us = timed_once(lambda: tpk.kv_quantize_pages(shape, kp, vp, s8, s8, n8, rec, stream))
        pack_us = timed_once(lambda: tpk.kv_pack13_pages(shape, kp, vp, ex_d, ex_d, ne_all, pool13, w.n_slots,
                                                         stream))

        def dec_exact(k=kp, v=vp):
            tpk.decode_hybrid_batched(shape, 1, q, k, v, rec, pt_e, off_all, we.n_ex, pt8_none, zeros8, we.n8, o,
                                      lse, ws, nbytes, stream)

        def dec_hybrid():
            tpk.decode_hybrid_batched(shape, 1, q, kp, vp, rec, pt_h, offh, w.n_ex, pt8_h, off8h, w.n8, o, lse, ws,
                                      nbytes, stream)

        def dec_13():
            tpk.kv_unpack13_pages(shape, pool13, pool13.numel(), offs_d, ex_d, ne_all, k2, v2, stream)
            dec_exact(k2, v2)

        dev_us = {"exact": statistics.median(graph_times(dec_exact, 20, 3, stream, flush, flush_r)) * 1e3,
                  "hybrid": statistics.median(graph_times(dec_hybrid, 20, 3, stream, flush, flush_r)) * 1e3,
                  "lossless": statistics.median(graph_times(dec_13, 20, 3, stream, flush, flush_r)) * 1e3}
        st, flags = tpk.get_device_status(reset=True, stream=stream)
        if st != 0:
            raise RuntimeError(f"device status {st} flags {flags} (gate {n})")
        # page conversion, amortised: one page of each head converts once per 64 tokens
        amort = {"exact": 0.0, "hybrid": conv_us / max(n8, 1) / 64.0,
                 "lossless": pack_us / max(ne_all, 1) / 64.0}
        hr = {"exact": run_host_resident(args, we, rec, shape, stream, dev, None, layers=layers_measured, steps=3,
                                         label=f"{layers_measured} layers x {n} tokens exact"),
              "hybrid": run_host_resident(args, w, rec, shape, stream, dev, None, layers=layers_measured, steps=3,
                                          label=f"{layers_measured} layers x {n} tokens hybrid"),
              "lossless": run_host_resident(args, we, rec, shape, stream, dev, None, layers=layers_measured,
                                            steps=3, label=f"{layers_measured} layers x {n} tokens 13-bit",
                                            pack13_dev=pool13)}
        cands = {k: gate.Candidate(k, hr[k]["slot_bytes"], dev_us[k] + amort[k]) for k in dev_us}
        row = {"tokens": n}
        for k, c in cands.items():
            step_only = gate.Candidate(k, c.link_bytes, dev_us[k])
            pred = gate.predict_step_us(link, step_only, layers_measured) * 1e-3
            meas = hr[k]["ms_per_step"]
            row[k] = {"link_bytes_per_layer": int(c.link_bytes), "device_us": round(dev_us[k], 2),
                      "conversion_us_per_token": round(amort[k], 4),
                      f"host_ms_{layers_measured}_layers": {"predicted": round(pred, 4), "measured": round(meas, 4),
                                                            "rel_err": round(pred / meas - 1.0, 4)}}
            if k != "exact":
                net = gate.net_saving_us(link, cands["exact"], c, layers=layers_model)
                row[k][f"net_saving_us_per_token_{layers_model}_layers"] = round(net, 2)
                row[k]["verdict"] = "accept" if gate.accept(link, cands["exact"], c, layers=layers_model) else "reject"
                row[k]["device_time_ratio"] = round(c.device_us / cands["exact"].device_us, 4)
                # history resident in HBM instead: no link to save on, the device time decides
                row[k]["device_resident_verdict"] = "accept" if c.device_us < cands["exact"].device_us else "reject"
        rows.append(row)
        print(json.dumps(row), flush=True, file=sys.stderr)
        del kp, vp, q, rec, pool13, k2, v2, ws
        torch.cuda.empty_cache()
    return {"link": {"latency_us": round(link.latency_us, 2), "rate_GBps": round(link.rate_GBps, 2),
                     "samples": len(samples), "copy_MB": sorted({int(b) >> 20 for b, _ in samples}),
                     "how": "least-squares line through stager copies timed on the device (tpk_stager_copy_ms)"},
            "rule": f"accept when (bytes saved per layer x {layers_model} layers) / link rate exceeds the device "
                    f"time added per token (decode and unpack per step, page conversion per 64 tokens)",
            "workload": "1 request, 4 KV heads x 8 q rows, head_dim 256, outlier keys, seed 20; hybrid: 4096 "
                        "recent BF16 tokens",
            "rows": rows}


def run_gate_sweep(args):
    """The economic gate over history lengths (--gate-lengths), printed as one
    JSON line: per size the candidates' bytes, device times, net saving per token
    and verdict, and the model's host-resident step beside the measured one."""
    import torch

    from tiered_paged_kv_gb300 import build as tbuild

    torch.cuda.set_device(0)
    tbuild.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        flush_r = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    sizes = [int(x) for x in args.gate_lengths.split(",")]
    out = run_gate(args, stream, dev, flush, flush_r, sizes, layers_measured=args.gate_layers)
    print(json.dumps({"mode": "gate_sweep", **out}), flush=True)


def run_lossless(args):
    """The lossless 13-bit exact tier as a third candidate format for the gate: per
    history length, one request of all-BF16 history (4 KV heads x 8 q rows,
    outlier keys, seed 20).  Page packing and unpacking rates (median of 5, L2
    flushed), the device step unpack + decode against decode alone, and the
    host-resident step per layer with the exact tier staged as BF16 or as
    compacted 13-bit records (unpacked on the device before the decode)."""
    import torch

    import tiered_paged_kv_gb300 as tpk
    from tiered_paged_kv_gb300 import build as tbuild
    from tiered_paged_kv_gb300 import synth

    torch.cuda.set_device(0)
    tbuild.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    R = tpk.PACK13_RECORD_BYTES
    with torch.cuda.stream(stream):
        flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        flush_r = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    peak, _ = hbm_peak()

    def timed(fn, reps=5):
        ev = []
        with torch.cuda.stream(stream):
            fn()
            for i in range(reps):
                flush.fill_(float(i))
                flush_r.max()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                ev.append((a, b))
            stream.synchronize()
        return statistics.median([a.elapsed_time(b) for a, b in ev])

    rows = []
    for n in [int(x) for x in args.gate_lengths.split(",")]:
        w = synth.make_workload([n], None, H=4, seed=20, key_sigma="outliers")
        H, G = w.H, w.G
        shape = tpk.Shape(H, kv_slots=w.n_slots, rec_slots=w.n_slots)
        ex, off_e = w.exact_page_table()
        ne = len(ex)
        with torch.cuda.stream(stream):
            kp = torch.from_numpy(w.k_pool.view(np.int16)).to(dev)
            vp = torch.from_numpy(w.v_pool.view(np.int16)).to(dev)
            q = torch.from_numpy(w.q.view(np.int16)).to(dev)
            rec = torch.zeros(16, dtype=torch.uint8, device=dev)
            pool = torch.zeros(w.n_slots * H * R, dtype=torch.uint8, device=dev)
            k2 = torch.zeros_like(kp)
            v2 = torch.zeros_like(vp)
            ex_d = torch.from_numpy(ex.astype(np.int32)).to(dev)
            offs = (np.repeat(ex.astype(np.int64), H) * H + np.tile(np.arange(H), ne)) * R
            offs_d = torch.from_numpy(offs).to(dev)
            pt_d = torch.from_numpy(np.concatenate([ex.astype(np.int32), np.zeros(1, np.int32)])).to(dev)
            pt8_d = torch.zeros(1, dtype=torch.int32, device=dev)
            off8 = np.zeros(2, np.int32)
            o = torch.empty(1, H * G, 256, dtype=torch.float32, device=dev)
            lse = torch.empty(1, H * G, dtype=torch.float32, device=dev)
            nbytes = tpk.hybrid_workspace_bytes(shape, 1)
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

        def pack():
            tpk.kv_pack13_pages(shape, kp, vp, ex_d, ex_d, ne, pool, w.n_slots, stream)

        def unpack():
            tpk.kv_unpack13_pages(shape, pool, pool.numel(), offs_d, ex_d, ne, k2, v2, stream)

        def decode(k, v):
            tpk.decode_hybrid_batched(shape, 1, q, k, v, rec, pt_d, off_e, w.n_ex, pt8_d, off8, w.n8, o, lse, ws,
                                      nbytes, stream)

        pack_ms = timed(pack)
        host = pool.cpu().numpy().reshape(w.n_slots, H, R)
        sizes = [16 + int(host[s, h, 0:4].view(np.uint32)[0]) + int(host[s, h, 4:8].view(np.uint32)[0])
                 for s in ex for h in range(H)]
        compact = int(sum((z + 15) & ~15 for z in sizes))
        bf16 = ne * H * 65536
        unpack_ms = timed(unpack)
        dec_ms = statistics.median(graph_times(lambda: decode(kp, vp), 20, 3, stream, flush, flush_r))
        both_ms = statistics.median(graph_times(lambda: (unpack(), decode(k2, v2)), 20, 3, stream, flush,
                                                flush_r))
        st, flags = tpk.get_device_status(reset=True, stream=stream)
        if st != 0:
            raise RuntimeError(f"device status {st} flags {flags} (lossless {n})")
        hr_bf16 = run_host_resident(args, w, rec, shape, stream, dev, None, layers=args.gate_layers, steps=3,
                                    label=f"{args.gate_layers} layers x {n} tokens BF16")
        hr_13 = run_host_resident(args, w, rec, shape, stream, dev, None, layers=args.gate_layers, steps=3,
                                  label=f"{args.gate_layers} layers x {n} tokens 13-bit", pack13_dev=pool)
        row = {"tokens": n, "bf16_bytes": bf16, "pack13_bytes": compact, "saving": round(1 - compact / bf16, 4),
               "planes_raw": int(sum((z - 16 - 2 * 26656) // (32768 - 26656) for z in sizes)),
               "pack_us": round(pack_ms * 1e3, 1),
               "pack_GBps": round((bf16 + compact) / (pack_ms * 1e-3) / 1e9, 1),
               "unpack_us": round(unpack_ms * 1e3, 1),
               "unpack_GBps": round((bf16 + compact) / (unpack_ms * 1e-3) / 1e9, 1),
               "hbm_peak_GBps": peak,
               "device_decode_us": round(dec_ms * 1e3, 2), "device_unpack_decode_us": round(both_ms * 1e3, 2),
               "host_ms_per_layer_bf16": round(hr_bf16["ms_per_step"] / hr_bf16["layers"], 4),
               "host_ms_per_layer_13bit": round(hr_13["ms_per_step"] / hr_13["layers"], 4),
               "link_GBps_bf16": hr_bf16["link_GBps"], "link_GBps_13bit": hr_13["link_GBps"],
               "link_peak_GBps": hr_13["link_peak_GBps"]}
        row["host_speedup"] = round(row["host_ms_per_layer_bf16"] / row["host_ms_per_layer_13bit"], 3)
        rows.append(row)
        print(json.dumps(row), flush=True, file=sys.stderr)
        del kp, vp, q, pool, k2, v2, ws
    print(json.dumps({"mode": "lossless_gate", "rows": rows}), flush=True)


def run_tiers_loop(args):
    """Decode loop with incremental conversion and publication: 16 requests of
    32,768 tokens grow by one token per step for `--tiers-steps` steps (recent
    window 2048 tokens, 4 KV heads x 8 q rows, outlier keys); per step the tier
    manager publishes finished conversions, starts new ones on a side stream and
    uploads the page tables, then the multi-request decode runs.  Compared with the
    same loop on fixed tables (no conversion, no upload); wall time per step with
    the host driving both streams, pages converted in the background reported."""
    import torch

    import tiered_paged_kv_gb300 as tpk
    from tiered_paged_kv_gb300 import build as tbuild
    from tiered_paged_kv_gb300 import synth

    torch.cuda.set_device(0)
    tbuild.build()
    dev = torch.device("cuda", 0)
    B, n0, steps, recent = 16, 32768, args.tiers_steps, 2048
    final = n0 + steps
    w = synth.make_workload([final] * B, None, H=4, seed=30, key_sigma="outliers")
    H, G = w.H, w.G
    max_pages = max(len(p) for p in w.pages)
    shape = tpk.Shape(H, kv_slots=w.n_slots, rec_slots=w.n_slots)
    dec, conv = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    with torch.cuda.stream(dec):
        kp = torch.from_numpy(w.k_pool.view(np.int16)).to(dev)
        vp = torch.from_numpy(w.v_pool.view(np.int16)).to(dev)
        q = torch.from_numpy(w.q.view(np.int16)).to(dev)
        rec = torch.zeros(w.n_slots * H * tpk.RECORD_BYTES, dtype=torch.uint8, device=dev)
        o = torch.empty(B, H * G, 256, dtype=torch.float32, device=dev)
        lse = torch.empty(B, H * G, dtype=torch.float32, device=dev)
        ws_bytes = tpk.hybrid_workspace_bytes(shape, B)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        sc_bytes = tpk.Tiers.device_bytes(B, max_pages)
        scratch = torch.empty(sc_bytes, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    result = {}
    with tpk.Tiers(shape, B, max_pages, recent, kp, vp, rec, scratch, sc_bytes) as tiers:
        # warm state: the starting histories fully converted and published
        for b in range(B):
            tiers.update(b, n0, w.pages[b][: (n0 + 63) // 64])
        tiers.step(conv, dec)
        tiers.sync()
        plan = tiers.step(conv, dec)
        tiers.sync()
        dec.synchronize()
        # the reference loop's fixed tables: the starting split (every eligible page 8-bit)
        n8_0 = (n0 - recent) // 64
        pt_h = np.concatenate([np.asarray(w.pages[b][n8_0:(n0 + 63) // 64]) for b in range(B)]).astype(np.int32)
        pt8_h = np.concatenate([np.asarray(w.pages[b][:n8_0]) for b in range(B)]).astype(np.int32)
        pt_fixed = torch.from_numpy(pt_h).to(dev)
        pt8_fixed = torch.from_numpy(pt8_h).to(dev)
        fixed = {"req_page_off": np.arange(B + 1, dtype=np.int32) * ((n0 + 63) // 64 - n8_0),
                 "req_page_off8": np.arange(B + 1, dtype=np.int32) * n8_0,
                 "n_exact_tokens": np.full(B, n0 - 64 * n8_0, np.int32), "n_int8_pages": np.full(B, n8_0, np.int32)}
        assert list(plan["n_int8_pages"]) == [n8_0] * B
        for mode in ("fixed tables", "tier manager"):
            n = n0
            published = started = 0
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for step in range(steps):
                n += 1
                if mode == "tier manager":
                    for b in range(B):
                        tiers.update(b, n, w.pages[b][: (n + 63) // 64])
                    pl = tiers.step(conv, dec)
                    published += pl["published"]
                    started += pl["started"]
                    tpk.decode_hybrid_batched(shape, B, q, kp, vp, rec, pl["page_table"], pl["req_page_off"],
                                              pl["n_exact_tokens"], pl["page_table8"], pl["req_page_off8"],
                                              pl["n_int8_pages"], o, lse, ws, ws_bytes, dec)
                else:
                    tpk.decode_hybrid_batched(shape, B, q, kp, vp, rec, pt_fixed, fixed["req_page_off"],
                                              fixed["n_exact_tokens"], pt8_fixed, fixed["req_page_off8"],
                                              fixed["n_int8_pages"], o, lse, ws, ws_bytes, dec)
            torch.cuda.synchronize()
            dt = (time.perf_counter() - t0) / steps
            result[mode] = {"us_per_step": round(dt * 1e6, 1), "pages_started": started,
                            "pages_published": published}
    out = {"mode": "tiers_loop", "requests": B, "start_tokens": n0, "steps": steps, "recent_tokens": recent,
           **result}
    out["overhead_us_per_step"] = round(result["tier manager"]["us_per_step"] - result["fixed tables"]["us_per_step"], 1)
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------- reference arm
def run_reference(args, dist, rank, world):
    """The CPU oracle as the reference arm, on the same workload as the GPU arm:
    each timed step is the oracle's whole 128K hybrid step (all KV heads, over
    pre-converted records) with its (request, KV head, query row) items spread
    over every core of the affinity set."""
    if rank != 0:
        return
    import oracle
    from tiered_paged_kv_gb300 import synth

    oracle.build()
    synth.build()
    w = build_workload()
    rec = np.zeros(w.n_slots * w.H * oracle.REC_BYTES, np.uint8)
    s = w.int8_slots()
    oracle.quantize_pages(w.H, w.k_pool, w.v_pool, s, s, rec)
    n_thr = host_cores()
    for _ in range(args.warmup):
        oracle.hybrid_workload(w, rec, n_threads=n_thr)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.hybrid_workload(w, rec, n_threads=n_thr)
        times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    value = w.history_bytes() / sec / 1e9
    cores = min(n_thr, w.B * w.H * w.G)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": "the whole 128K hybrid step (all 4 KV heads) per timed step"},
            "cpu_baseline": {"kind": "oracle", "cores": cores, "value": round(value, 4), "unit": "GB/s",
                             "sample": f"the whole 128K hybrid step per timed step, (request, KV head, query row) "
                                       f"items on {cores} threads"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="tpk", choices=["tpk", "reference"])
    ap.add_argument("--kernel", default="default", choices=["default", "simt", "tensor"])
    ap.add_argument("--int-query", action="store_true",
                    help="time the integer-query variant of the 8-bit tier as the main step")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of back-to-back steps before timing")
    ap.add_argument("--layers", type=int, default=16, help="layers of the host-resident measurement (0: skip)")
    ap.add_argument("--host-steps", type=int, default=5, help="timed steps of the host-resident measurement")
    ap.add_argument("--tier-steps", type=int, default=20, help="timed steps of each single-tier 128K line (0: skip)")
    ap.add_argument("--gate-sweep", action="store_true",
                    help="instead of the bench line: exact vs hybrid over history lengths (device and host-resident)")
    ap.add_argument("--gate-lengths", default="8192,16384,32768,65536,131072")
    ap.add_argument("--lossless", action="store_true",
                    help="lossless 13-bit exact tier against BF16 over --gate-lengths (pack, unpack, device and "
                         "host-resident steps)")
    ap.add_argument("--gate-layers", type=int, default=4)
    ap.add_argument("--no-gate", dest="gate", action="store_false",
                    help="skip the economic gate at 32K, 64K and 128K in the bench line")
    ap.add_argument("--tiers-loop", action="store_true",
                    help="instead of the bench line: a decode loop with incremental conversion and publication")
    ap.add_argument("--tiers-steps", type=int, default=256)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "tpk":
        args.warmup = 3
    dist, rank, world = dist_init()
    try:
        if args.impl == "reference":
            run_reference(args, dist, rank, world)
        elif args.gate_sweep:
            run_gate_sweep(args)
        elif args.lossless:
            run_lossless(args)
        elif args.tiers_loop:
            run_tiers_loop(args)
        else:
            run_gpu(args, dist, rank, world)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
