"""Worst merged error of the hybrid tier against unquantised attention, computed
with the oracle alone (the page conversion, the hybrid step and the full-precision
reference are all oracle functions).  Prints one line per workload.

    python oracle/hybrid_error_report.py [--full]

Each workload is reported twice: with the query in floating point, and with the
integer-query variant ("SYCL", "Attention that reads 8-bit history": the query
folded with each page's channel scales coded to 8 bits per page and row).

The pages' quality bound is 0.005 on the worst merged error ("model
quantization": a fixed loss bound against the format's own higher-precision
reference); this reports max |o_hybrid - o_fp| over all rows and channels, the
same over max |o_fp|, and the RMS error over the RMS output.
"""
import argparse
import os
import sys
import time

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import oracle  # noqa: E402
from tiered_paged_kv_gb300 import synth  # noqa: E402


def report(name, w, threads):
    t0 = time.time()
    rec = np.zeros(w.n_slots * w.H * oracle.REC_BYTES, np.uint8)
    s = w.int8_slots()
    oracle.quantize_pages(w.H, w.k_pool, w.v_pool, s, s, rec)
    of, _ = oracle.full_precision_workload(w, n_threads=threads)
    for query in ("float", "integer"):
        oh, _ = oracle.hybrid_workload(w, rec, n_threads=threads, int_query=query == "integer")
        err = np.abs(oh - of)
        print(f"{name:34s} {query:7s} query  max_abs {err.max():.5f}  max_abs/max|o| "
              f"{err.max() / np.abs(of).max():.5f}  rms_rel {np.sqrt((err ** 2).mean() / (of ** 2).mean()):.5f}  "
              f"max|o| {np.abs(of).max():.4f}  bound 0.005 {'met' if err.max() <= 0.005 else 'exceeded'}  "
              f"({time.time() - t0:.1f} s)", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--full", action="store_true", help="also the 128K and 16-request workloads")
    args = ap.parse_args()
    th = os.cpu_count() or 1
    for seed in range(3):
        report(f"tiny hybrid (1024 tok) seed {seed}", synth.tiny_hybrid(seed=seed), th)
    report("128K shape at 16K tokens, unit keys", synth.make_workload([16384], 4096, H=4, seed=2), th)
    report("128K shape at 16K tokens, outliers", synth.hybrid_128k(seed=2, n_tokens=16384), th)
    if args.full:
        for seed in (2, 3):
            report(f"hybrid 128K seed {seed}", synth.hybrid_128k(seed=seed), th)
        report("batched 16 requests seed 3", synth.batched_hybrid(seed=3), th)


if __name__ == "__main__":
    main()
