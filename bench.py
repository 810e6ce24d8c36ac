#!/usr/bin/env python3
"""Benchmark of the paged latent-cache attention path on GB300.

One step is one pass of the whole path over one batch of synthetic input that
is already resident in HBM: per cache, append each stream's current rows
(tf_paged_append) and attend over its pages (tf_paged_mla_attend); for the
full-model workload, then copy a kept state's first `at` rows
(tf_state_copy_rows).  The default workload is the decode batch (8 streams,
64 heads, lengths U[4,096, 65,536], streams 0-3 sharing 16 pages).

Prints ONE JSON line (rank 0).  With --gpus N > 1 (torchrun), every rank runs an
independent replica of the workload on its own GPU ("replicas only": the path
has no exchange step), value = the units of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
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

WORKLOADS = ["decode_batch", "tiny_decode", "long_window", "prefill_100k", "prefill_208k", "full_model",
             "sparse_decode", "fp8_decode", "sparse_fp8_decode", "topk_prefill"]
TOPK = {"topk_prefill"}
METRIC = "paged MLA decode KV GB/s + tokens/s vs HBM roofline; prefill TFLOP/s"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=WORKLOADS, default="decode_batch")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the short runs of the other workloads reported under 'workloads'")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The slowest rank's time: every rank gets the maximum of `value` over the group."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, slowest_ms: float) -> float:
    """Units of all ranks (replicas of the same workload) over the slowest rank's time, per second."""
    return world * units_per_rank / (slowest_ms / 1e3)


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the dominant
# kernel, from the ncu captures summarised in profiles/, keyed by the first 16 hex digits of
# the SHA-256 of the kernel's source the capture was taken on: once the kernel changes, the
# counters no longer describe it and "traffic" is reported null until it is re-captured.
NCU_TRAFFIC = {
    # attention on source 7d9fa675422c97da, one launch each: `--metrics dram__bytes_read.sum,
    # dram__bytes_write.sum,gpu__time_duration.sum --cache-control none` (L2 as the back-to-back
    # steps leave it); the prefill chunk with ncu's default cache flush; profiles/mla_attend_*.md.
    # e00360dc80e0534f differs from it only in how many columns a CTA's last cut partial stages (those PV
    # computed, in 32-column steps): all 64 for every workload below, so the same bytes move.
    "e00360dc80e0534f": {"decode_batch": 370_056_704 + 2_340_864,
                         "long_window": 1_207_117_312 + 827_392,
                         "sparse_decode": 155_352_064 + 22_679_040,
                         "fp8_decode": 216_005_888 + 17_167_104,
                         "prefill_100k": 20_034_719_744 + 158_304_512},
    # top-k: both launches of one call (first level 811.1 + 8.6 MB, merge 58.8 + 0.2 MB), taken
    # on source 4e5c0b41cdefdfb7; 689a485f4717fede differs from it in comments and host-side argument
    # checks only (the cubins built without line info hash the same)
    "689a485f4717fede": {"topk_prefill": 811_079_680 + 8_606_208 + 58_786_560 + 240_640},
}


def ncu_traffic(workload: str, source: str = "attend.cu"):
    import hashlib
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "paged_mla_kv_gb300", "csrc", source)
    try:
        key = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    return NCU_TRAFFIC.get(key, {}).get(workload)


def read_kernel_times(pool) -> dict:
    """(total ms, launches) of each launch kind the library recorded while the pool's profiling
    was on (CUDA events around each launch, on its stream); reading clears the records."""
    from paged_mla_kv_gb300 import binding as B
    kinds = {"append": B.PROF_APPEND, "attend": B.PROF_ATTEND, "combine": B.PROF_COMBINE,
             "state_copy": B.PROF_COPY, "poison": B.PROF_POISON}
    return {name: pool.profile_read(kind) for name, kind in kinds.items()}


def kernels_per_step(times: dict, steps: int) -> dict:
    """Device ms and launches a step of every launch kind that ran."""
    return {name: {"ms": t / steps, "launches": n / steps} for name, (t, n) in times.items() if n}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def make_workload(name):
    from paged_mla_kv_gb300 import synth as Y
    return Y.WORKLOADS[name]()


def step_units(w):
    """Algorithmic work of one step: bytes, flops, tokens."""
    from paged_mla_kv_gb300 import synth as Y
    S, R, H, C = w.S, w.R, w.H, w.num_caches
    # an FP8 row is 512 code bytes, a 4-byte scale and the 128-byte bf16 rope
    row = 644 if w.extra.get("fp8") else Y.ROW_BYTES
    if "nidx" in w.extra:
        # attention over listed rows: each stream reads its listed rows once for all heads
        n = [min(int(w.extra["nidx"]), int(L)) for L in w.lens]
        kv = sum(n) * row
        q = S * H * Y.DK * 2
        out = S * H * (512 * 2 + 4)
        app = S * (Y.ROW_BYTES + row)
        flops = 2 * (Y.DK + 512) * H * sum(n)
        return dict(bytes=kv + q + out + app, attend_bytes=kv + q + out, flops=flops, attend_flops=flops,
                    tokens=S, kv=kv)
    kv = int(np.sum(w.lens)) * row
    # the same rows with each shared prefix page counted once (what the pool holds)
    unique_kv = sum(int(w.lens[s]) - w.shared_pages(s) * Y.PAGE_ROWS for s in range(S)) * row
    q = S * R * H * Y.DK * 2
    out = S * R * H * (512 * 2 + 4)
    app = S * R * (Y.ROW_BYTES + row)
    attend_bytes = kv + q + out
    at = int(w.extra.get("at", 0))
    copy = 2 * at * Y.ROW_BYTES * C
    pairs = 0
    for s in range(S):
        L = int(w.lens[s])
        pairs += sum(L - R + r + 1 for r in range(R)) if R <= 4096 else 0
    flops = 2 * (Y.DK + 512) * H * pairs * C
    return dict(bytes=C * (attend_bytes + app) + copy, attend_bytes=attend_bytes, flops=flops,
                attend_flops=flops // C, tokens=S * R if R <= 2 else S * R, kv=kv, unique_kv=unique_kv)


def topk_bytes(w) -> int:
    """Algorithmic bytes of one blocked top-k call: the logits in play read once (4 bytes a key),
    each row's k columns and values written once (8 bytes a pair)."""
    return 4 * int(np.sum(w.lens)) + 8 * w.rows * w.k


class ClockSampler:
    def __init__(self, index: int):
        self.index, self.rows, self.proc, self.th = index, [], None, None

    def start(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return

        def rd():
            for line in self.proc.stdout:
                self.rows.append([x.strip() for x in line.split(",")])
        self.th = threading.Thread(target=rd, daemon=True)
        self.th.start()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
            except (ValueError, IndexError):
                pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


class OracleSample:
    """The oracle, as it stands, timed on a bounded sample of the workload.

    The workload is cut into items, one (stream, query row, head) each, and the sample is the
    k cheapest items (a stream's items in head order; ties in stream, row, head order).  The
    rate is the sample's work over its time: in KV GB/s for decode (a stream's key rows count
    once for all its heads and rows, so an item carries 1/(R*H) of them; for listed rows the
    listed rows), in TFLOP/s of causal (row, key) pairs for a prefill chunk.  k is calibrated
    once so that a sample takes about `seconds` on the host cores; the smallest sample is one
    item, so a step can be made as short as the run's number of steps needs."""

    def __init__(self, w, seconds: float):
        from oracle import attend as OA
        self.OA, self.w = OA, w
        self.threads = os.cpu_count() or 1
        self.prefill = w.R > 2
        self.q = w.q(0)
        self.rows = [w.stream_rows(0, s) for s in range(w.S)]
        self.row_bytes = 1152
        self.lists = None
        if "nidx" in w.extra:
            from paged_mla_kv_gb300 import synth as Y
            self.lists = Y.listed_rows(w.seed, w.lens, int(w.extra["nidx"]))
            # only the listed rows are read: keep those, and list positions into them
            self.rows = [(a[x], b[x]) for (a, b), x in zip(self.rows, self.lists)]
            self.lists = [np.arange(len(x)) for x in self.lists]
        if w.extra.get("fp8"):   # the oracle attends over the rows as FP8 pages hold them
            from oracle import fp8 as F
            from paged_mla_kv_gb300 import synth as Y
            self.rows = [(F.dequantize_rows(*F.quantize_rows(Y.bf16_bits_to_f32(a))), b) for a, b in self.rows]
            self.row_bytes = 644
        # items (work, stream, row, head), cheapest first
        its = []
        for s in range(w.S):
            L = int(w.lens[s])
            for r in range(w.R):
                keys = len(self.lists[s]) if self.lists is not None else L - w.R + r + 1
                if self.prefill:
                    work = 2.0 * 1088 * keys
                else:
                    nrows = len(self.lists[s]) if self.lists is not None else L
                    work = nrows * self.row_bytes / (w.R * w.H)
                for h in range(w.H):
                    its.append((work, keys, s, r, h))
        its.sort(key=lambda x: (x[1], x[2], x[4], x[3]))
        self.its = [(wk, s, r, h) for wk, _, s, r, h in its]
        # calibrate on the cheapest items: the rate, then the longest prefix of items whose work
        # fits `seconds` at that rate (items differ in cost by the stream's length)
        k0 = min(len(self.its), max(1, self.threads))
        t0, w0 = self.run(k0)
        budget = w0 / max(t0, 1e-4) * seconds
        cum = np.cumsum([x[0] for x in self.its])
        self.k = int(max(1, min(len(self.its), np.searchsorted(cum, budget, side="right"))))

    def run(self, k):
        w = self.w
        chosen = self.its[:k]
        by_stream = {}
        for wk, s, r, h in chosen:
            by_stream.setdefault(s, []).append(r * w.H + h)
        t0 = time.perf_counter()
        for s, items in by_stream.items():
            if self.lists is not None:   # R = 1; a stream's items are its first heads
                self.OA.attend_sparse(self.q[s, 0, :len(items)], self.rows[s][0], self.rows[s][1], self.lists[s],
                                      w.scale, self.threads)
            else:
                self.OA.attend_stream(self.q[s], self.rows[s][0], self.rows[s][1], w.scale,
                                      np.array(items, np.int32), self.threads)
        return time.perf_counter() - t0, sum(x[0] for x in chosen)

    def measure(self):
        t, work = self.run(self.k)
        w = self.w
        streams = len({s for _, s, _, _ in self.its[:self.k]})
        cores = min(self.threads, max(1, self.k))
        what = (f"the {self.k} cheapest of {len(self.its)} (stream, row, head) items ({streams} of {w.S} streams"
                f"{', listed rows' if self.lists is not None else ''}), cache 0 ({t:.2f} s)")
        if self.prefill:
            return dict(value=work / t / 1e12, unit="TFLOP/s", cores=cores, kind="oracle", sample=what)
        return dict(value=work / t / 1e9, unit="GB/s", cores=cores, kind="oracle", sample=what)


class TopkOracleSample:
    """The top-k oracle, as it stands, on a bounded sample of rows spread over the chunk; the rate
    is in GB/s of logits scanned (4 bytes a key in play)."""

    def __init__(self, w, seconds: float):
        from oracle import topk as OT
        from paged_mla_kv_gb300 import synth as Y
        self.OT, self.Y, self.w = OT, Y, w
        t0, _ = self.run(2)
        self.n = int(max(1, min(w.rows, 2 * seconds / max(t0, 1e-3))))

    def rows(self, n):
        return np.unique(np.linspace(0, self.w.rows - 1, n).round().astype(int))

    def run(self, n):
        w = self.w
        rows = self.rows(n)
        x = self.Y.topk_logits(w.seed, rows, w.n)
        t0 = time.perf_counter()
        self.OT.topk_rows(x, w.k, w.lens[rows])
        return time.perf_counter() - t0, 4.0 * float(np.sum(w.lens[rows]))

    def measure(self):
        t, work = self.run(self.n)
        return dict(value=work / t / 1e9, unit="GB/s", cores=1, kind="oracle",
                    sample=f"{len(self.rows(self.n))} of {self.w.rows} rows spread over the chunk ({t:.1f} s, "
                           f"one numpy sort a row)")


REFERENCE_SECONDS = 150.0   # the reference arm's whole run, warm-up included, on the host cores


def reference_arm(args, rank, world):
    """The oracle timed as the reference arm (host cores, the same bounded sample each step)."""
    if rank != 0:
        return
    if args.workload in TOPK:
        from paged_mla_kv_gb300 import synth as Y
        w = Y.TOPK_WORKLOADS[args.workload]()
        o = TopkOracleSample(w, min(20.0, REFERENCE_SECONDS / max(1, args.steps + args.warmup)))
        for _ in range(args.warmup):
            o.run(o.n)
        vals = [o.measure() for _ in range(args.steps)]
        v = statistics.median(x["value"] for x in vals)
        scanned = 4.0 * float(np.sum(w.lens))   # the logits in play, the sample's unit of work
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": scanned / (v * 1e9) * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic",
                "config": {"workload": w.name, "rows": w.rows, "n": w.n, "k": w.k, "lens_sum": int(np.sum(w.lens)),
                           "parallelism": "one host core"},
                "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": vals[0]["sample"], "value": v},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    w = make_workload(args.workload)
    per_step = min(20.0, REFERENCE_SECONDS / max(1, args.steps + args.warmup))
    o = OracleSample(w, per_step)
    for _ in range(args.warmup):
        o.run(o.k)
    vals = [o.measure() for _ in range(args.steps)]
    v = statistics.median(x["value"] for x in vals)
    units = step_units(w)
    # ms_per_step: the whole workload's step at the sample's rate (flops of a prefill chunk; the
    # key rows of every cache for decode)
    if vals[0]["unit"] == "TFLOP/s":
        ms = units["flops"] / (v * 1e12) * 1e3
    else:
        ms = w.num_caches * units["kv"] / (v * 1e9) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": vals[0]["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "S": w.S, "R": w.R, "H": w.H, "caches": w.num_caches,
                       "lens_sum": int(np.sum(w.lens)), "kv_bytes": units["kv"], "tokens_per_step": units["tokens"],
                       "parallelism": f"host cores x{vals[0]['cores']}"},
            "cpu_baseline": {"kind": "oracle", "cores": vals[0]["cores"], "sample": vals[0]["sample"], "value": v},
            "e2e": {"value": v, "unit": vals[0]["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def topk_main(args, rank, world, pg, peaks, peak_src):
    """Blocked top-k over a prefill chunk's indexer logits: one step = one tf_topk_blocked call
    (a first-level launch and a merge launch) over the resident 2,048 x 100,000 fp32 matrix."""
    import torch
    from paged_mla_kv_gb300 import binding as B
    from paged_mla_kv_gb300 import synth as Y
    w = Y.TOPK_WORKLOADS[args.workload]()
    x = torch.from_numpy(Y.topk_logits(w.seed, range(w.rows), w.n)).cuda()
    lens = torch.from_numpy(w.lens).cuda()
    ws = torch.empty(max(B.tf_topk_workspace_bytes(w.rows, w.n, w.k), 16), dtype=torch.uint8, device="cuda")
    idx = torch.empty((w.rows, w.k), dtype=torch.int32, device="cuda")
    val = torch.empty((w.rows, w.k), dtype=torch.float32, device="cuda")
    algo = topk_bytes(w)

    def step(src=x, oi=idx, ov=val):
        B.tf_topk_blocked(src, w.k, oi, ov, lens=lens, ws=ws)

    def barrier():
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    barrier()
    n0 = B.tf_launch_count()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    barrier()
    launches = B.tf_launch_count() - n0
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, pg, "cuda")
    clocks = sampler.stop() if sampler else None
    value = whole_job_rate(algo, world, ms) / 1e9
    peak = peaks.get("hbm_gbs", 6800.0)
    achieved = algo / (ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": ncu_traffic(args.workload, "topk.cu"), "peak_kind": f"{peak_src} HBM copy",
            "kernel": "topk_level_kernel (both levels of one call)", "avg_launch_ms": ms}

    e2e = None
    if not args.no_e2e:
        hx = x.cpu().pin_memory()
        hi = torch.empty(idx.shape, dtype=idx.dtype).pin_memory()
        hv = torch.empty(val.shape, dtype=val.dtype).pin_memory()
        dx = torch.empty_like(x)
        for _ in range(max(2, args.warmup)):
            dx.copy_(hx, non_blocking=True)
            step(dx)
            hi.copy_(idx, non_blocking=True)
            hv.copy_(val, non_blocking=True)
        barrier()
        k_ = max(2, min(args.steps, 20))
        e0.record()
        for _ in range(k_):
            dx.copy_(hx, non_blocking=True)
            step(dx)
            hi.copy_(idx, non_blocking=True)
            hv.copy_(val, non_blocking=True)
        e1.record()
        barrier()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / k_, pg, "cuda")
        e2e = {"value": world * algo / 1e9 / (e_ms / 1e3), "unit": "GB/s", "h2d_bytes_per_step": x.numel() * 4,
               "d2h_bytes_per_step": idx.numel() * 4 + val.numel() * 4, "ms_per_step": e_ms}
    cpu = TopkOracleSample(w, args.cpu_seconds).measure() if rank == 0 and not args.no_cpu_baseline else None
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": w.name, "rows": w.rows, "n": w.n, "k": w.k, "lens_sum": int(np.sum(w.lens)),
                           "l2": "inputs larger than L2", "parallelism": f"replicas x{world}"},
                "gpu_launches": launches, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks}
        print(json.dumps(line), flush=True)


def measure(name, steps, warmup, with_e2e, pg, world, peaks, peak_src):
    """One workload on this GPU: `steps` timed steps after `warmup` (CUDA events; L2 flushed
    between steps when the inputs fit in it), each kernel kind's own duration in a second pass,
    the clocks over both, and, with `with_e2e`, the end-to-end step with host buffers."""
    import torch
    from paged_mla_kv_gb300 import binding as B
    from paged_mla_kv_gb300.harness import Resident
    rank = int(os.environ.get("RANK", "0"))
    w = make_workload(name)
    prefill = w.R > 2
    units = step_units(w)
    res = Resident(w, poison=True, fp8=bool(w.extra.get("fp8")))
    qs = [res.q(c) for c in range(w.num_caches)]
    cur = [res.current_rows(c) for c in range(w.num_caches)]
    out = torch.empty((w.S, w.R, w.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.S, w.R, w.H), dtype=torch.float32, device="cuda")
    ws = res.workspace()
    at = int(w.extra.get("at", 0))
    if at:
        pages = -(-at // 512)
        dst = torch.from_numpy(res.pool.take(pages)).cuda()
        src = torch.from_numpy(res.pt_host[0, :pages].copy()).cuda()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda") \
        if units["kv"] < 2 * L2_BYTES else None

    sparse = "nidx" in w.extra
    if sparse:
        from paged_mla_kv_gb300 import synth as Y
        lists = Y.listed_rows(w.seed, w.lens, int(w.extra["nidx"]))
        nidx = np.array([len(x) for x in lists], np.int32)
        idx_h = np.zeros((w.S, int(nidx.max())), np.int32)
        for s_, x in enumerate(lists):
            idx_h[s_, :len(x)] = x
        idx_d = torch.from_numpy(idx_h).cuda()
        nws = B.tf_paged_mla_sparse_workspace_bytes(res.pool, w.S, w.H, nidx)
        ws = torch.empty(max(nws, 256), dtype=torch.uint8, device="cuda") if nws else None

    def step(q_list=qs, rows=cur, o=out, l=lse):
        for c in range(w.num_caches):
            res.append_current(c, rows[c][0], rows[c][1])
            if sparse:
                B.tf_paged_mla_attend_sparse(res.pool, c, res.pt, res.max_pages, res.lens, idx_d, nidx, q_list[c],
                                             w.scale, o, l, ws)
            else:
                B.tf_paged_mla_attend(res.pool, c, res.pt, res.max_pages, res.lens, q_list[c], w.scale, o, l, ws)
        if at:
            B.tf_state_copy_rows(res.pool, -1, src, dst, at)

    def barrier():
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    for _ in range(warmup):
        step()
    barrier()
    n0 = B.tf_launch_count()
    barrier()
    if flush is None:
        # inputs larger than L2: K steps back to back between one pair of events
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(steps):
            step()
        e1.record()
        barrier()
        total_ms = e0.elapsed_time(e1)
    else:
        # L2 flushed between steps, outside each step's pair of events
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            ev[i][0].record()
            step()
            ev[i][1].record()
        barrier()
        total_ms = sum(a.elapsed_time(b) for a, b in ev)
    launches = B.tf_launch_count() - n0
    # each kernel's own duration (the attention's for the roofline; every kind for
    # "kernels_per_step"): CUDA events around each launch, on its stream, in a second pass of
    # the same steps (the events cost ~15 us a step and serialise the launches, so they stay
    # out of the timed region above, and the kinds' times may add up to more than a step)
    res.pool.profile(True)
    read_kernel_times(res.pool)
    nprof = min(steps, 200)
    for i in range(nprof):
        if flush is not None:
            flush.zero_()
        step()
    barrier()
    times = read_kernel_times(res.pool)
    att_ms, att_n = times["attend"]
    res.pool.profile(False)
    clocks = sampler.stop() if sampler else None
    rc, detail = res.pool.last_error()
    if rc != 0:
        raise SystemExit(f"device error {rc} ({detail})")
    total_ms = max_over_ranks(total_ms, pg, "cuda")
    ms = total_ms / steps
    if prefill:
        value = whole_job_rate(units["flops"], world, ms) / 1e12
        unit = "TFLOP/s"
    else:
        value = whole_job_rate(units["bytes"], world, ms) / 1e9
        unit = "GB/s"
    tokens_s = whole_job_rate(units["tokens"], world, ms)

    # roofline of the dominant kernel (the attention main pass), timed by events on its stream
    avg_att = att_ms / max(att_n, 1)
    if prefill:
        achieved = units["attend_flops"] / (avg_att / 1e3) / 1e12
        peak = peaks.get("bf16_tflops_sustained", 1700.0)
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": ncu_traffic(name), "peak_kind": f"{peak_src} bf16 sustained",
                "kernel": "mla_attend_kernel",
                "avg_launch_ms": avg_att}
    else:
        achieved = units["attend_bytes"] / (avg_att / 1e3) / 1e9
        peak = peaks.get("hbm_gbs", 6800.0)
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": ncu_traffic(name), "peak_kind": f"{peak_src} HBM copy",
                "kernel": ("mla_attend_kernel, FP8 instance (codes expanded in shared memory)"
                           if w.extra.get("fp8") else "mla_attend_kernel"),
                "avg_launch_ms": avg_att}

    # end to end through the C-ABI with host buffers: queries and new rows in, outputs out
    e2e = None
    if not not with_e2e:
        # one pinned host buffer and one device buffer a direction, so a step is one copy each way:
        # in = every cache's queries, then its new rows' latent and rope parts; out = the outputs,
        # then the lse (each part starts on a 256-byte boundary)
        def layout(ts):
            offs, n = [], 0
            for t in ts:
                offs.append(n)
                n += -(-t.numel() * t.element_size() // 256) * 256
            return offs, n

        def views(buf, ts, offs):
            return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(ts, offs)]

        ins = [t for c in range(w.num_caches) for t in (qs[c], cur[c][0], cur[c][1])]
        in_offs, in_n = layout(ins)
        outs = [out, lse]
        out_offs, out_n = layout(outs)
        nb = 2   # double buffers: step i+1's inputs and step i-1's outputs move while step i runs
        hin = torch.empty(in_n, dtype=torch.uint8).pin_memory()
        for t, v in zip(ins, views(hin, ins, in_offs)):
            v.copy_(t.cpu())
        din = [torch.empty(in_n, dtype=torch.uint8, device="cuda") for _ in range(nb)]
        dout_b = [torch.empty(out_n, dtype=torch.uint8, device="cuda") for _ in range(nb)]
        hout = [torch.empty(out_n, dtype=torch.uint8).pin_memory() for _ in range(nb)]
        dq, drows, dout, dlse = [], [], [], []
        for b_ in range(nb):
            v = views(din[b_], ins, in_offs)
            dq.append([v[3 * c] for c in range(w.num_caches)])
            drows.append([(v[3 * c + 1], v[3 * c + 2]) for c in range(w.num_caches)])
            o = views(dout_b[b_], outs, out_offs)
            dout.append(o[0])
            dlse.append(o[1])
        main = torch.cuda.current_stream()
        cs = torch.cuda.Stream()
        in_ready = [torch.cuda.Event() for _ in range(nb)]
        done = [torch.cuda.Event() for _ in range(nb)]
        out_read = [torch.cuda.Event() for _ in range(nb)]
        for b_ in range(nb):           # every event recorded once, so the first waits pass
            done[b_].record(main)
            out_read[b_].record(main)

        def h2d(i):
            b_ = i % nb
            cs.wait_event(done[b_])        # step i-2 has consumed this buffer
            din[b_].copy_(hin, non_blocking=True)
            in_ready[b_].record(cs)

        def compute(i):
            b_ = i % nb
            main.wait_event(in_ready[b_])
            main.wait_event(out_read[b_])      # step i-2's outputs have left this buffer
            step(dq[b_], drows[b_], dout[b_], dlse[b_])
            done[b_].record(main)

        def d2h(i):
            b_ = i % nb
            cs.wait_event(done[b_])
            hout[b_].copy_(dout_b[b_], non_blocking=True)
            out_read[b_].record(cs)

        def run_e2e(n):
            with torch.cuda.stream(cs):
                h2d(0)
            for i in range(n):
                compute(i)
                with torch.cuda.stream(cs):
                    if i + 1 < n:
                        h2d(i + 1)
                    d2h(i)
            main.wait_event(out_read[(n - 1) % nb])

        run_e2e(max(2, warmup))
        barrier()
        if flush is None:
            # inputs larger than L2: the steps run back to back, copies overlapped, one pair of events
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(main)
            run_e2e(steps)
            e1.record(main)
            barrier()
            e_ms = max_over_ranks(e0.elapsed_time(e1) / steps, pg, "cuda")
        else:
            # the L2 flush between steps stays outside the events: each step is copied in,
            # run and copied out on its own
            e2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            for i in range(steps):
                flush.zero_()
                e2[i][0].record(main)
                run_e2e(1)
                e2[i][1].record(main)
            barrier()
            e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2) / steps, pg, "cuda")
        h2d, d2h = in_n, out_n   # the bytes each step's two copies move (parts padded to 256 bytes)
        ev_ = world * (units["flops"] / 1e12 if prefill else units["bytes"] / 1e9) / (e_ms / 1e3)
        e2e = {"value": ev_, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}

    return dict(w=w, units=units, ms=ms, value=value, unit=unit, tokens_s=tokens_s, launches=launches, roof=roof,
                e2e=e2e, clocks=clocks, times=times, nprof=nprof, flush=flush is not None, prefill=prefill)


# The rest of the metric ("...; prefill TFLOP/s") in the same run: short in-process runs of the
# other configurations, after the headline decode batch, reported under "workloads".  Steps are
# few (each still W >= 3 warm-ups, CUDA events, the L2 rule of the headline) so the whole run
# stays within a couple of minutes; no end-to-end pass and no CPU baseline for these.
EXTRA_WORKLOADS = (("long_window", 50), ("prefill_100k", 5), ("prefill_208k", 5), ("full_model", 10))


def extra_workloads(args, pg, world, peaks, peak_src):
    if args.no_extra or args.workload != "decode_batch":
        return None
    import gc
    import torch
    out = {}
    for name, steps in EXTRA_WORKLOADS:
        gc.collect()
        torch.cuda.empty_cache()
        r = measure(name, steps, 3, False, pg, world, peaks, peak_src)
        roof = dict(r["roof"])
        if r["prefill"]:
            burst = peaks.get("bf16_tflops", 1900.0)
            roof["frac_of_burst"] = roof["achieved"] / burst
            roof["peak_burst"] = burst
        out[name] = {"ms_per_step": r["ms"], "value": r["value"], "unit": r["unit"], "steps": steps, "warmup": 3,
                     "tokens_per_s": r["tokens_s"], "gpu_launches": r["launches"], "roofline": roof,
                     "clocks": r["clocks"], "kernels_per_step": kernels_per_step(r["times"], r["nprof"]),
                     "l2": "flushed between steps" if r["flush"] else "inputs larger than L2",
                     "config": {"S": r["w"].S, "R": r["w"].R, "H": r["w"].H, "caches": r["w"].num_caches,
                                "lens_sum": int(np.sum(r["w"].lens))}}
        del r
    return out


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    import torch
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    from paged_mla_kv_gb300 import binding as B
    from paged_mla_kv_gb300 import build as BUILD
    from paged_mla_kv_gb300.harness import Resident
    BUILD.build()
    peaks, peak_src = load_peaks()
    if args.workload in TOPK:
        topk_main(args, rank, world, pg, peaks, peak_src)
        if pg is not None:
            pg.destroy_process_group()
        return
    r = measure(args.workload, args.steps, args.warmup, not args.no_e2e, pg, world, peaks, peak_src)
    w, units, ms, value, unit = r["w"], r["units"], r["ms"], r["value"], r["unit"]
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = OracleSample(w, args.cpu_seconds).measure()

    # the other configurations, on one GPU only (the scaling runs time the headline alone)
    extra = extra_workloads(args, pg, world, peaks, peak_src) if world == 1 else None
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": w.name, "S": w.S, "R": w.R, "H": w.H, "caches": w.num_caches,
                           "lens_sum": int(np.sum(w.lens)), "kv_bytes": units["kv"],
                           "unique_kv_bytes": units.get("unique_kv", units["kv"]),
                           "l2": "flushed between steps" if r["flush"] else "inputs larger than L2",
                           "parallelism": f"replicas x{world}", "tokens_per_step": units["tokens"]},
                "tokens_per_s": r["tokens_s"], "gpu_launches": r["launches"], "roofline": r["roof"],
                "cpu_baseline": cpu, "e2e": r["e2e"], "clocks": r["clocks"],
                "kernels_per_step": kernels_per_step(r["times"], r["nprof"])}
        if extra:
            line["workloads"] = extra
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
