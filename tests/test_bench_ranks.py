"""The multi-rank bench logic on CPU with gloo (world size 2): every rank gets the
slowest rank's time, and the whole-job rate counts the units of all replicas."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [3.0, 7.5][rank]
    slowest = bench.max_over_ranks(mine, dist, "cpu")
    rate = bench.whole_job_rate(100.0, world, slowest)
    q.put((rank, slowest, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [7.5, 7.5]
    assert got[0][2] == pytest.approx(2 * 100.0 / 7.5e-3)


def test_single_rank_needs_no_group():
    assert bench.max_over_ranks(4.25) == 4.25
    assert bench.whole_job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)


def test_kernel_times_read_every_kind_and_scale_per_step():
    """The bench's per-kind kernel times: every launch kind is read (and cleared) from the pool's
    records, and only kinds that ran appear, per step.  The pool sits over host bytes it never
    touches; with nothing recorded no CUDA call is made."""
    from paged_mla_kv_gb300 import binding as B
    from paged_mla_kv_gb300 import build as BUILD
    BUILD.build()
    mem = torch.empty(B.tf_kvpool_bytes(B.make_desc(1, 4)) + 1024, dtype=torch.uint8)
    pool = B.KVPool(1, 4, memory=mem)
    pool.profile(True)
    t = bench.read_kernel_times(pool)
    assert set(t) == {"append", "attend", "combine", "state_copy", "poison"}
    assert all(v == (0.0, 0) for v in t.values())
    assert bench.kernels_per_step(t, 10) == {}
    got = bench.kernels_per_step({"attend": (5.0, 20), "append": (1.0, 10), "combine": (0.0, 0)}, 10)
    assert got == {"attend": {"ms": 0.5, "launches": 2.0}, "append": {"ms": 0.1, "launches": 1.0}}
    pool.close()


@pytest.mark.parametrize("workload", ["tiny_decode", "topk_prefill"])
def test_reference_arm_line(workload, capsys, monkeypatch):
    """The reference arm on the host: one JSON line with the contract's keys, the oracle as its
    baseline and no host-device bytes (the run's time budget cut to a few seconds here)."""
    import argparse
    import json
    monkeypatch.setattr(bench, "REFERENCE_SECONDS", 3.0)
    args = argparse.Namespace(workload=workload, steps=3, warmup=3, gpus=1, impl="reference",
                              no_cpu_baseline=False, no_e2e=False, cpu_seconds=1.0)
    bench.reference_arm(args, 0, 1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["config"]["workload"] == workload
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    bench.reference_arm(args, 1, 2)            # other ranks print nothing
    assert capsys.readouterr().out == ""


def test_algorithmic_work_matches_the_stated_formulas():
    """The roofline's numerator: the bytes and flops a step is credited with, recomputed here from
    the per-unit figures (a key row read once a stream for all heads; q, out and lse once; a
    (row, head, key) triple is 2 x (576 + 512) flops)."""
    from paged_mla_kv_gb300 import synth as Y
    w = Y.WORKLOADS["decode_batch"]()
    u = bench.step_units(w)
    S, R, H = w.S, w.R, w.H
    assert u["attend_bytes"] == int(np.sum(w.lens)) * 1152 + S * R * H * (576 * 2 + 512 * 2 + 4)
    assert u["kv"] == int(np.sum(w.lens)) * 1152 and u["tokens"] == S * R
    shared = sum(w.share[s][1] for s in range(S)) * 512 * 1152          # streams 1-3's prefix pages
    assert u["unique_kv"] == u["kv"] - shared and shared > 0
    f = Y.WORKLOADS["fp8_decode"]()
    assert bench.step_units(f)["attend_bytes"] == int(np.sum(f.lens)) * 644 + S * R * H * (576 * 2 + 512 * 2 + 4)
    p = Y.WORKLOADS["prefill_100k"]()
    T, L = 2048, 100000
    pairs = sum(L + t + 1 for t in range(T))              # row t sees L + t + 1 keys
    assert bench.step_units(p)["attend_flops"] == 2176 * 64 * pairs
    assert abs(2176 * 64 * pairs / 1e12 - 28.81) < 0.01    # the chunk's 28.81 TFLOP
    sp = Y.WORKLOADS["sparse_decode"]()
    assert bench.step_units(sp)["attend_bytes"] == 64 * 2048 * 1152 + 64 * 64 * (576 * 2 + 512 * 2 + 4)
    fm = Y.WORKLOADS["full_model"]()
    uf = bench.step_units(fm)
    one = 16 * 40960 * 1152 + 16 * 64 * (576 * 2 + 512 * 2 + 4)
    assert uf["attend_bytes"] == one
    assert uf["bytes"] == 12 * (one + 16 * 2 * 1152) + 2 * 32768 * 1152 * 12   # appends and the state copy
    tk = Y.TOPK_WORKLOADS["topk_prefill"]()
    keys = sum(100000 - 2048 + 1 + t for t in range(2048))
    assert bench.topk_bytes(tk) == 4 * keys + 2048 * 512 * 8
    assert abs(bench.topk_bytes(tk) / 1e6 - 819.2) < 0.1  # 810.8 MB of logits in play + 8.4 MB written
