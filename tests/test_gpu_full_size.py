"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

Attention is compared with the fp64 oracle on every (stream, row, head) the oracle
finishes in seconds (all of them for the decode batch and the long window), on a
seeded sample of query rows for the prefill chunks, and on a subset of caches for
the full-model step; the state copy and appends are compared byte for byte.
"""
import numpy as np
import pytest
import torch

from oracle import attend as OA
from paged_mla_kv_gb300 import binding as B
from paged_mla_kv_gb300 import build as BUILD
from paged_mla_kv_gb300 import synth as Y
from paged_mla_kv_gb300.harness import Resident
from tests.gpu_common import bits, compare, no_device_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    BUILD.build()
    B.lib()


def run_step(res, cache=0):
    """One bench step for a cache: append the current rows, then attend."""
    lat, rope = res.current_rows(cache)
    res.append_current(cache, lat, rope)
    out, lse = res.attend(res.q(cache), cache=cache)
    torch.cuda.synchronize()
    return out, lse


def test_tiny_decode():
    w = Y.tiny_decode()
    res = Resident(w)
    out, lse = run_step(res)
    no_device_error(res.pool)
    compare(w, out, lse)


def test_decode_batch_all_heads():
    w = Y.decode_batch()
    res = Resident(w)
    out, lse = run_step(res)
    no_device_error(res.pool)
    compare(w, out, lse)


def test_long_window_all_heads():
    w = Y.long_window()
    assert w.pages_needed() <= 2056
    res = Resident(w)
    out, lse = run_step(res)
    no_device_error(res.pool)
    compare(w, out, lse)


@pytest.mark.parametrize("variant", ["sharp", "ramp"])
def test_decode_batch_peaked_scores(variant):
    """The decode batch with peaked scores, so the running maximum moves and the lazy rescale
    of O^T runs inside the streams' long key runs: q ~ N(0, 1) with scale 0.5 (scores of
    std ~1.2), or a ramp (rope column 0 grows with position, later keys dominate)."""
    w = Y.decode_batch()
    if variant == "sharp":
        w.q_std, w.scale = 1.0, 0.5
    else:
        w.ramp = 600.0
    res = Resident(w)
    out, lse = run_step(res)
    no_device_error(res.pool)
    compare(w, out, lse)


@pytest.mark.parametrize("variant", ["sharp", "ramp"])
def test_long_window_peaked_scores(variant):
    """The long window (one 1,048,576-key stream, R = 2) with peaked scores: with the ramp
    the scores climb ~25 nats across the window, so the reference maximum moves several
    times along the 16,384 key tiles of stream 0 and O^T is rescaled in flight."""
    w = Y.long_window()
    if variant == "sharp":
        w.q_std, w.scale = 1.0, 0.5
    else:
        w.ramp = 600.0
    res = Resident(w)
    out, lse = run_step(res)
    no_device_error(res.pool)
    compare(w, out, lse)


@pytest.mark.parametrize("name", ["prefill_100k", "prefill_208k"])
def test_prefill_sampled_rows(name):
    w = Y.WORKLOADS[name]()
    res = Resident(w)
    out, lse = run_step(res)
    no_device_error(res.pool)
    g = np.random.default_rng(9)
    rows = np.unique(np.concatenate([[0, 1, w.R - 2, w.R - 1], g.choice(w.R, 12, replace=False)]))
    items = [np.array([r * w.H + h for r in rows for h in range(w.H)], np.int32)]
    compare(w, out, lse, items_per_stream=items)


def test_full_model_step():
    w = Y.full_model()
    at = w.extra["at"]
    res = Resident(w, caches=[0, 5, 11])   # rows written for three of the twelve caches
    for c in (0, 5, 11):
        out, lse = run_step(res, c)
        compare(w, out, lse, cache=c)
    # kept-state copy of stream 0's first 32,768 rows into fresh pages, every cache, bit-exact
    pages = -(-at // 512)
    dst = res.pool.take(pages)
    src = res.pt_host[0, :pages].copy()
    B.tf_state_copy_rows(res.pool, -1, torch.from_numpy(src).cuda(), torch.from_numpy(dst.copy()).cuda(), at)
    torch.cuda.synchronize()
    no_device_error(res.pool)
    img = res.pool.view()
    for c in (0, 5, 11):
        a = bits(img[c, torch.from_numpy(src.astype(np.int64)).cuda()])
        b = bits(img[c, torch.from_numpy(dst.astype(np.int64)).cuda()])
        assert np.array_equal(a, b)         # at is page-aligned here: whole pages equal
    # and the copied state attends exactly like the original stream
    pt2 = res.pt.clone()
    pt2[0, :pages] = torch.from_numpy(dst.copy()).cuda()
    q = res.q(5)
    o1 = torch.empty((w.S, 1, w.H, 512), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    B.tf_paged_mla_attend(res.pool, 5, res.pt, res.max_pages, res.lens, q, w.scale, o1, None, res.workspace())
    B.tf_paged_mla_attend(res.pool, 5, pt2, res.max_pages, res.lens, q, w.scale, o2, None, res.workspace())
    torch.cuda.synchronize()
    assert np.array_equal(bits(o1), bits(o2))


def test_fp8_decode_all_heads():
    """The decode batch on FP8 pages, as bench.py runs it: a quantizing append, then the
    expansion and the attention, against the oracle over the dequantized rows."""
    w = Y.WORKLOADS["fp8_decode"]()
    res = Resident(w, fp8=True)
    out, lse = run_step(res)
    no_device_error(res.pool)
    compare(w, out, lse, fp8=True)


def test_sparse_decode_full_size():
    """64 streams, 64 heads, 2,048 listed rows each, in the benchmark's launch configuration."""
    from tests.test_gpu_sparse import check, run_sparse
    w = Y.WORKLOADS["sparse_decode"]()
    lists = Y.listed_rows(w.seed, w.lens, int(w.extra["nidx"]))
    res = Resident(w)
    lat, rope = res.current_rows(0)
    res.append_current(0, lat, rope)
    out, lse = run_sparse(res, w, lists)
    no_device_error(res.pool)
    check(w, out, lse, lists)
