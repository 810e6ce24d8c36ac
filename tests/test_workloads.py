"""The synthetic workloads hold the shapes, sizes, sharing and value distributions of the input
recipe (host only).  Each named workload is checked against its stated form: stream count,
heads, query rows, caches, length ranges, the prefix pages streams share, pool sizes, listed
rows, and that generation is deterministic in the seed."""
import numpy as np
import pytest

from paged_mla_kv_gb300 import synth as Y


def test_tiny_decode():
    w = Y.WORKLOADS["tiny_decode"]()
    assert (w.S, w.R, w.H, w.num_caches, w.seed) == (1, 1, 16, 1, 1)
    assert list(w.lens) == [2048] and w.pages_of(0) == 4 and w.pool_pages == 16


def test_decode_batch():
    w = Y.WORKLOADS["decode_batch"]()
    assert (w.S, w.R, w.H, w.num_caches, w.seed) == (8, 1, 64, 1, 2)
    assert np.all((w.lens >= 4096) & (w.lens <= 65536))
    for s in range(8):
        src, n = w.share[s]
        if 1 <= s <= 3:   # streams 1-3 read stream 0's first pages, at most 16 (8,192 rows)
            want = min(16, (int(w.lens[s]) - 1) // 512, (int(w.lens[0]) - 1) // 512)
            assert (src, n) == (0, want) and n > 0
        else:
            assert n == 0
    need = w.pages_needed()
    assert w.pool_pages == need + round(0.10 * need)      # 10% spare pages


def test_long_window():
    w = Y.WORKLOADS["long_window"]()
    assert (w.S, w.R, w.H, w.seed, w.pool_pages) == (8, 2, 64, 3, 2056)
    assert int(w.lens[0]) == 1048576 and w.pages_of(0) == 2048
    assert np.all((w.lens[1:] >= 2) & (w.lens[1:] <= 8192))
    for s in range(1, 8):
        assert w.share[s] == (0, (int(w.lens[s]) - 1) // 512) and w.own_pages(s) == 1
    assert w.pages_needed() == 2048 + 7    # one spare page of the 2,056


@pytest.mark.parametrize("name,T,L", [("prefill_100k", 2048, 100000), ("prefill_208k", 1024, 208000)])
def test_prefill_chunks(name, T, L):
    w = Y.WORKLOADS[name]()
    assert (w.S, w.R, w.H, w.seed) == (1, T, 64, 4)
    assert int(w.lens[0]) == L + T          # query row t sits at L + t
    assert w.pool_pages >= w.pages_of(0)


def test_full_model():
    w = Y.WORKLOADS["full_model"]()
    assert (w.S, w.R, w.H, w.num_caches, w.seed) == (16, 1, 64, 12, 5)
    assert np.all(w.lens == 40960) and w.extra["at"] == 32768
    assert w.pool_pages == w.pages_needed() + 64   # room for the kept state's 64 pages


@pytest.mark.parametrize("name", ["sparse_decode", "sparse_fp8_decode"])
def test_listed_row_workloads(name):
    w = Y.WORKLOADS[name]()
    assert (w.S, w.R, w.H, w.seed, w.extra["nidx"]) == (64, 1, 64, 6, 2048)
    assert np.all((w.lens >= 4096) & (w.lens <= 65536))
    lists = Y.listed_rows(w.seed, w.lens, 2048)
    for L, x in zip(w.lens, lists):
        assert len(x) == 2048 and len(np.unique(x)) == 2048 and x.min() >= 0 and x.max() < L
        assert not np.all(np.diff(x) > 0)   # a random order, not sorted
    assert bool(w.extra.get("fp8")) == (name == "sparse_fp8_decode")


def test_fp8_decode_is_the_decode_batch_on_fp8_pages():
    a, b = Y.WORKLOADS["decode_batch"](), Y.WORKLOADS["fp8_decode"]()
    assert b.extra.get("fp8") and not a.extra.get("fp8")
    assert np.array_equal(a.lens, b.lens) and a.share == b.share and a.pool_pages == b.pool_pages
    assert np.array_equal(a.stream_rows(0, 5, 100, 300)[0], b.stream_rows(0, 5, 100, 300)[0])


def test_shared_pages_are_the_owners_bytes_and_private_pages_differ():
    w = Y.WORKLOADS["decode_batch"]()
    n = w.shared_pages(1)
    lat1, rope1 = w.stream_rows(0, 1, 0, n * 512)
    lat0, rope0 = w.stream_rows(0, 0, 0, n * 512)
    assert np.array_equal(lat1, lat0) and np.array_equal(rope1, rope0)
    assert not np.array_equal(w.page_rows(0, 1, n)[0], w.page_rows(0, 0, n)[0])
    assert not np.array_equal(w.page_rows(1, 0, 0)[0], w.page_rows(0, 0, 0)[0])   # caches differ


def test_values_are_bf16_normal_and_deterministic():
    w = Y.WORKLOADS["decode_batch"]()
    lat, rope = w.stream_rows(0, 2, 0, 2048)
    q = w.q(0)
    for bits in (lat, rope, q):
        v = Y.bf16_bits_to_f32(bits).astype(np.float64)
        assert abs(v.mean()) < 0.01 and abs(v.std() - 0.1) < 0.005
        # bf16 bit patterns: the float32 of each value has a zero low half
        assert np.all((Y.bf16_bits_to_f32(bits).view(np.uint32) & 0xFFFF) == 0)
    w2 = Y.WORKLOADS["decode_batch"]()
    assert np.array_equal(w2.stream_rows(0, 2, 0, 2048)[0], lat) and np.array_equal(w2.q(0), q)
    assert not np.array_equal(Y.decode_batch(seed=9).q(0), q)


def test_topk_prefill():
    w = Y.TOPK_WORKLOADS["topk_prefill"]()
    assert (w.rows, w.n, w.k, w.seed) == (2048, 100000, 512, 7)
    assert np.array_equal(w.lens, 100000 - 2048 + 1 + np.arange(2048))   # causal: row t sees L - T + 1 + t
    x = Y.topk_logits(w.seed, [0, 2047], 1000)
    assert np.all(np.round(x * 64) == x * 64)                          # multiples of 1/64
    assert len(np.unique(x[0])) < 1000                                 # equal scores are common
    assert np.array_equal(Y.topk_logits(w.seed, [2047], 1000)[0], x[1])   # a row depends on its index only
