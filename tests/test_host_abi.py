"""Host-side tests of the C-ABI library: it loads, exports every declared symbol,
its plan arithmetic equals the oracle's, its pool bookkeeping behaves, and bad
arguments are refused on the host before any launch.  No GPU is needed: the
pool is created over a fake (aligned, never dereferenced) device address."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import plan as OP
from paged_mla_kv_gb300 import binding as B
from paged_mla_kv_gb300 import build as BUILD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    BUILD.build()
    return B.lib()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(tf_\w+)\s*\(", txt))
    return names


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert "tf_paged_mla_attend" in names and "tf_paged_append" in names
    assert "tf_kvpool_create" in names and "tf_state_copy_rows" in names
    for n in sorted(names):
        assert hasattr(L, n), n


def _fake_pool(num_pages=16, caches=1, seed=0, poison=False):
    desc = B.make_desc(caches, num_pages, poison, seed)
    nbytes = B.tf_kvpool_bytes(desc)
    h = ctypes.c_void_p()
    rc = B.lib().tf_kvpool_create(ctypes.byref(desc), ctypes.c_void_p(1 << 40), nbytes, ctypes.byref(h))
    assert rc == 0
    return h, desc


def _take(h, n):
    ids = np.zeros(max(n, 1), np.int32)
    rc = B.lib().tf_kvpool_take(h, n, ids.ctypes.data_as(ctypes.c_void_p), None)
    return rc, ids[:n]


def _ids(a):
    a = np.ascontiguousarray(np.asarray(a, np.int32))
    return a, a.ctypes.data_as(ctypes.c_void_p), len(a)


def test_pool_bytes_and_descriptor_checks(L):
    d = B.make_desc(12, 1344)
    assert B.tf_kvpool_bytes(d) == 12 * 1344 * 589824 + 256
    bad = B.make_desc(1, 16)
    bad.page_rows = 256
    assert B.tf_kvpool_bytes(bad) == 0
    assert B.tf_kvpool_bytes(B.make_desc(65535, 1)) == 65535 * 589824 + 256
    assert B.tf_kvpool_bytes(B.make_desc(65536, 1)) == 0      # caches are a launch's grid.y
    assert B.tf_kvpool_bytes(B.make_desc(2, 1 << 30)) == 0    # 2^31 pages over all caches
    h = ctypes.c_void_p()
    good = B.make_desc(1, 16)
    n = B.tf_kvpool_bytes(good)
    assert L.tf_kvpool_create(ctypes.byref(good), ctypes.c_void_p((1 << 40) + 512), n, ctypes.byref(h)) == B.TF_E_ARG
    assert L.tf_kvpool_create(ctypes.byref(good), ctypes.c_void_p(1 << 40), n - 1, ctypes.byref(h)) == B.TF_E_NOMEM


def test_take_ref_release(L):
    h, _ = _fake_pool(8)
    rc, a = _take(h, 5)
    assert rc == 0 and sorted(a) == [0, 1, 2, 3, 4]
    assert L.tf_kvpool_free_pages(h) == 3
    rc, _ = _take(h, 4)
    assert rc == B.TF_E_NOMEM and L.tf_kvpool_free_pages(h) == 3
    arr, p, n = _ids(a[:2])
    assert L.tf_kvpool_ref(h, p, n) == 0
    assert L.tf_kvpool_refcount(h, int(a[0])) == 2
    assert L.tf_kvpool_release(h, p, n) == 0
    assert L.tf_kvpool_refcount(h, int(a[0])) == 1 and L.tf_kvpool_free_pages(h) == 3
    assert L.tf_kvpool_release(h, p, n) == 0
    assert L.tf_kvpool_free_pages(h) == 5 and L.tf_kvpool_refcount(h, int(a[0])) == 0
    # releasing a free page, or a page twice in one call beyond its count, changes nothing
    arr, p, n = _ids([a[0]])
    assert L.tf_kvpool_release(h, p, n) == B.TF_E_RANGE
    arr, p, n = _ids([a[2], a[2]])
    assert L.tf_kvpool_release(h, p, n) == B.TF_E_RANGE and L.tf_kvpool_refcount(h, int(a[2])) == 1
    arr, p, n = _ids([99])
    assert L.tf_kvpool_ref(h, p, n) == B.TF_E_RANGE
    arr, p, n = _ids([a[0]])
    assert L.tf_kvpool_ref(h, p, n) == B.TF_E_RANGE          # a free page cannot be shared
    # freed pages come back last (FIFO), so a just-freed page is not reused at once
    rc, b = _take(h, 3)
    assert rc == 0 and set(b) == {5, 6, 7}
    L.tf_kvpool_destroy(h)


def test_seeded_free_list_is_a_permutation(L):
    h1, _ = _fake_pool(64, seed=1234)
    h2, _ = _fake_pool(64, seed=1234)
    h3, _ = _fake_pool(64, seed=99)
    _, a = _take(h1, 64)
    _, b = _take(h2, 64)
    _, c = _take(h3, 64)
    assert sorted(a) == list(range(64)) and np.array_equal(a, b) and not np.array_equal(a, c)
    assert not np.array_equal(a, np.arange(64))
    for h in (h1, h2, h3):
        L.tf_kvpool_destroy(h)


def test_page_ptr(L):
    h, _ = _fake_pool(10, caches=3)
    assert L.tf_kvpool_page_ptr(h, 2, 7) == (1 << 40) + (2 * 10 + 7) * 589824
    assert not L.tf_kvpool_page_ptr(h, 3, 0)
    assert not L.tf_kvpool_page_ptr(h, 0, 10)
    L.tf_kvpool_destroy(h)


GiB, MiB = 1 << 30, 1 << 20


@pytest.mark.parametrize("paged", [False, True])
def test_plan_equals_oracle(L, paged):
    rng = np.random.default_rng(5)
    for _ in range(400):
        kw = dict(room_bytes=int(rng.integers(0, 300 * GiB)), context_tokens=int(rng.integers(1, 2_000_000)),
                  lanes=int(rng.integers(1, 65)), bytes_per_token=int(rng.choice([1152, 13056, 13824, 6912])),
                  fixed_bytes=int(rng.integers(0, 400 * MiB)), cache_budget_bytes=int(rng.integers(0, 32 * GiB)),
                  engine_paged=paged)
        got = B.tf_kvpool_plan(**kw)
        want = OP.plan(OP.PlanIn(kw["room_bytes"], kw["context_tokens"], kw["lanes"], kw["bytes_per_token"],
                                 kw["fixed_bytes"], kw["cache_budget_bytes"], engine_paged=paged))
        if want is None:
            assert got is None
            continue
        assert (got.n_windows, got.window_pages, got.stream_pages, got.cache_bytes, got.other_pages,
                got.pool_pages, got.pool_tokens) == (want.n_windows, want.window_pages, want.stream_pages,
                                                     want.cache_bytes, want.other_pages, want.pool_pages,
                                                     want.pool_tokens)


def test_plan_worked_example(L):
    room = int(round(2.33 * GiB)) + 1048576 * 13056 + 180 * MiB
    out = B.tf_kvpool_plan(room_bytes=room, context_tokens=1048576, lanes=8, bytes_per_token=13056,
                           fixed_bytes=180 * MiB, cache_budget_bytes=16 * GiB)
    assert out.pool_pages == 2056 and out.pool_tokens == 1052672


def _args_refused(L, h, fn, *args):
    before = L.tf_launch_count()
    rc = fn(h, *args)
    assert L.tf_launch_count() == before
    return rc


def test_bad_arguments_are_refused_before_launch(L):
    h, _ = _fake_pool(8, caches=2)
    fake = ctypes.c_void_p(1 << 41)
    lens = np.array([100, 5000], np.int64)
    lp = lens.ctypes.data_as(ctypes.c_void_p)
    A = L.tf_paged_mla_attend
    # cache out of range
    assert _args_refused(L, h, A, 2, fake, 16, lp, 2, 1, 16, fake, 0.1, fake, None, None, 0, None) == B.TF_E_RANGE
    # length beyond the table
    assert _args_refused(L, h, A, 0, fake, 4, lp, 2, 1, 16, fake, 0.1, fake, None, None, 0, None) == B.TF_E_RANGE
    # a length shorter than the query rows
    short = np.array([1, 50], np.int64)
    assert _args_refused(L, h, A, 0, fake, 16, short.ctypes.data_as(ctypes.c_void_p), 2, 2, 16, fake, 0.1, fake,
                         None, None, 0, None) == B.TF_E_RANGE
    # too many heads, NaN scale, null q
    assert _args_refused(L, h, A, 0, fake, 16, lp, 2, 1, 129, fake, 0.1, fake, None, None, 0, None) == B.TF_E_ARG
    assert _args_refused(L, h, A, 0, fake, 16, lp, 2, 1, 16, fake, float("nan"), fake, None, None, 0,
                         None) == B.TF_E_ARG
    assert _args_refused(L, h, A, 0, fake, 16, lp, 2, 1, 16, None, 0.1, fake, None, None, 0, None) == B.TF_E_ARG
    assert _args_refused(L, h, A, 0, fake, 16, lp, 2, 1, 16, fake, 0.0, fake, None, None, 0, None) == B.TF_E_ARG
    assert _args_refused(L, h, A, 0, fake, 16, lp, 2, 1, 16, fake, -0.5, fake, None, None, 0, None) == B.TF_E_ARG
    # a null table needs S * max_pages pool pages
    assert _args_refused(L, h, A, 0, None, 16, lp, 2, 1, 16, fake, 0.1, fake, None, None, 0, None) == B.TF_E_RANGE
    # workspace missing or too small
    need = L.tf_paged_mla_workspace_bytes(h, 2, 1, 16, lp)
    assert need > 0
    assert _args_refused(L, h, A, 0, fake, 16, lp, 2, 1, 16, fake, 0.1, fake, None, None, 0, None) == B.TF_E_ARG
    assert _args_refused(L, h, A, 0, fake, 16, lp, 2, 1, 16, fake, 0.1, fake, None, fake, need - 1,
                         None) == B.TF_E_NOMEM
    # a stream longer than INT32_MAX rows (only a table that repeats page ids can hold one)
    long_ = np.array([(1 << 31) + 7, 5000], np.int64)
    wide = (1 << 31) // 512 + 1
    lq = long_.ctypes.data_as(ctypes.c_void_p)
    assert _args_refused(L, h, A, 0, fake, wide, lq, 2, 1, 16, fake, 0.1, fake, None, fake, 1 << 40,
                         None) == B.TF_E_UNSUPPORTED
    assert L.tf_paged_mla_workspace_bytes(h, 2, 1, 16, lq) == 0
    # S * R * H above 2^30: both the sizing call and the allocation-free entry point refuse it
    # before any plan arithmetic (R * H alone would overflow the plan's int column count)
    lbig = np.array([1 << 25], np.int64)
    lb = lbig.ctypes.data_as(ctypes.c_void_p)
    assert L.tf_paged_mla_workspace_bytes(h, 1, 1 << 25, 128, lb) == 0
    assert L.tf_paged_mla_workspace_bytes(None, 1, 1 << 25, 128, lb) == 0
    assert _args_refused(L, h, L.tf_paged_mla_attend_static, 0, fake, 1 << 16, lb, 1, 1 << 25, 128, fake, 0.1,
                         fake, None, None) == B.TF_E_UNSUPPORTED
    nidx = np.array([8, 8], np.int32)
    assert _args_refused(L, h, L.tf_paged_mla_attend_sparse, 0, fake, wide, lq, fake, 8,
                         nidx.ctypes.data_as(ctypes.c_void_p), 2, 16, fake, 0.1, fake, None, fake, 1 << 40,
                         None) == B.TF_E_UNSUPPORTED
    # append: position past the table
    pos = np.array([16 * 512 - 1], np.int64)
    assert _args_refused(L, h, L.tf_paged_append, 0, fake, 16, pos.ctypes.data_as(ctypes.c_void_p), 1, 2, fake,
                         fake, None) == B.TF_E_RANGE
    assert _args_refused(L, h, L.tf_paged_append, 5, fake, 16, pos.ctypes.data_as(ctypes.c_void_p), 1, 1, fake,
                         fake, None) == B.TF_E_RANGE
    huge = np.array([(1 << 63) - 1], np.int64)     # a position whose sum with n would overflow
    assert _args_refused(L, h, L.tf_paged_append, 0, fake, 16, huge.ctypes.data_as(ctypes.c_void_p), 1, 2, fake,
                         fake, None) == B.TF_E_RANGE
    # state copy: at past the pool, cache out of range
    assert _args_refused(L, h, L.tf_state_copy_rows, 0, fake, fake, 8 * 512 + 1, None) == B.TF_E_RANGE
    assert _args_refused(L, h, L.tf_state_copy_rows, 2, fake, fake, 10, None) == B.TF_E_RANGE
    assert _args_refused(L, h, L.tf_state_copy_rows, 0, fake, fake, -1, None) == B.TF_E_ARG
    L.tf_kvpool_destroy(h)


def test_workspace_is_bounded_by_the_cta_ranges(L):
    # partials come only from (stream, group) units cut by a CTA range boundary: at most
    # two a CTA, so the workspace does not grow with the lengths
    def ws(lens, R=1, H=64):
        a = np.array(lens, np.int64)
        return L.tf_paged_mla_workspace_bytes(None, len(a), R, H, a.ctypes.data_as(ctypes.c_void_p))
    assert ws([256]) == 0                       # four key tiles: one CTA, no partials
    w1, w2, w3 = ws([65536]), ws([65536, 4096]), ws([1 << 20, 7000, 9])
    assert 0 < w1 == w2 == w3
    slot = 64 * 512 * 4
    assert w1 <= 2 * 240 * slot + 2 * 240 * 64 * 2 * 4 + 255
    assert w1 <= 64 << 20                       # fits the static scratch of the allocation-free call


def test_fp8_pool_sizes_and_workspace(L):
    """FP8 pages: 329,728 bytes a page (codes, scales, rope).  On a batch-invariant pool
    attention's workspace adds the rows expanded to BF16 pages, a table and 1 KiB of alignment
    room; on a default pool the kernel expands the codes itself and needs only the partials.
    No device memory is touched."""
    desc = B.make_desc(3, 10, fp8=True, invariant=True)
    n = B.tf_kvpool_bytes(desc)
    assert n == 3 * 10 * B.PAGE_BYTES_FP8 + 256
    h = ctypes.c_void_p()
    assert L.tf_kvpool_create(ctypes.byref(desc), ctypes.c_void_p(1 << 40), n, ctypes.byref(h)) == B.TF_OK
    base = L.tf_kvpool_page_ptr(h, 0, 0)
    assert L.tf_kvpool_page_ptr(h, 1, 2) - base == (10 + 2) * B.PAGE_BYTES_FP8
    lens = np.array([1000, 513, 7], np.int64)
    lp = lens.ctypes.data_as(ctypes.c_void_p)
    dinv = B.make_desc(3, 10, invariant=True)   # the same partials on a BF16 invariant pool
    hb = ctypes.c_void_p()
    assert L.tf_kvpool_create(ctypes.byref(dinv), ctypes.c_void_p(1 << 40), B.tf_kvpool_bytes(dinv),
                              ctypes.byref(hb)) == B.TF_OK
    plain = L.tf_paged_mla_workspace_bytes(hb, 3, 1, 16, lp)
    L.tf_kvpool_destroy(hb)
    fp8 = L.tf_paged_mla_workspace_bytes(h, 3, 1, 16, lp)
    pages = 2 + 2 + 1
    assert fp8 == (plain + 1023) // 1024 * 1024 + 1024 + 1024 + pages * B.PAGE_BYTES_BF16
    L.tf_kvpool_destroy(h)
    d2 = B.make_desc(3, 10, fp8=True)
    assert L.tf_kvpool_create(ctypes.byref(d2), ctypes.c_void_p(1 << 40), n, ctypes.byref(h)) == B.TF_OK
    assert L.tf_paged_mla_workspace_bytes(h, 3, 1, 16, lp) == L.tf_paged_mla_workspace_bytes(None, 3, 1, 16, lp)
    L.tf_kvpool_destroy(h)
    bad = B.make_desc(1, 4)
    bad.flags = 8
    assert B.tf_kvpool_bytes(bad) == 0


def test_topk_bad_arguments_are_refused_before_launch(L):
    fake = ctypes.c_void_p(1 << 41)
    T = L.tf_topk_blocked

    def refused(*a):
        before = L.tf_launch_count()
        rc = T(*a)
        assert L.tf_launch_count() == before
        return rc

    for k in (0, 2049):
        assert refused(fake, 2, 64, 64, None, k, fake, fake, None, 0, None) == B.TF_E_ARG
    assert refused(fake, -1, 64, 64, None, 8, fake, fake, None, 0, None) == B.TF_E_ARG        # rows < 0
    assert refused(fake, 2, 64, 63, None, 8, fake, fake, None, 0, None) == B.TF_E_ARG         # ld < n
    assert refused(fake, 2, 60, 62, None, 8, fake, fake, None, 0, None) == B.TF_E_ARG         # ld % 4
    assert refused(ctypes.c_void_p((1 << 41) + 4), 2, 64, 64, None, 8, fake, fake, None, 0,
                   None) == B.TF_E_ARG                                                          # unaligned
    assert refused(None, 2, 64, 64, None, 8, fake, fake, None, 0, None) == B.TF_E_ARG         # null logits
    assert refused(fake, 2, 64, 64, None, 8, fake, None, None, 0, None) == B.TF_E_ARG         # null values
    # sizes the launch cannot number
    assert refused(fake, 1 << 31, 64, 64, None, 8, fake, fake, fake, 1 << 62, None) == B.TF_E_UNSUPPORTED
    assert refused(fake, 2, 1 << 31, 1 << 31, None, 8, fake, fake, fake, 1 << 62, None) == B.TF_E_UNSUPPORTED
    # two levels need a workspace of the stated size
    need = L.tf_topk_workspace_bytes(2, 40000, 8)
    assert need == 2 * 3 * 8 * 8            # a row's 3 first-level blocks keep 8 (key, column) pairs each
    # 17 blocks of 512 candidates need two merge blocks, then a last level: both lower levels are held
    assert L.tf_topk_workspace_bytes(1, 17 * 16384, 512) == (17 + 2) * 512 * 8
    assert refused(fake, 2, 40000, 40000, None, 8, fake, fake, None, 0, None) == B.TF_E_NOMEM
    assert refused(fake, 2, 40000, 40000, None, 8, fake, fake, fake, need - 1, None) == B.TF_E_NOMEM
    assert L.tf_topk_workspace_bytes(2, 16384, 8) == 0     # one block a row: a single level
    assert refused(None, 0, 64, 64, None, 8, None, None, None, 0, None) == B.TF_OK            # no rows


C_CALLER = r"""
#include <stdio.h>
#include "tf_paged_mla.h"
#include "tf_topk.h"

int main(void)
{
    /* the plan of a TP=2 pair at a 1M window with 8 lanes (the pages' worked example) */
    const int64_t GiB = (int64_t)1 << 30, MiB = (int64_t)1 << 20;
    tf_plan_in in = {0};
    tf_plan_out out = {0};
    in.room_bytes = (int64_t)(2.33 * (double)GiB + 0.5) + (int64_t)1048576 * 13056 + 180 * MiB;
    in.context_tokens = 1048576;
    in.lanes = 8;
    in.page_rows = TF_PAGE_ROWS;
    in.lookahead = 1;
    in.engine_paged = 0;
    in.bytes_per_token = 13056;
    in.fixed_bytes = 180 * MiB;
    in.cache_budget_bytes = 16 * GiB;
    if (tf_kvpool_plan(&in, &out) != TF_OK) return 1;
    tf_kvpool_desc d = {12, 1344, TF_PAGE_ROWS, TF_LATENT_DIM, TF_ROPE_DIM, 0u, 0u};
    tf_kvpool_desc f = d;
    f.flags = TF_POOL_FP8;
    tf_kvpool *pool = NULL;
    int rc = tf_kvpool_create(&d, (void *)0, 0, &pool);   /* a null base is refused */
    printf("%lld %lld %zu %zu %zu %d %d\n", (long long)out.pool_pages, (long long)out.pool_tokens,
           tf_kvpool_bytes(&d), tf_kvpool_bytes(&f), tf_topk_workspace_bytes(2, 40000, 8), rc, pool == NULL);
    return 0;
}
"""


def test_headers_compile_as_c_and_the_library_links_from_c(L, tmp_path):
    """The C ABI as a C caller sees it: both headers compile as strict C99 with every warning an
    error, and a C program linked to the library gets the same answers as the binding."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(B.LIB_PATH)
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-ltf_paged_mla", "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    got = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    want = [2056, 1052672, 12 * 1344 * 589824 + 256, 12 * 1344 * 329728 + 256, 2 * 3 * 8 * 8, B.TF_E_ARG, 1]
    assert [int(x) for x in got] == want


def _weighted_sizes(bounds, lens, seg):
    """Tiles of each range plus `seg` for every stream after the first that starts inside it (a
    segment start costs a query reload, an extra epilogue and the pipeline's refill)."""
    tiles = -(-np.asarray(lens, np.int64) // 64)
    starts = np.cumsum(tiles)[:-1]
    return [int(bounds[i + 1] - bounds[i]) + seg * int(np.sum((starts >= bounds[i]) & (starts < bounds[i + 1])))
            for i in range(len(bounds) - 1)]


@pytest.mark.parametrize("name", ["decode_batch", "long_window", "full_model", "tiny_decode"])
def test_decode_plan_deals_every_tile_once_in_balanced_ranges(L, name):
    from paged_mla_kv_gb300 import synth as Y
    w = Y.WORKLOADS[name]()
    pl = B.tf_paged_mla_plan_info(w.S, w.R, w.H, w.lens, sms=152)
    tiles = int(np.sum(-(-w.lens // 64)))
    assert pl["mode"] == 0 and pl["work"] == tiles and pl["groups"] == -(-w.R * w.H // 64)
    b = pl["bounds"]
    assert b[0] == 0 and b[-1] == tiles and np.all(np.diff(b) >= 1)     # every tile in exactly one range
    assert pl["ctas"] == pl["nranges"] * pl["groups"] <= 152
    assert pl["nranges"] == min(-(-tiles // 4), 152 // pl["groups"])     # at least 4 tiles a range
    # the weight the library gives a segment start: 5 tiles with one column group, 12 with more;
    # a cut inside a stream's start weight moves to the stream's start, so sizes differ by up to it
    seg = 5 if pl["groups"] == 1 else 12
    wsz = _weighted_sizes(b, w.lens, seg)
    assert max(wsz) - min(wsz) <= 8 + seg, (min(wsz), max(wsz))
    assert pl["slots"] in (0, 2 * pl["ctas"])                           # two partial slots a CTA


def test_plan_and_workspace_agree(L):
    from paged_mla_kv_gb300 import synth as Y
    w = Y.WORKLOADS["decode_batch"]()
    pl = B.tf_paged_mla_plan_info(w.S, w.R, w.H, w.lens)               # the same SM count as the sizing
    slots = pl["slots"]
    assert slots > 0
    want = slots * 64 * 512 * 4 + (-(-(slots * 64 * 2 * 4) // 256)) * 256
    assert B.tf_paged_mla_workspace_bytes(None, w.S, w.R, w.H, w.lens) == want


def _unit_ranges(pl, lens, R, H):
    """Per range of a mode-1 plan: (64-key tiles, segments, cut positions inside units), walking
    the bounds over units that each hold as many tiles as their last column sees."""
    G, ncols = pl["groups"], R * H

    def nt(u):
        s, g = divmod(u, G)
        clast = min(64 * g + 63, ncols - 1)
        return -(-(int(lens[s]) - R + clast // H + 1) // 64)

    out = []
    b = [divmod(int(x), 1 << 32) for x in pl["bounds"]]
    for c in range(pl["nranges"]):
        (u, t), end = b[c], b[c + 1]
        tiles = segs = 0
        while (u, t) < end:
            e = end[1] if u == end[0] else nt(u)
            tiles += e - t
            segs += 1
            u, t = u + 1, 0
        out.append((tiles, segs))
    cuts = [(u, t, nt(u)) for u, t in b[1:-1] if t != 0]
    return out, cuts, sum(nt(u) for u in range(pl["work"]))


@pytest.mark.parametrize("name", ["prefill_100k", "prefill_208k"])
def test_prefill_plan_balances_tile_ranges(L, name):
    """A prefill chunk's units are cut into equal ranges of key tiles, one CTA each: no CTA
    carries a whole extra unit (2,048 or 1,024 units over 152 SMs dealt round robin leave 14
    against 13.5, or 7 against 6.7), cuts inside a unit fall on its eighths, and each unit reads
    only the tiles its last row sees."""
    from paged_mla_kv_gb300 import synth as Y
    w = Y.WORKLOADS[name]()
    pl = B.tf_paged_mla_plan_info(w.S, w.R, w.H, w.lens, sms=152)
    assert pl["mode"] == 1 and pl["groups"] == w.R and pl["work"] == w.R
    assert pl["ctas"] == pl["nranges"] == 152 and pl["slots"] == 2 * 152
    assert pl["bounds"][0] == 0 and pl["bounds"][-1] == w.R << 32
    ranges, cuts, total = _unit_ranges(pl, w.lens, w.R, w.H)
    L0 = int(w.lens[0])
    # row r of the chunk sees L0 - R + r + 1 keys; a 64-head group is one row
    assert total == sum(-(-(L0 - w.R + r + 1) // 64) for r in range(w.R))
    assert sum(t for t, _ in ranges) == total
    loads = [t + 3 * n for t, n in ranges]     # a segment start weighs three tiles
    mean = sum(loads) / len(loads)
    unit = total / w.R
    assert max(loads) <= mean + unit / 8 + 6   # within an eighth of a unit of the mean
    assert max(loads) <= 1.01 * mean
    assert max(loads) < 0.99 * (-(-w.R // 152)) * unit    # whole units round robin: 3-4% more
    assert cuts and all(t in [k * n // 8 for k in range(1, 8)] for _, t, n in cuts)
    # the workspace holds the partials of the plan made for the current device (or without one)
    slots = B.tf_paged_mla_plan_info(w.S, w.R, w.H, w.lens)["slots"]
    want = slots * 64 * 512 * 4 + (-(-(slots * 64 * 2 * 4) // 256)) * 256
    assert slots > 0 and B.tf_paged_mla_workspace_bytes(None, w.S, w.R, w.H, w.lens) == want


def test_unit_plan_ranges_cover_every_tile_once(L):
    """Mode 1 on small and ragged shapes: the ranges tile the units' numbering without gaps or
    overlaps, every range is non-empty, and short units are cut at tile granularity."""
    for lens, R, H, sms in [([1200, 700, 160], 160, 64, 152), ([3000, 400], 200, 16, 152),
                            ([5000], 300, 64, 7), ([300, 260, 256], 256, 64, 152), ([64] * 3, 64, 64, 152)]:
        pl = B.tf_paged_mla_plan_info(len(lens), R, H, lens, sms=sms)
        assert pl["mode"] == 1 and 1 <= pl["ctas"] == pl["nranges"] <= sms
        ranges, cuts, total = _unit_ranges(pl, lens, R, H)
        assert all(t > 0 for t, _ in ranges)
        assert sum(t for t, _ in ranges) == total
        assert pl["slots"] == (2 * pl["ctas"] if cuts else 0)


def test_invariant_splits_depend_on_the_stream_alone(L):
    """On a batch-invariant pool a stream's split is a function of its own length, R and H: the
    same in any batch, a multiple of 256 keys, and the items are the splits of every group."""
    from paged_mla_kv_gb300 import synth as Y
    w = Y.WORKLOADS["decode_batch"]()
    pl = B.tf_paged_mla_plan_info(w.S, w.R, w.H, w.lens, sms=152, invariant=True)
    assert pl["mode"] == 2
    sk = pl["split_keys"]
    for s in range(w.S):
        alone = B.tf_paged_mla_plan_info(1, w.R, w.H, w.lens[s:s + 1], sms=152, invariant=True)
        assert alone["split_keys"][0] == sk[s] and sk[s] % 256 == 0
        other = B.tf_paged_mla_plan_info(2, w.R, w.H, [int(w.lens[s]), 777], sms=7, invariant=True)
        assert other["split_keys"][0] == sk[s]
    nsplit = -(-w.lens // sk)
    assert pl["ctas"] == pl["work"] == int(np.sum(nsplit)) * pl["groups"]
    assert pl["slots"] == int(np.sum(nsplit[nsplit > 1])) * pl["groups"]
    # a prefill chunk with 128 or more column groups is one split
    p = Y.WORKLOADS["prefill_208k"]()
    pp = B.tf_paged_mla_plan_info(p.S, p.R, p.H, p.lens, invariant=True)
    assert pp["mode"] == 2 and pp["split_keys"][0] == p.lens[0] and pp["slots"] == 0


def test_plan_info_refuses_bad_sizes(L):
    lens = np.array([100, 200], np.int64)
    info = B.tf_attend_plan()
    lp = lens.ctypes.data_as(ctypes.c_void_p)
    assert L.tf_paged_mla_plan_info(2, 1, 129, lp, 0, 0, ctypes.byref(info), None, None) == B.TF_E_ARG
    assert L.tf_paged_mla_plan_info(0, 1, 16, lp, 0, 0, ctypes.byref(info), None, None) == B.TF_E_ARG
    assert L.tf_paged_mla_plan_info(2, 1, 16, lp, 0, 0, None, None, None) == B.TF_E_ARG
    assert L.tf_paged_mla_plan_info(2, 101, 16, lp, 0, 0, ctypes.byref(info), None, None) == B.TF_E_RANGE
    assert L.tf_paged_mla_plan_info(2, 1, 16, lp, 0, 0, ctypes.byref(info), None, None) == B.TF_OK


def test_plans_of_random_shapes_keep_their_invariants(L):
    """Random batches in both range modes: the bounds cover the numbering exactly once in
    non-empty ranges, there are at most as many ranges as SMs allow, and the plan has partial
    slots exactly when a bound cuts a unit (host arithmetic only)."""
    rng = np.random.default_rng(11)
    for _ in range(300):
        S = int(rng.integers(1, 40))
        sms = int(rng.choice([7, 64, 148, 152, 240]))
        if rng.random() < 0.5:
            R, H = int(rng.integers(1, 3)), int(rng.choice([8, 16, 64, 128]))
        else:
            R, H = int(rng.integers(40, 400)), int(rng.choice([16, 64]))
        lens = np.maximum(rng.integers(1, 40000, S), R).astype(np.int64)
        pl = B.tf_paged_mla_plan_info(S, R, H, lens, sms=sms)
        G = pl["groups"]
        b = pl["bounds"]
        if pl["mode"] == 0:
            tiles = -(-lens // 64)
            assert b[0] == 0 and b[-1] == tiles.sum() and np.all(np.diff(b) >= 1)
            assert pl["nranges"] * G == pl["ctas"] <= sms
            starts = np.concatenate([[0], np.cumsum(tiles)])
            cut = any(x not in set(starts.tolist()) for x in b[1:-1])
            assert pl["slots"] == (2 * pl["ctas"] if cut else 0)
        else:
            assert pl["mode"] == 1 and G * 4 > sms and pl["work"] == S * G
            ranges, cuts, total = _unit_ranges(pl, lens, R, H)
            assert 1 <= pl["ctas"] == pl["nranges"] <= sms
            assert all(t > 0 for t, _ in ranges) and sum(t for t, _ in ranges) == total
            assert b[0] == 0 and b[-1] == (S * G) << 32
            assert pl["slots"] == (2 * pl["ctas"] if cuts else 0)
