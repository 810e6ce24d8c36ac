"""GPU parity of the CUDA path against the oracle, through the C-ABI.

Append and kept-state copy are compared byte for byte with the oracle's pool
image; attention within max-abs 2e-3 / relative-L2 1e-2 of the fp64 oracle.
"""
import numpy as np
import pytest
import torch

from oracle import paged as OG
from paged_mla_kv_gb300 import binding as B
from paged_mla_kv_gb300 import build as BUILD
from paged_mla_kv_gb300 import synth as Y
from paged_mla_kv_gb300.harness import Resident, bf16_tensor
from tests.gpu_common import bits, compare, no_device_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    BUILD.build()
    B.lib()


def pool_image(res: Resident) -> np.ndarray:
    torch.cuda.synchronize()
    return bits(res.pool.view()).reshape(res.pool.num_caches, res.pool.num_pages, OG.PAGE_WORDS)


# ---------------------------------------------------------------- append / copy


@pytest.mark.parametrize("windowed", [False, True])
def test_append_is_bit_exact(windowed):
    w = Y.custom("append", 11, lens=[1, 511, 512, 513, 1700], R=1, H=16, num_caches=2,
                 share=[(-1, 0), (-1, 0), (-1, 0), (2, 1), (-1, 0)])
    if windowed:
        w.share = [(-1, 0)] * w.S
    res = Resident(w, poison=True, windowed=windowed)
    img = pool_image(res)
    want = OG.new_pool(w.num_caches, res.pool.num_pages)
    pt = res.pt_host
    for c in range(w.num_caches):
        for s in range(w.S):
            lo = 0 if windowed else w.shared_pages(s) * 512
            lat, rope = w.stream_rows(c, s, lo, int(w.lens[s]))
            OG.append(want, c, None if windowed else pt[s:s + 1], res.max_pages if not windowed else
                      res.max_pages * w.S, [lo + (s * res.max_pages * 512 if windowed else 0)],
                      lat[None], rope[None])
    # pages never taken are not compared (their content is the allocator's); taken ones are, in full
    taken = np.unique(pt[pt >= 0])
    assert np.array_equal(img[:, taken], want[:, taken])
    no_device_error(res.pool)


def test_append_many_streams_one_call_and_bad_page():
    w = Y.custom("append2", 12, lens=[700, 1300, 90], R=1, H=16)
    res = Resident(w, poison=True)
    # append 3 more rows to every stream in one call
    n = 3
    g = np.random.default_rng(1)
    lat = g.integers(0, 0x7F00, (w.S, n, 512)).astype(np.uint16)
    rope = g.integers(0, 0x7F00, (w.S, n, 64)).astype(np.uint16)
    before = pool_image(res)
    pos = np.array([10, 1100, 50], np.int64)
    B.tf_paged_append(res.pool, 0, res.pt, res.max_pages, pos, bf16_tensor(lat), bf16_tensor(rope))
    after = pool_image(res)
    OG.append(before, 0, res.pt_host, res.max_pages, pos, lat, rope)
    assert np.array_equal(after, before)
    no_device_error(res.pool)
    # a table entry outside the pool is recorded, and the row skipped
    bad = res.pt.clone()
    bad[1, 2] = 10_000
    B.tf_paged_append(res.pool, 0, bad, res.max_pages, np.array([0, 1030, 0], np.int64),
                      bf16_tensor(lat[:, :1]), bf16_tensor(rope[:, :1]))
    rc, detail = res.pool.last_error()
    assert rc == B.TF_E_DEVICE and detail == 10_000
    assert res.pool.last_error()[0] == 0     # reading clears it


@pytest.mark.parametrize("at", [1, 511, 512, 1000, 1536])
def test_state_copy_moves_only_rows_below_at(at):
    w = Y.custom("copy", 13, lens=[1600], R=1, H=16, num_caches=3, pool_pages=12)
    res = Resident(w, poison=True)
    pages = -(-at // 512)
    dst = res.pool.take(pages, stream=None)
    before = pool_image(res)
    src_t = torch.from_numpy(res.pt_host[0, :pages].copy()).cuda()
    dst_t = torch.from_numpy(dst.copy()).cuda()
    for cache in (-1, 1):
        B.tf_state_copy_rows(res.pool, cache, src_t, dst_t, at)
        after = pool_image(res)
        want = before.copy()
        OG.state_copy_rows(want, cache, res.pt_host[0, :pages], dst, at)
        assert np.array_equal(after, want)
        before = after
    no_device_error(res.pool)


# ---------------------------------------------------------------- attention


def run(w, **kw):
    res = Resident(w, **kw)
    out, lse = res.attend(res.q())
    torch.cuda.synchronize()
    no_device_error(res.pool)
    return res, out, lse


def test_tiny_decode_full_size():
    w = Y.tiny_decode()
    _, out, lse = run(w)
    compare(w, out, lse)


@pytest.mark.parametrize("H", [8, 16, 64, 128])
@pytest.mark.parametrize("R", [1, 2])
def test_decode_ragged_lengths(H, R):
    lens = [2, 63, 64, 65, 511, 513, 1000, 4097]
    w = Y.custom(f"ragged_H{H}_R{R}", 100 + H + R, lens=lens, R=R, H=H)
    _, out, lse = run(w)
    compare(w, out, lse)


@pytest.mark.parametrize("R,H", [(1, 64), (2, 128)])
def test_decode_ragged_lengths_batch_invariant_pool(R, H):
    lens = [2, 63, 64, 65, 511, 513, 1000, 4097, 70000]
    w = Y.custom(f"ragged_inv_H{H}_R{R}", 200 + H + R, lens=lens, R=R, H=H)
    _, out, lse = run(w, invariant=True)
    compare(w, out, lse)


@pytest.mark.parametrize("variant", ["sharp", "ramp"])
def test_decode_score_distributions(variant):
    kw = dict(q_std=1.0, scale=0.5) if variant == "sharp" else dict(ramp=60.0)
    w = Y.custom(f"dist_{variant}", 21, lens=[3000, 9000, 700], R=2, H=32, **kw)
    _, out, lse = run(w)
    compare(w, out, lse)


def test_decode_long_split_stream():
    w = Y.custom("long", 22, lens=[70000, 40], R=1, H=64)
    _, out, lse = run(w)
    compare(w, out, lse)


@pytest.mark.parametrize("T,L,H", [(64, 1000, 16), (300, 700, 8), (256, 3000, 64)])
def test_prefill_chunk(T, L, H):
    w = Y.chunked_prefill(seed=30 + T, T=T, L=L, H=H)
    _, out, lse = run(w)
    compare(w, out, lse)


def _lens(seed, n, lo, hi):
    return np.random.default_rng(seed).integers(lo, hi + 1, n).tolist()


# Batches shaped to reach every branch of the work plan: many short streams (CTAs walking
# several segments, with query reloads and mid-range epilogues), the most streams and heads
# the API takes, column groups side by side (2, 4 and 10 groups, ragged last group), ranges
# over (stream, column group) units (prefill-like, several streams; 64 and 16 heads, so a group
# is one row or four), and the batch-invariant split plan.
PLAN_SHAPES = [
    ("segments", 60, _lens(60, 200, 1, 600), 1, 8, False),
    ("max_streams", 61, _lens(61, 512, 1, 300), 1, 16, False),
    ("max_heads_r2", 62, [5000, 17, 900, 12000], 2, 128, False),
    ("ragged_groups", 63, [3000, 40, 700], 5, 24, False),
    ("ten_groups", 64, [2500, 1300], 40, 16, False),
    ("units", 65, [1200, 700, 160], 160, 64, False),
    ("units_h16", 69, [3000, 400], 200, 16, False),
    ("invariant_groups", 66, [5000, 17, 900, 12000], 2, 128, True),
    ("invariant_units", 67, [1200, 700, 160], 160, 64, True),
]


@pytest.mark.parametrize("name,seed,lens,R,H,invariant", PLAN_SHAPES, ids=[x[0] for x in PLAN_SHAPES])
def test_work_plan_shapes(name, seed, lens, R, H, invariant):
    lens = [max(int(x), R) for x in lens]
    w = Y.custom(name, seed, lens=lens, R=R, H=H)
    _, out, lse = run(w, invariant=invariant)
    compare(w, out, lse)


# ---------------------------------------------------------------- invariants


@pytest.mark.parametrize("invariant", [False, True])
def test_paged_equals_windowed_bit_exact(invariant):
    lens = [3000, 700, 5000]
    w = Y.custom("pw", 40, lens=lens, R=2, H=64)
    _, o1, l1 = run(w, windowed=False, invariant=invariant)
    _, o2, l2 = run(w, windowed=True, invariant=invariant)
    assert np.array_equal(bits(o1), bits(o2)) and np.array_equal(l1.cpu().numpy(), l2.cpu().numpy())


def test_pool_permutation_invariance_bit_exact():
    w = Y.custom("perm", 41, lens=[2500, 9000], R=1, H=64, pool_pages=40)
    _, o1, l1 = run(w, pool_seed=1)
    _, o2, l2 = run(w, pool_seed=987654)
    assert np.array_equal(bits(o1), bits(o2)) and np.array_equal(l1.cpu().numpy(), l2.cpu().numpy())


def test_poison_is_never_read():
    # NaN in every taken page before the writes, and in rows past each length
    w = Y.custom("poison", 42, lens=[777, 1025, 64], R=2, H=16)
    _, o1, l1 = run(w, poison=True)
    _, o2, l2 = run(w, poison=False)
    assert torch.isfinite(o1.float()).all() and torch.isfinite(l1).all()
    assert np.array_equal(bits(o1), bits(o2)) and np.array_equal(l1.cpu().numpy(), l2.cpu().numpy())


def _rel_l2(a: torch.Tensor, b: torch.Tensor) -> float:
    a, b = a.double(), b.double()
    return ((a - b).norm() / b.norm()).item()


def test_concurrent_matches_solo():
    # a stream attended inside a batch or alone: the work is dealt out differently (the
    # CTA ranges follow the whole batch), so the sums run in another order; each output
    # matches the oracle, and the two outputs match each other, in max-abs and in rel-L2
    lens = [5000, 130, 20000, 2]
    w = Y.custom("conc", 43, lens=lens, R=2, H=64)
    _, ob, lb = run(w)
    compare(w, ob, lb)
    qb = w.q()
    for s in [0, 2, 3]:
        ws = Y.custom("solo", 43, lens=[lens[s]], R=2, H=64)
        # same values: the solo stream's pages and queries must be the batch stream's
        ws.page_rows = lambda c, ss, p, _s=s: w.page_rows(c, _s, p)
        ws.q = lambda cache=0, _s=s: qb[_s:_s + 1]
        res = Resident(ws)
        out, lse = res.attend(bf16_tensor(qb[s:s + 1]))
        torch.cuda.synchronize()
        compare(ws, out, lse)
        assert (out[0].float() - ob[s].float()).abs().max().item() <= 2e-3
        assert _rel_l2(out[0].float(), ob[s].float()) <= 1e-2
        assert (lse[0] - lb[s]).abs().max().item() <= 2e-3


def test_concurrent_equals_solo_bit_exact_on_a_batch_invariant_pool():
    # splits depend on a stream's own length only, merged in split order: a stream's
    # bits are the same alone and inside any batch
    lens = [5000, 130, 20000, 2]
    w = Y.custom("conc_inv", 43, lens=lens, R=2, H=64)
    _, ob, lb = run(w, invariant=True)
    compare(w, ob, lb)
    for s in [0, 2, 3]:
        ws = Y.custom("solo_inv", 43, lens=[lens[s]], R=2, H=64)
        ws.page_rows = lambda c, ss, p, _s=s: w.page_rows(c, _s, p)
        qb = w.q()
        res = Resident(ws, invariant=True)
        out, lse = res.attend(bf16_tensor(qb[s:s + 1]))
        torch.cuda.synchronize()
        assert np.array_equal(bits(out[0]), bits(ob[s]))
        assert np.array_equal(lse[0].cpu().numpy(), lb[s].cpu().numpy())


def test_resumed_equals_fresh_bit_exact():
    # keep the first `at` rows into fresh pages, append the rest after them, attend
    L, at = 6000, 2048 + 300
    w = Y.custom("resume", 44, lens=[L], R=1, H=64, pool_pages=40)
    res, o_fresh, l_fresh = run(w)
    pages_at = -(-at // 512)
    total = -(-L // 512)
    new = res.pool.take(total)
    B.tf_state_copy_rows(res.pool, -1, torch.from_numpy(res.pt_host[0, :pages_at].copy()).cuda(),
                         torch.from_numpy(new[:pages_at].copy()).cuda(), at)
    res.pt = torch.from_numpy(new[None, :].copy()).cuda()
    res.pt_host = new[None, :].copy()
    res.append_rows(0, 0, at, L)
    out, lse = res.attend(res.q())
    torch.cuda.synchronize()
    no_device_error(res.pool)
    assert np.array_equal(bits(out), bits(o_fresh)) and np.array_equal(lse.cpu().numpy(), l_fresh.cpu().numpy())


@pytest.mark.parametrize("variant", ["plain", "sharp"])
def test_drafted_row_equals_plain_decode(variant):
    # PR #1732's lookahead of 1: the draft row of an R = 2 decode at length L sees keys
    # 0..L-2, exactly what an R = 1 decode at length L - 1 sees.  Both outputs match the
    # oracle and each other in max-abs and rel-L2.  With near-uniform weights one key too
    # many or too few moves the row by about 1/sqrt(L) = 1.7% in rel-L2, so the rel-L2
    # checks are the ones that would catch an off-by-one causal limit.
    L = 3333
    kw = dict(q_std=1.0, scale=0.5) if variant == "sharp" else {}
    w2 = Y.custom("draft", 45, lens=[L], R=2, H=64, **kw)
    _, o2, l2 = run(w2)
    compare(w2, o2, l2)
    w1 = Y.custom("plain", 45, lens=[L - 1], R=1, H=64, **kw)
    w1.page_rows = w2.page_rows
    q2 = w2.q()
    w1.q = lambda cache=0: q2[:, :1]
    res = Resident(w1)
    o1, l1 = res.attend(bf16_tensor(q2[:, :1]))
    torch.cuda.synchronize()
    compare(w1, o1, l1)
    d = (o1[0, 0].float() - o2[0, 0].float()).abs().max().item()
    assert d <= 2e-3
    assert _rel_l2(o1[0, 0].float(), o2[0, 0].float()) <= 1e-2
    assert (l1[0, 0] - l2[0, 0]).abs().max().item() <= 2e-3


def test_bad_page_table_is_recorded_not_faulted():
    w = Y.custom("badpt", 46, lens=[3000], R=1, H=16)
    res = Resident(w)
    bad = res.pt.clone()
    bad[0, 3] = 1 << 20
    out = torch.zeros((1, 1, 16, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 16), dtype=torch.float32, device="cuda")
    B.tf_paged_mla_attend(res.pool, 0, bad, res.max_pages, res.lens, res.q(), w.scale, out, lse, res.workspace())
    rc, detail = res.pool.last_error()
    assert rc == B.TF_E_DEVICE and detail == 1 << 20
    # the pool stays usable
    out2, lse2 = res.attend(res.q())
    torch.cuda.synchronize()
    no_device_error(res.pool)
    compare(w, out2, lse2)


def test_repeated_calls_are_bit_identical():
    # the kernels are deterministic: a race between pipeline roles shows up as a call
    # whose bits differ from the others (a wait passing early, a buffer read too soon)
    lens = [2, 63, 64, 65, 511, 513, 1000, 4097, 70000]
    w = Y.custom("repeat", 47, lens=lens, R=2, H=64)
    res = Resident(w)
    q, ws = res.q(), res.workspace()
    o0, l0 = res.attend(q, ws=ws)
    torch.cuda.synchronize()
    compare(w, o0, l0)
    ref = bits(o0)
    for _ in range(30):
        o, l = res.attend(q, ws=ws)
        torch.cuda.synchronize()
        assert np.array_equal(bits(o), ref) and torch.equal(l, l0)
    no_device_error(res.pool)


@pytest.mark.parametrize("name", ["tiny_decode", "decode_batch"])
def test_step_captured_in_a_cuda_graph_replays_bit_exact(name):
    # a serving loop may capture its decode step (append, attention and combine) into a CUDA
    # graph: every call takes its plan from host arrays and launches on the given stream only,
    # so a replay must give the eager call's bits
    w = Y.WORKLOADS[name]()
    res = Resident(w)
    q, ws, cur = res.q(), res.workspace(), res.current_rows(0)
    out = torch.empty((w.S, w.R, w.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.S, w.R, w.H), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def step():
        res.append_current(0, *cur)
        B.tf_paged_mla_attend(res.pool, 0, res.pt, res.max_pages, res.lens, q, w.scale, out, lse, ws)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    compare(w, out, lse)
    ref, ref_l = bits(out), lse.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for _ in range(3):
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), ref) and torch.equal(lse, ref_l)
    no_device_error(res.pool)


def test_bounded_wait_gives_up_and_the_context_survives():
    # a wait on a barrier that nothing completes must end, record TF_E_TIMEOUT, and leave
    # the context usable for the next call
    w = Y.custom("timeout", 48, lens=[1500], R=1, H=16)
    res = Resident(w)
    B.tf_diag_wait_timeout(res.pool, 1 << 20)
    rc, detail = res.pool.last_error()
    assert rc == B.TF_E_TIMEOUT and detail == 99
    out, lse = res.attend(res.q())
    torch.cuda.synchronize()
    no_device_error(res.pool)
    compare(w, out, lse)
