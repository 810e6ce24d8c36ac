"""GPU parity of the blocked top-k (tf_topk_blocked) against the oracle, through the C-ABI.

Columns and values must match the oracle bit for bit: the order (IEEE total order, ties by
column) makes the top-k unique.  Shapes span one block, a ragged second block, one and several
merge levels, k up to its maximum, ragged row lengths (empty, shorter than k, exactly k), a row
stride wider than the row, and the values that stress the order: heavy ties, all-equal rows,
NaN, signed zeros and infinities.  The integer rows put tens, hundreds or thousands of keys on
the k-th value of a block, so ties are settled by counting, by a radix pass over columns, and
by the path that re-reads the block when the keys near the k-th do not fit shared memory.
"""
import numpy as np
import pytest
import torch

from oracle import topk as OT
from paged_mla_kv_gb300 import binding as B
from paged_mla_kv_gb300 import build as BUILD
from paged_mla_kv_gb300 import synth as Y

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    BUILD.build()
    B.lib()


def values(kind: str, rows: int, n: int, seed: int) -> np.ndarray:
    g = np.random.default_rng(seed)
    if kind == "normal":
        return g.standard_normal((rows, n), dtype=np.float32)
    if kind == "grid":
        return Y.topk_logits(seed, range(rows), n)
    if kind == "few":
        return g.integers(0, 4, (rows, n)).astype(np.float32)
    if kind.startswith("int"):   # int<m>: integers below m, ~16384/m equal keys a block per value
        return g.integers(0, int(kind[3:]), (rows, n)).astype(np.float32)
    if kind == "const":
        return np.full((rows, n), 0.5, np.float32)
    if kind == "special":
        x = np.round(g.standard_normal((rows, n)) * 2).astype(np.float32) / 2
        sp = np.array([np.nan, 0.0, -0.0, np.inf, -np.inf], np.float32)
        m = g.random((rows, n)) < 0.2
        x[m] = g.choice(sp, int(m.sum()))
        return x
    raise ValueError(kind)


def run(x: np.ndarray, k: int, lens=None, ld: int | None = None):
    rows, n = x.shape
    ld = ld or (n + 3) // 4 * 4
    buf = torch.zeros((rows, ld), dtype=torch.float32)
    buf[:, :n] = torch.from_numpy(x)
    d = buf.cuda()
    dl = None if lens is None else torch.from_numpy(np.asarray(lens, np.int32)).cuda()
    ws_bytes = B.tf_topk_workspace_bytes(rows, n, k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") if ws_bytes else None
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    val = torch.empty((rows, k), dtype=torch.float32, device="cuda")
    B.tf_topk_blocked(d, k, idx, val, lens=dl, n=n, ws=ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), val.cpu().numpy()


def check(x, k, lens=None, ld=None):
    gi, gv = run(x, k, lens, ld)
    ri, rv = OT.topk_rows(x, k, lens)
    for r in range(x.shape[0]):
        assert np.array_equal(gi[r], ri[r]), f"row {r}: first differing rank {np.argmax(gi[r] != ri[r])}"
        assert np.array_equal(gv[r].view(np.uint32), rv[r].view(np.uint32)), f"row {r}: values differ"


CASES = [
    # rows, n, k, kind
    (3, 1, 1, "normal"),
    (4, 100, 7, "normal"),
    (5, 16384, 512, "grid"),
    (5, 16385, 512, "grid"),
    (3, 50000, 2048, "normal"),
    (2, 300000, 512, "grid"),
    (2, 600000, 2048, "grid"),
    (3, 40000, 512, "few"),
    (3, 40000, 512, "int32"),
    (3, 40000, 512, "int256"),
    (2, 40000, 2048, "int1000"),
    (2, 40000, 300, "const"),
    (4, 40000, 64, "special"),
    (2, 70000, 2048, "special"),
]


@pytest.mark.parametrize("rows,n,k,kind", CASES)
def test_topk_matches_oracle(rows, n, k, kind):
    check(values(kind, rows, n, seed=rows * 7 + n % 1000 + k), k)


def test_ragged_lengths():
    n, k = 40000, 512
    lens = [0, 1, 511, 512, 513, 16384, 16385, 39999, 40000, 12345]
    check(values("grid", len(lens), n, 11), k, lens=lens)


def test_lengths_are_clamped():
    x = values("normal", 3, 1000, 12)
    gi, _ = run(x, 16, lens=[-5, 5000, 10])
    ri, _ = OT.topk_rows(x, 16, [0, 1000, 10])
    assert np.array_equal(gi, ri)


def test_row_stride_wider_than_row():
    check(values("grid", 3, 20001, 13), 100, ld=20480)


def test_repeatable_bits():
    x = values("few", 4, 90000, 14)
    a = run(x, 1000)
    b = run(x, 1000)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))


def test_bad_arguments():
    d = torch.zeros((2, 64), dtype=torch.float32, device="cuda")
    idx = torch.empty((2, 8), dtype=torch.int32, device="cuda")
    val = torch.empty((2, 8), dtype=torch.float32, device="cuda")
    for k in (0, 2049):
        with pytest.raises(B.TFError):
            B.tf_topk_blocked(d, k, idx, val)
    with pytest.raises(B.TFError):          # misaligned base
        B.tf_topk_blocked(d[:, 1:], 8, idx, val)
    odd = torch.zeros((2, 63), dtype=torch.float32, device="cuda")
    with pytest.raises(B.TFError):          # row stride not a multiple of 4
        B.tf_topk_blocked(odd, 8, idx, val)
    big = torch.zeros((2, 40000), dtype=torch.float32, device="cuda")
    with pytest.raises(B.TFError):          # workspace missing
        B.tf_topk_blocked(big, 8, idx, val)
    B.tf_topk_blocked(d[:0], 8, idx[:0], val[:0])   # no rows: nothing to do, any pointers
    torch.cuda.synchronize()


def _ord(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> int64 keys in the IEEE total order (NaN lowest), for the full-size properties."""
    u = x.view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    neg = (u & 0x80000000) != 0
    k = torch.where(neg, (~u) & 0xFFFFFFFF, u | 0x80000000)
    return torch.where(torch.isnan(x), torch.zeros_like(k), k)


def test_full_size_prefill_chunk():
    """The 2,048 x 100,000 causal chunk at k = 512, launched as the benchmark launches it:
    sampled rows against the oracle, every row against the properties that fix a top-k."""
    w = Y.topk_prefill()
    x = Y.topk_logits(w.seed, range(w.rows), w.n)
    d = torch.from_numpy(x).cuda()
    lens = torch.from_numpy(w.lens).cuda()
    ws = torch.empty(B.tf_topk_workspace_bytes(w.rows, w.n, w.k), dtype=torch.uint8, device="cuda")
    idx = torch.empty((w.rows, w.k), dtype=torch.int32, device="cuda")
    val = torch.empty((w.rows, w.k), dtype=torch.float32, device="cuda")
    B.tf_topk_blocked(d, w.k, idx, val, lens=lens, ws=ws)
    torch.cuda.synchronize()
    gi, gv = idx.cpu().numpy(), val.cpu().numpy()
    for r in (0, 1, 513, 1024, 2046, 2047):
        ri, rv = OT.topk(x[r, : w.lens[r]], w.k)
        assert np.array_equal(gi[r], ri) and np.array_equal(gv[r].view(np.uint32), rv.view(np.uint32)), r
    # every row: columns in range and distinct, values copied, sorted, and exactly k-1 keys beat the last
    li = idx.long()
    assert bool((li >= 0).all()) and bool((li < lens[:, None]).all())
    assert bool((li.sort(1).values.diff(1) > 0).all())
    assert torch.equal(d.gather(1, li).view(torch.int32), val.view(torch.int32))
    kv = _ord(val)
    assert bool(((kv[:, :-1] > kv[:, 1:]) | ((kv[:, :-1] == kv[:, 1:]) & (li[:, :-1] < li[:, 1:]))).all())
    cols = torch.arange(w.n, device="cuda")
    live = cols[None, :] < lens[:, None]
    beat = torch.zeros(w.rows, dtype=torch.int64, device="cuda")
    for r0 in range(0, w.rows, 256):
        kx = _ord(d[r0:r0 + 256])
        last_k, last_c = kv[r0:r0 + 256, -1:], li[r0:r0 + 256, -1:]
        better = (kx > last_k) | ((kx == last_k) & (cols[None, :] < last_c))
        beat[r0:r0 + 256] = (better & live[r0:r0 + 256]).sum(1)
    assert bool((beat == w.k - 1).all())
