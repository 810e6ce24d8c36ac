"""GPU parity of attention over listed rows (tf_paged_mla_attend_sparse) against the
fp64 oracle's gathered-rows definition, through the C-ABI."""
import numpy as np
import pytest
import torch

from oracle import attend as OA
from paged_mla_kv_gb300 import binding as B
from paged_mla_kv_gb300 import build as BUILD
from paged_mla_kv_gb300 import synth as Y
from paged_mla_kv_gb300.harness import Resident
from tests.gpu_common import LSE_ABS, MAX_ABS, REL_L2, bits, no_device_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    BUILD.build()
    B.lib()


def run_sparse(res, w, lists):
    nidx = np.array([len(x) for x in lists], np.int32)
    idx = np.zeros((w.S, int(nidx.max())), np.int32)
    for s, x in enumerate(lists):
        idx[s, :len(x)] = x
    q = res.q()
    out = torch.empty((w.S, 1, w.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.S, 1, w.H), dtype=torch.float32, device="cuda")
    n = B.tf_paged_mla_sparse_workspace_bytes(res.pool, w.S, w.H, nidx)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda") if n else None
    B.tf_paged_mla_attend_sparse(res.pool, 0, res.pt, res.max_pages, res.lens, torch.from_numpy(idx).cuda(), nidx,
                                 q, w.scale, out, lse, ws)
    torch.cuda.synchronize()
    return out, lse


def check(w, out, lse, lists):
    qall = w.q(0)
    o = out.float().cpu().numpy().reshape(w.S, w.H, 512)
    lz = lse.float().cpu().numpy().reshape(w.S, w.H)
    for s, x in enumerate(lists):
        lat, rope = w.stream_rows(0, s)
        o_ref, l_ref = OA.attend_sparse(qall[s, 0], lat, rope, x, w.scale)
        got = o[s].astype(np.float64)
        assert np.all(np.isfinite(got)), f"stream {s}: non-finite output"
        ma = float(np.max(np.abs(got - o_ref)))
        rl = float(np.linalg.norm(got - o_ref) / max(np.linalg.norm(o_ref), 1e-30))
        le = float(np.max(np.abs(lz[s] - l_ref)))
        assert ma <= MAX_ABS and rl <= REL_L2 and le <= LSE_ABS, (s, ma, rl, le)


@pytest.mark.parametrize("H", [16, 64, 128])
def test_listed_rows_ragged_counts(H):
    # list lengths on and around the 64-key tile, a single row, and the pages' 2,048
    lens = [3000, 700, 9000, 66000, 130, 5000]
    counts = [1, 63, 64, 65, 130, 2048]
    w = Y.custom(f"sparse_H{H}", 300 + H, lens=lens, R=1, H=H)
    lists = [Y.listed_rows(7 + H, [L], n)[0] for L, n in zip(lens, counts)]
    res = Resident(w)
    out, lse = run_sparse(res, w, lists)
    no_device_error(res.pool)
    check(w, out, lse, lists)


def test_listed_rows_with_repeats_shared_pages_and_poison():
    lens = [9000, 4000, 6000]
    share = [(-1, 0), (0, 5), (0, 7)]
    w = Y.custom("sparse_share", 310, lens=lens, R=1, H=64, share=share)
    lists = Y.listed_rows(11, lens, 1500, repeats=True)
    res = Resident(w, poison=True)
    out, lse = run_sparse(res, w, lists)
    no_device_error(res.pool)
    check(w, out, lse, lists)


def test_listed_rows_paged_equals_windowed_and_repeat_bit_exact():
    lens = [5000, 800, 12000]
    w = Y.custom("sparse_pw", 320, lens=lens, R=1, H=64)
    lists = Y.listed_rows(12, lens, 700)
    r1 = Resident(w, windowed=False)
    o1, l1 = run_sparse(r1, w, lists)
    o1b, l1b = run_sparse(r1, w, lists)
    r2 = Resident(w, windowed=True)
    o2, l2 = run_sparse(r2, w, lists)
    assert np.array_equal(bits(o1), bits(o1b)) and torch.equal(l1, l1b)
    assert np.array_equal(bits(o1), bits(o2)) and torch.equal(l1, l2)
    check(w, o1, l1, lists)


def test_listed_rows_many_streams():
    lens = Y.listed_rows(3, [60000], 200)[0] + 1    # 200 lengths in [1, 60,000]
    lens = [int(x) for x in lens]
    w = Y.custom("sparse_many", 330, lens=lens, R=1, H=16)
    lists = Y.listed_rows(13, lens, 300)
    res = Resident(w)
    out, lse = run_sparse(res, w, lists)
    no_device_error(res.pool)
    check(w, out, lse, lists)


def test_listed_row_outside_the_stream_is_recorded_not_faulted():
    lens = [3000, 900]
    w = Y.custom("sparse_bad", 340, lens=lens, R=1, H=16)
    lists = Y.listed_rows(14, lens, 100)
    lists[1] = lists[1].copy()
    lists[1][37] = 900                                # one past the stream's last row
    res = Resident(w)
    run_sparse(res, w, lists)
    rc, detail = res.pool.last_error()
    assert rc == B.TF_E_DEVICE and detail == 900
    good = Y.listed_rows(14, lens, 100)
    out, lse = run_sparse(res, w, good)
    no_device_error(res.pool)
    check(w, out, lse, good)
