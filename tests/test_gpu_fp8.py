"""GPU checks of FP8 pages (TF_POOL_FP8; issue #1313, step 1.3, item 3) through the C-ABI.

The append must store the oracle's codes, scales and rope bit for bit; attention must match the
oracle's attention over the dequantized rows within the attention tolerance; the kept-state copy
must move exactly the rows below `at`; poison must fill whole pages.
"""
import numpy as np
import pytest
import torch

from oracle import fp8 as F
from paged_mla_kv_gb300 import binding as B
from paged_mla_kv_gb300 import build as BUILD
from paged_mla_kv_gb300 import synth as Y
from paged_mla_kv_gb300.harness import Resident
from tests.gpu_common import bits, compare, no_device_error

pytestmark = pytest.mark.gpu

LAT_BYTES = 512 * 512
ROPE_OFF = LAT_BYTES + 512 * 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    BUILD.build()
    B.lib()


def page_fields(img: np.ndarray, cache: int, page: int):
    """(codes uint8[512][512], scales float32[512], rope uint16[512][64]) of one FP8 page."""
    pg = img[cache, page]
    codes = pg[:LAT_BYTES].reshape(512, 512)
    scales = pg[LAT_BYTES:ROPE_OFF].view(np.float32)
    rope = pg[ROPE_OFF:].view(np.uint16).reshape(512, 64)
    return codes, scales, rope


def run(w, **kw):
    res = Resident(w, fp8=True, **kw)
    out, lse = res.attend(res.q())
    torch.cuda.synchronize()
    no_device_error(res.pool)
    return res, out, lse


def test_append_stores_the_oracle_codes_scales_and_rope():
    w = Y.custom("f8app", 61, lens=[1000, 513, 7], R=1, H=16, num_caches=2)
    res = Resident(w, fp8=True, poison=True)
    img = res.pool.bytes_view().cpu().numpy()
    for c in range(2):
        for s in range(w.S):
            lat, rope = w.stream_rows(c, s)
            want_c, want_s = F.quantize_rows(Y.bf16_bits_to_f32(lat))
            L = int(w.lens[s])
            for j in range(-(-L // 512)):
                codes, scales, rp = page_fields(img, c, int(res.pt_host[s, j]))
                n = min(512, L - 512 * j)
                assert np.array_equal(codes[:n], want_c[512 * j:512 * j + n]), (c, s, j)
                assert np.array_equal(scales[:n].view(np.uint32), want_s[512 * j:512 * j + n].view(np.uint32))
                assert np.array_equal(rp[:n], rope[512 * j:512 * j + n])
                # rows past the length keep the poison (0xFF bytes)
                assert (codes[n:] == 0xFF).all() and (scales[n:].view(np.uint32) == 0xFFFFFFFF).all()
                assert (rp[n:] == 0xFFFF).all()
    no_device_error(res.pool)


def test_zero_rows_store_zero_scale():
    pool = B.KVPool(1, 2, poison=True, fp8=True)
    pt = torch.from_numpy(pool.take(1)[None].astype(np.int32)).cuda()
    lat = torch.zeros((1, 3, 512), dtype=torch.bfloat16, device="cuda")
    lat[0, 1, 7] = -2.5
    rope = torch.ones((1, 3, 64), dtype=torch.bfloat16, device="cuda")
    B.tf_paged_append(pool, 0, pt, 1, np.array([0], np.int64), lat, rope)
    torch.cuda.synchronize()
    codes, scales, _ = page_fields(pool.bytes_view().cpu().numpy(), 0, int(pt[0, 0]))
    assert scales[0] == 0 and scales[2] == 0 and not codes[0].any() and not codes[2].any()
    assert scales[1] == np.float32(2.5) / np.float32(448) and codes[1, 7] == 0xFE and not np.delete(codes[1], 7).any()


@pytest.mark.parametrize("R,H", [(1, 16), (1, 64), (2, 64), (1, 128)])
def test_attention_matches_oracle_over_dequantized_rows(R, H):
    lens = [2, 65, 511, 513, 1000, 4097]
    w = Y.custom(f"f8att_{R}_{H}", 62 + R + H, lens=lens, R=R, H=H)
    _, out, lse = run(w)
    compare(w, out, lse, fp8=True)


def test_shared_prefix_pages_and_a_prefill_chunk():
    w = Y.custom("f8share", 63, lens=[3000, 2600, 700], R=1, H=64, share=[(-1, 0), (0, 4), (0, 1)])
    _, out, lse = run(w)
    compare(w, out, lse, fp8=True)
    wp = Y.custom("f8prefill", 64, lens=[2000], R=96, H=16)
    _, out, lse = run(wp)
    compare(wp, out, lse, fp8=True, items_per_stream=[np.arange(0, 96 * 16, 37)])


@pytest.mark.parametrize("invariant", [False, True])
def test_paged_equals_windowed_and_repeats_bit_exact(invariant):
    w = Y.custom("f8pw", 65, lens=[3000, 700, 5000], R=2, H=64)
    res, o1, l1 = run(w, invariant=invariant)
    _, o2, l2 = run(w, windowed=True, invariant=invariant)
    assert np.array_equal(bits(o1), bits(o2)) and np.array_equal(l1.cpu().numpy(), l2.cpu().numpy())
    o3, l3 = res.attend(res.q())
    torch.cuda.synchronize()
    assert np.array_equal(bits(o1), bits(o3)) and np.array_equal(l1.cpu().numpy(), l3.cpu().numpy())


@pytest.mark.parametrize("at", [1, 511, 700, 1024])
def test_state_copy_moves_only_rows_below_at(at):
    w = Y.custom("f8copy", 66, lens=[1600], R=1, H=16, num_caches=3, pool_pages=12)
    res = Resident(w, fp8=True, poison=True)
    pages = -(-at // 512)
    dst = res.pool.take(pages)
    src_t = torch.from_numpy(res.pt_host[0, :pages].copy()).cuda()
    dst_t = torch.from_numpy(dst.copy()).cuda()
    before = res.pool.bytes_view().cpu().numpy().copy()
    B.tf_state_copy_rows(res.pool, -1, src_t, dst_t, at)
    after = res.pool.bytes_view().cpu().numpy()
    want = before.copy()
    for c in range(3):
        for j in range(pages):
            n = min(512, at - 512 * j)
            sp, dp = int(res.pt_host[0, j]), int(dst[j])
            want[c, dp, :n * 512] = before[c, sp, :n * 512]
            want[c, dp, LAT_BYTES:LAT_BYTES + 4 * n] = before[c, sp, LAT_BYTES:LAT_BYTES + 4 * n]
            want[c, dp, ROPE_OFF:ROPE_OFF + 128 * n] = before[c, sp, ROPE_OFF:ROPE_OFF + 128 * n]
    assert np.array_equal(after, want)
    no_device_error(res.pool)


def test_poison_fills_whole_fp8_pages():
    pool = B.KVPool(2, 3, poison=True, fp8=True)
    ids = pool.take(2)
    torch.cuda.synchronize()
    img = pool.bytes_view().cpu().numpy()
    assert img.shape[-1] == B.PAGE_BYTES_FP8
    for p in ids:
        assert (img[:, int(p)] == 0xFF).all()


def test_invariant_pool_workspace_and_static_call():
    # a batch-invariant FP8 pool: attention expands the rows into the workspace first
    w = Y.custom("f8err", 67, lens=[900, 40], R=1, H=16)
    res = Resident(w, fp8=True, invariant=True)
    q = res.q()
    out = torch.empty((w.S, 1, w.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.S, 1, w.H), dtype=torch.float32, device="cuda")
    need = B.tf_paged_mla_workspace_bytes(res.pool, w.S, 1, w.H, res.lens)
    assert need >= 2 * 589824   # the expanded pages of both streams
    small = torch.empty(need - 4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.TFError) as e:
        B.tf_paged_mla_attend(res.pool, 0, res.pt, res.max_pages, res.lens, q, w.scale, out, lse, small)
    assert e.value.code == -3
    with pytest.raises(B.TFError) as e:
        B.tf_paged_mla_attend_static(res.pool, 0, res.pt, res.max_pages, res.lens, q, w.scale, out, lse)
    assert e.value.code == -6
    # on a default FP8 pool the codes are expanded in the kernel: no extra workspace, and the
    # call that needs no workspace works
    res2 = Resident(w, fp8=True)
    assert B.tf_paged_mla_workspace_bytes(res2.pool, w.S, 1, w.H, res2.lens) == \
        B.tf_paged_mla_workspace_bytes(None, w.S, 1, w.H, res2.lens)
    B.tf_paged_mla_attend_static(res2.pool, 0, res2.pt, res2.max_pages, res2.lens, res2.q(), w.scale, out, lse)
    torch.cuda.synchronize()
    compare(w, out, lse, fp8=True)
    no_device_error(res.pool)


@pytest.mark.parametrize("R,H", [(1, 64), (2, 64), (64, 64)])
def test_fp8_attention_is_bf16_attention_over_the_expanded_rows(R, H):
    """The kernel reads FP8 codes and expands them to bf16(code * scale) in shared memory, then
    runs the BF16 pipeline: so it must equal, bit for bit, the BF16 attention over a pool that
    holds those bf16 values.  R = 64 at 64 heads runs the prefill plan (ranges over
    (stream, row) units), the others ranges of key tiles shared by the column groups."""
    lens = [700, 3000, 65]
    share = [(-1, 0), (0, 1), (-1, 0)]   # the owner's first page is full (700 rows)
    w8 = Y.custom(f"f8eq_{R}", 68 + R, lens=lens, R=R, H=H, share=share)
    wb = Y.custom(f"f8eq_{R}", 68 + R, lens=lens, R=R, H=H, share=share)
    orig = wb.page_rows

    def expanded(c, s, p):
        lat, rope = orig(c, s, p)
        codes, scales = F.quantize_rows(Y.bf16_bits_to_f32(lat))
        vals = F.decode_table()[codes].astype(np.float32) * scales[:, None]   # fp32 product, rounded
        return Y.f32_to_bf16_bits(vals.astype(np.float32)), rope

    wb.page_rows = expanded
    _, o8, l8 = run(w8)
    rb = Resident(wb)
    ob, lb = rb.attend(rb.q())
    torch.cuda.synchronize()
    no_device_error(rb.pool)
    assert np.array_equal(bits(o8), bits(ob))
    assert np.array_equal(l8.cpu().numpy().view(np.uint32), lb.cpu().numpy().view(np.uint32))


def run_sparse8(res, w, lists):
    nidx = np.array([len(x) for x in lists], np.int32)
    idx = np.zeros((w.S, int(nidx.max())), np.int32)
    for s, x in enumerate(lists):
        idx[s, :len(x)] = x
    q = res.q()[:, 0]
    out = torch.empty((w.S, w.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.S, w.H), dtype=torch.float32, device="cuda")
    n = B.tf_paged_mla_sparse_workspace_bytes(res.pool, w.S, w.H, nidx)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda") if n else None
    B.tf_paged_mla_attend_sparse(res.pool, 0, res.pt, res.max_pages, res.lens, torch.from_numpy(idx).cuda(), nidx,
                                 q, w.scale, out, lse, ws)
    torch.cuda.synchronize()
    no_device_error(res.pool)
    return out, lse


@pytest.mark.parametrize("H", [16, 64])
def test_listed_rows_on_fp8_pages(H):
    """Listed-row attention gathers codes, scales and rope rows of an FP8 pool: against the
    oracle over the dequantized rows, and bit for bit against the BF16 pool that holds
    bf16(code * scale)."""
    from oracle import attend as OA
    lens = [5000, 700, 64, 3000]
    w8 = Y.custom(f"f8sp_{H}", 80 + H, lens=lens, R=1, H=H)
    wb = Y.custom(f"f8sp_{H}", 80 + H, lens=lens, R=1, H=H)
    orig = wb.page_rows

    def expanded(c, s, p):
        lat, rope = orig(c, s, p)
        codes, scales = F.quantize_rows(Y.bf16_bits_to_f32(lat))
        vals = F.decode_table()[codes].astype(np.float32) * scales[:, None]
        return Y.f32_to_bf16_bits(vals.astype(np.float32)), rope

    wb.page_rows = expanded
    lists = Y.listed_rows(90 + H, lens, 300, repeats=True)
    r8 = Resident(w8, fp8=True)
    o8, l8 = run_sparse8(r8, w8, lists)
    rb = Resident(wb)
    ob, lb = run_sparse8(rb, wb, lists)
    assert np.array_equal(bits(o8), bits(ob))
    assert np.array_equal(l8.cpu().numpy().view(np.uint32), lb.cpu().numpy().view(np.uint32))
    qall = w8.q(0)
    o = o8.float().cpu().numpy()
    for s, x in enumerate(lists):
        lat, rope = w8.stream_rows(0, s)
        deq = F.dequantize_rows(*F.quantize_rows(Y.bf16_bits_to_f32(lat)))
        ref, lref = OA.attend_sparse(qall[s, 0], deq, rope, x, w8.scale)
        assert float(np.max(np.abs(o[s] - ref))) <= 2e-3, s
        assert float(np.max(np.abs(l8.cpu().numpy()[s] - lref))) <= 2e-3, s
