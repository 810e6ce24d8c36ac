"""The allocation-free attention entry point, called through the C-ABI.

tf_paged_mla_attend_static serves callers that cannot allocate device memory: it
keeps its split partials in the library's own device array instead of a
caller-provided workspace.  Its results must equal tf_paged_mla_attend's on the
same inputs, call after call, since the array keeps whatever the last call left.
This file is collected last so that a run stopping at the first failure has run
every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_mla_kv_gb300 import binding as B
from paged_mla_kv_gb300 import build as BUILD
from paged_mla_kv_gb300 import synth as Y
from paged_mla_kv_gb300.harness import Resident, bf16_tensor
from tests.gpu_common import MAX_ABS, REL_L2, bits, no_device_error

pytestmark = pytest.mark.gpu


def _static_call(res, q, out, lse):
    w = res.w
    lens = np.ascontiguousarray(res.lens, np.int64)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return B.lib().tf_paged_mla_attend_static(
        res.pool.handle, 0, ctypes.c_void_p(res.pt.data_ptr()), res.max_pages,
        lens.ctypes.data_as(ctypes.c_void_p), w.S, w.R, w.H, ctypes.c_void_p(q.data_ptr()),
        ctypes.c_float(w.scale), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), stream)


def test_static_scratch_matches_workspace_entry_point_twice():
    BUILD.build()
    w = Y.custom("noalloc", 77, lens=[9000, 3000, 65, 40000], R=2, H=64)
    res = Resident(w)
    need = B.tf_paged_mla_workspace_bytes(res.pool, w.S, w.R, w.H, w.lens)
    assert 0 < need <= B.TF_STATIC_WS_BYTES          # the case really uses scratch
    q1 = res.q()
    g = np.random.default_rng(3)
    q2 = bf16_tensor(Y.f32_to_bf16_bits(g.normal(0, 0.5, (w.S, w.R, w.H, 576)).astype(np.float32)))
    for q in (q1, q2):                                 # two calls in a row, different queries
        ref_out, ref_lse = res.attend(q)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        rc = _static_call(res, q, out, lse)
        assert rc == B.TF_OK
        torch.cuda.synchronize()
        no_device_error(res.pool)
        a, b = out.float(), ref_out.float()
        assert torch.isfinite(a).all()
        assert (a - b).abs().max().item() <= MAX_ABS
        assert ((a - b).norm() / b.norm()).item() <= REL_L2
        assert (lse - ref_lse).abs().max().item() <= 2e-3
        # the same kernels over the same bytes: identical bits
        assert np.array_equal(bits(out), bits(ref_out))
    # a third call of another shape: other streams and lengths move the range cuts and change
    # how many slots hold partials, so a slot that kept a stale partial would show here
    w3 = Y.custom("noalloc_shape", 80, lens=[70000, 5, 2100, 333, 12000], R=1, H=64)
    res3 = Resident(w3)
    need3 = B.tf_paged_mla_workspace_bytes(res3.pool, w3.S, w3.R, w3.H, w3.lens)
    assert 0 < need3 <= B.TF_STATIC_WS_BYTES
    q3 = res3.q()
    ref_out, ref_lse = res3.attend(q3)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    assert _static_call(res3, q3, out, lse) == B.TF_OK
    torch.cuda.synchronize()
    no_device_error(res3.pool)
    assert np.array_equal(bits(out), bits(ref_out))
    assert np.array_equal(bits(lse), bits(ref_lse))


def test_static_scratch_covers_every_default_launch():
    BUILD.build()
    # on a default pool, partials come only from units cut by a CTA range boundary, two
    # a CTA at most, so the scratch serves any batch: many long streams, a 1M-token
    # window, prefill chunks (ranges of key tiles over the chunk's units)
    cases = [(np.full(512, 65536, np.int64), 1, 64), (np.array([1 << 20] + [8192] * 7, np.int64), 2, 64),
             (np.array([102048], np.int64), 2048, 64), (np.array([209024], np.int64), 1024, 64),
             (np.full(64, 300000, np.int64), 2, 128)]
    for lens, R, H in cases:
        need = B.tf_paged_mla_workspace_bytes(None, len(lens), R, H, lens)
        assert need <= B.TF_STATIC_WS_BYTES
    assert B.tf_paged_mla_workspace_bytes(None, 512, 1, 64, cases[0][0]) > 0


def test_static_scratch_refuses_oversize_calls():
    BUILD.build()
    # a batch-invariant pool keeps one partial a split, so long batches outgrow the scratch
    w = Y.custom("noalloc_big", 78, lens=[100], R=1, H=64)
    res = Resident(w, invariant=True)
    huge = np.full(512, 65536, np.int64)
    assert B.tf_paged_mla_workspace_bytes(res.pool, 512, 1, 64, huge) > B.TF_STATIC_WS_BYTES
    before = B.tf_launch_count()
    rc = B.lib().tf_paged_mla_attend_static(
        res.pool.handle, 0, None, 128, huge.ctypes.data_as(ctypes.c_void_p), 512, 1, 64,
        ctypes.c_void_p(res.q().data_ptr()), ctypes.c_float(0.1), ctypes.c_void_p(res.q().data_ptr()), None,
        None)
    assert rc == B.TF_E_NOMEM
    assert B.tf_launch_count() == before


def test_static_entry_refuses_bad_arguments():
    BUILD.build()
    w = Y.custom("noalloc_bad", 79, lens=[100], R=1, H=64)
    res = Resident(w)
    lens = np.ascontiguousarray(res.lens, np.int64)
    before = B.tf_launch_count()
    rc = B.lib().tf_paged_mla_attend_static(
        res.pool.handle, 0, ctypes.c_void_p(res.pt.data_ptr()), res.max_pages, lens.ctypes.data_as(ctypes.c_void_p),
        1, 1, 64, ctypes.c_void_p(res.q().data_ptr()), ctypes.c_float(0.0), ctypes.c_void_p(res.q().data_ptr()),
        None, None)
    assert rc == B.TF_E_ARG
    assert B.tf_launch_count() == before
