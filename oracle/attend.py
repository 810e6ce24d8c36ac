"""Attention over contiguous latent rows in fp64 -- TEST INFRASTRUCTURE ONLY.

Thin ctypes wrapper over ``mla_oracle.c`` (see that file for the definition it
follows: absorbed-query attention over one shared latent, issue #1313 "Step 2"
decode bullet and issue #1142 "What happens now"; causal rows per PR #1732
"What this changes" and the chunked-prefill note, section 1).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.oracle_mla_attend.restype = ctypes.c_int
        lib.oracle_mla_attend.argtypes = [
            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_double, ctypes.c_int32, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
        lib.oracle_mla_attend_f64.restype = ctypes.c_int
        lib.oracle_mla_attend_f64.argtypes = lib.oracle_mla_attend.argtypes
        _lib = lib
    return _lib


def default_threads() -> int:
    return int(os.environ.get("ORACLE_THREADS", os.cpu_count() or 1))


def attend_stream(q: np.ndarray, lat: np.ndarray, rope: np.ndarray, scale: float,
                  items=None, threads: int | None = None):
    """Attention of one stream.

    q: bf16 bits [R][H][576]; lat: [len][512] bf16 bits, or float64 values (the dequantized
    rows of FP8 pages, oracle.fp8); rope: [len][64] bf16 bits (contiguous rows).
    items: iterable of r*H + h (default: all).  Returns (out [n][512], lse [n]) in float64.
    """
    lib = _load()
    q = np.ascontiguousarray(q, np.uint16)
    f64 = np.asarray(lat).dtype == np.float64   # dequantized FP8 rows: the latent as doubles
    lat = np.ascontiguousarray(lat, np.float64 if f64 else np.uint16)
    rope = np.ascontiguousarray(rope, np.uint16)
    R, H, dk = q.shape
    assert dk == 576 and lat.shape[1] == 512 and rope.shape[1] == 64 and lat.shape[0] == rope.shape[0]
    n = lat.shape[0]
    if items is None:
        items = np.arange(R * H, dtype=np.int32)
    items = np.ascontiguousarray(np.asarray(items, np.int32))
    out = np.zeros((len(items), 512), np.float64)
    lse = np.zeros(len(items), np.float64)
    if len(items) == 0:
        return out, lse
    fn = lib.oracle_mla_attend_f64 if f64 else lib.oracle_mla_attend
    rc = fn(n, R, H, q.ctypes.data, lat.ctypes.data, rope.ctypes.data,
                               float(scale), len(items), items.ctypes.data,
                               out.ctypes.data, lse.ctypes.data,
                               threads if threads is not None else default_threads())
    if rc != 0:
        raise ValueError("oracle_mla_attend rejected its arguments")
    return out, lse


def attend_sparse(q: np.ndarray, lat: np.ndarray, rope: np.ndarray, idx, scale: float,
                  threads: int | None = None):
    """Attention of one query row over listed rows of a stream.

    Issue #1313, step 2: a sparse decode row touches at most 2,048 latent rows; issue #1142,
    "What stays as it is": the sparse path reads the same rows.  The keys are the rows
    idx[0..n) in list order (a row listed twice counts twice), so this is the contiguous
    definition above applied to the gathered rows.
    q: bf16 bits [H][576]; lat: [len][512]; rope: [len][64]; idx: n row numbers in [0, len).
    Returns (out [H][512], lse [H]) in float64.
    """
    idx = np.asarray(idx, np.int64)
    assert idx.ndim == 1 and len(idx) >= 1 and idx.min() >= 0 and idx.max() < lat.shape[0]
    return attend_stream(np.asarray(q)[None], np.asarray(lat)[idx], np.asarray(rope)[idx], scale, threads=threads)


def attend_workload(w, cache: int = 0, items_per_stream=None, threads: int | None = None, fp8: bool = False):
    """Oracle outputs for every stream of a synth.Workload.

    items_per_stream: None (all r*H+h) or a list of per-stream item arrays.  fp8: attend over
    the rows quantized as an FP8 pool stores them.
    Returns a list of (items, out, lse) per stream.
    """
    qall = w.q(cache)
    res = []
    for s in range(w.S):
        lat, rope = w.stream_rows(cache, s)
        if fp8:   # the rows as an FP8 pool holds them (issue #1313, step 1.3, item 3)
            from . import fp8 as F
            x = (np.ascontiguousarray(lat, np.uint16).astype(np.uint32) << 16).view(np.float32)
            lat = F.dequantize_rows(*F.quantize_rows(x))
        items = None if items_per_stream is None else items_per_stream[s]
        if items is None:
            items = np.arange(w.R * w.H, dtype=np.int32)
        out, lse = attend_stream(qall[s], lat, rope, w.scale, items, threads)
        res.append((np.asarray(items, np.int32), out, lse))
    return res
