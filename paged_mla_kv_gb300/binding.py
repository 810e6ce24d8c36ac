"""Thin Python binding of libtf_paged_mla.so (include/tf_paged_mla.h).

Argument marshalling only: tensors become device pointers, the current torch
CUDA stream becomes the launch stream, host arrays become C arrays, and a
negative status becomes a TFError.  Every step of the path runs in the
library's kernels; there is no fallback, and loading fails loudly when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libtf_paged_mla.so")

TF_OK, TF_E_ARG, TF_E_RANGE, TF_E_NOMEM, TF_E_CUDA, TF_E_TIMEOUT, TF_E_UNSUPPORTED, TF_E_DEVICE = \
    0, -1, -2, -3, -4, -5, -6, -7
TF_POOL_POISON = 1
TF_POOL_BATCH_INVARIANT = 2
TF_POOL_FP8 = 4
PAGE_BYTES_BF16 = 589824
PAGE_BYTES_FP8 = 329728    # 512 x 512 E4M3 codes, 512 fp32 scales, 512 x 64 bf16 rope
ERR_NAMES = {0: "TF_OK", -1: "TF_E_ARG", -2: "TF_E_RANGE", -3: "TF_E_NOMEM", -4: "TF_E_CUDA",
             -5: "TF_E_TIMEOUT", -6: "TF_E_UNSUPPORTED", -7: "TF_E_DEVICE"}
PROF_APPEND, PROF_ATTEND, PROF_COMBINE, PROF_COPY, PROF_POISON = range(5)


class TFError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} failed: {ERR_NAMES.get(code, code)}")
        self.code = code


class tf_kvpool_desc(ctypes.Structure):
    _fields_ = [("num_caches", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("page_rows", ctypes.c_int32),
                ("latent_dim", ctypes.c_int32), ("rope_dim", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("seed", ctypes.c_uint64)]


class tf_plan_in(ctypes.Structure):
    _fields_ = [("room_bytes", ctypes.c_int64), ("context_tokens", ctypes.c_int64), ("lanes", ctypes.c_int32),
                ("page_rows", ctypes.c_int32), ("lookahead", ctypes.c_int32), ("engine_paged", ctypes.c_int32),
                ("bytes_per_token", ctypes.c_int64), ("fixed_bytes", ctypes.c_int64),
                ("cache_budget_bytes", ctypes.c_int64)]


class tf_attend_plan(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("ctas", ctypes.c_int32), ("nranges", ctypes.c_int32),
                ("groups", ctypes.c_int32), ("work", ctypes.c_int64), ("slots", ctypes.c_int64)]


TF_PLAN_MAX_RANGES = 240


class tf_plan_out(ctypes.Structure):
    _fields_ = [("n_windows", ctypes.c_int32), ("window_pages", ctypes.c_int64), ("stream_pages", ctypes.c_int64),
                ("cache_bytes", ctypes.c_int64), ("other_pages", ctypes.c_int64), ("pool_pages", ctypes.c_int64),
                ("pool_tokens", ctypes.c_int64)]


_P, _I32, _I64, _U64, _SZ, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t, \
    ctypes.c_float
_SIGS = {
    "tf_kvpool_bytes": (_SZ, [ctypes.POINTER(tf_kvpool_desc)]),
    "tf_kvpool_create": (ctypes.c_int, [ctypes.POINTER(tf_kvpool_desc), _P, _SZ, ctypes.POINTER(_P)]),
    "tf_kvpool_destroy": (ctypes.c_int, [_P]),
    "tf_kvpool_take": (ctypes.c_int, [_P, _I32, _P, _P]),
    "tf_kvpool_ref": (ctypes.c_int, [_P, _P, _I32]),
    "tf_kvpool_release": (ctypes.c_int, [_P, _P, _I32]),
    "tf_kvpool_free_pages": (_I32, [_P]),
    "tf_kvpool_refcount": (_I32, [_P, _I32]),
    "tf_kvpool_page_ptr": (_P, [_P, _I32, _I32]),
    "tf_kvpool_plan": (ctypes.c_int, [ctypes.POINTER(tf_plan_in), ctypes.POINTER(tf_plan_out)]),
    "tf_paged_append": (ctypes.c_int, [_P, _I32, _P, _I32, _P, _I32, _I32, _P, _P, _P]),
    "tf_paged_mla_workspace_bytes": (_SZ, [_P, _I32, _I32, _I32, _P]),
    "tf_paged_mla_attend": (ctypes.c_int, [_P, _I32, _P, _I32, _P, _I32, _I32, _I32, _P, _F, _P, _P, _P, _SZ, _P]),
    "tf_paged_mla_attend_static": (ctypes.c_int, [_P, _I32, _P, _I32, _P, _I32, _I32, _I32, _P, _F, _P, _P, _P]),
    "tf_paged_mla_sparse_workspace_bytes": (_SZ, [_P, _I32, _I32, _P]),
    "tf_paged_mla_attend_sparse": (ctypes.c_int, [_P, _I32, _P, _I32, _P, _P, _I32, _P, _I32, _I32, _P, _F, _P, _P,
                                                  _P, _SZ, _P]),
    "tf_state_copy_rows": (ctypes.c_int, [_P, _I32, _P, _P, _I64, _P]),
    "tf_last_error": (ctypes.c_int, [_P, ctypes.POINTER(_I64)]),
    "tf_diag_wait_timeout": (ctypes.c_int, [_P, _I64, _P]),
    "tf_launch_count": (_I64, []),
    "tf_paged_mla_plan_info": (ctypes.c_int, [_I32, _I32, _I32, _P, _I32, _I32, _P, _P, _P]),
    "tf_topk_workspace_bytes": (_SZ, [_I64, _I64, _I32]),
    "tf_topk_blocked": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _SZ, _P]),
    "tf_profile_enable": (ctypes.c_int, [_P, _I32]),
    "tf_profile_read": (ctypes.c_int, [_P, _I32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I64)]),
}

_lib = None


def lib():
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libtf_paged_mla.so is not built ({LIB_PATH}); run paged_mla_kv_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != TF_OK:
        raise TFError(rc, what)


# Argument marshalling is on every call's path, so pointers travel as plain ints (ctypes turns
# an int into a void * for a c_void_p argument) and arrays already in the right form are used
# as they are.

def _ptr(t):
    if t is None:
        return None
    return t.data_ptr()


_current_stream = None


def _stream(stream):
    """The raw CUDA stream: `stream` as given, else torch's current stream on the current device."""
    if stream is not None:
        return int(stream)
    global _current_stream
    if _current_stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        get_dev = getattr(torch._C, "_cuda_getDevice", None)
        if raw is not None and get_dev is not None:
            _current_stream = lambda: raw(get_dev())
        else:
            _current_stream = lambda: torch.cuda.current_stream().cuda_stream
    return _current_stream()


def _i64(a):
    if not (isinstance(a, np.ndarray) and a.dtype == np.int64 and a.flags.c_contiguous):
        a = np.ascontiguousarray(a, dtype=np.int64)
    return a, a.ctypes.data


def make_desc(num_caches: int, num_pages: int, poison: bool = False, seed: int = 0,
              invariant: bool = False, fp8: bool = False) -> tf_kvpool_desc:
    flags = ((TF_POOL_POISON if poison else 0) | (TF_POOL_BATCH_INVARIANT if invariant else 0) |
             (TF_POOL_FP8 if fp8 else 0))
    return tf_kvpool_desc(num_caches, num_pages, 512, 512, 64, flags, seed)


def tf_kvpool_bytes(desc: tf_kvpool_desc) -> int:
    return int(lib().tf_kvpool_bytes(ctypes.byref(desc)))


def tf_kvpool_plan(**kw) -> tf_plan_out:
    pin = tf_plan_in(kw["room_bytes"], kw["context_tokens"], kw["lanes"], kw.get("page_rows", 512),
                     kw.get("lookahead", 1), int(kw.get("engine_paged", 0)), kw["bytes_per_token"],
                     kw["fixed_bytes"], kw["cache_budget_bytes"])
    out = tf_plan_out()
    rc = lib().tf_kvpool_plan(ctypes.byref(pin), ctypes.byref(out))
    if rc == TF_E_NOMEM:
        return None
    _check(rc, "tf_kvpool_plan")
    return out


class KVPool:
    """A pool over caller device memory (a torch uint8 tensor kept alive here)."""

    def __init__(self, num_caches: int, num_pages: int, poison: bool = False, seed: int = 0, device=None,
                 memory=None, invariant: bool = False, fp8: bool = False):
        self.desc = make_desc(num_caches, num_pages, poison, seed, invariant, fp8)
        self.fp8 = fp8
        self.page_bytes = PAGE_BYTES_FP8 if fp8 else PAGE_BYTES_BF16
        self.bytes = tf_kvpool_bytes(self.desc)
        if self.bytes == 0:
            raise TFError(TF_E_ARG, "tf_kvpool_bytes")
        if memory is None:
            import torch
            memory = torch.empty(self.bytes + 1024, dtype=torch.uint8, device=device or "cuda")
        self.memory = memory
        base = memory.data_ptr()
        off = (-base) % 1024
        self.base = base + off
        h = ctypes.c_void_p()
        _check(lib().tf_kvpool_create(ctypes.byref(self.desc), ctypes.c_void_p(self.base),
                                      self.bytes, ctypes.byref(h)), "tf_kvpool_create")
        self.handle = h
        self.num_caches, self.num_pages = num_caches, num_pages

    def close(self):
        if self.handle:
            lib().tf_kvpool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # host page bookkeeping
    def take(self, n: int, stream=None) -> np.ndarray:
        ids = np.zeros(max(n, 1), np.int32)
        _check(lib().tf_kvpool_take(self.handle, n, ids.ctypes.data_as(ctypes.c_void_p),
                                    _stream(stream) if self.desc.flags else None), "tf_kvpool_take")
        return ids[:n]

    def ref(self, ids) -> None:
        a = np.ascontiguousarray(np.asarray(ids, np.int32))
        _check(lib().tf_kvpool_ref(self.handle, a.ctypes.data_as(ctypes.c_void_p), len(a)), "tf_kvpool_ref")

    def release(self, ids) -> None:
        a = np.ascontiguousarray(np.asarray(ids, np.int32))
        _check(lib().tf_kvpool_release(self.handle, a.ctypes.data_as(ctypes.c_void_p), len(a)), "tf_kvpool_release")

    def free_pages(self) -> int:
        return int(lib().tf_kvpool_free_pages(self.handle))

    def refcount(self, page: int) -> int:
        return int(lib().tf_kvpool_refcount(self.handle, page))

    def page_ptr(self, cache: int, page: int) -> int:
        return int(lib().tf_kvpool_page_ptr(self.handle, cache, page) or 0)

    def view(self):
        """The pool's device bytes as a uint16 tensor [caches][pages][294912] (BF16 pages)."""
        return self.bytes_view().view(__import__("torch").int16)

    def bytes_view(self):
        """The pool's device bytes as a uint8 tensor [caches][pages][page bytes]."""
        off = self.base - self.memory.data_ptr()
        n = self.num_caches * self.num_pages * self.page_bytes
        return self.memory[off:off + n].view(self.num_caches, self.num_pages, self.page_bytes)

    def last_error(self):
        d = ctypes.c_int64(0)
        rc = lib().tf_last_error(self.handle, ctypes.byref(d))
        return rc, d.value

    def profile(self, on: bool = True):
        _check(lib().tf_profile_enable(self.handle, 1 if on else 0), "tf_profile_enable")

    def profile_read(self, kind: int):
        ms, n = ctypes.c_double(0.0), ctypes.c_int64(0)
        _check(lib().tf_profile_read(self.handle, kind, ctypes.byref(ms), ctypes.byref(n)), "tf_profile_read")
        return ms.value, n.value


def tf_paged_append(pool: KVPool, cache: int, pt, max_pages: int, pos, latent, rope, stream=None) -> None:
    """latent: bf16 [S][n][512], rope: bf16 [S][n][64] (CUDA tensors); pt: int32 [S][max_pages] or None."""
    S, n = int(latent.shape[0]), int(latent.shape[1])
    pos_a, pos_p = _i64(pos)
    _check(lib().tf_paged_append(pool.handle, cache, _ptr(pt), max_pages, pos_p, S, n, _ptr(latent), _ptr(rope),
                                 _stream(stream)), "tf_paged_append")


def tf_paged_mla_workspace_bytes(pool, S: int, R: int, H: int, lens) -> int:
    """Workspace bytes for an attend call on `pool` (a KVPool, or None for the default plan)."""
    a, p = _i64(lens)
    return int(lib().tf_paged_mla_workspace_bytes(pool.handle if pool is not None else None, S, R, H, p))


def tf_paged_mla_attend(pool: KVPool, cache: int, pt, max_pages: int, lens, q, scale: float, out, lse=None,
                        ws=None, stream=None) -> None:
    """q: bf16 [S][R][H][576]; out: bf16 [S][R][H][512]; lse: fp32 [S][R][H] or None; ws: uint8 workspace."""
    S, R, H = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
    a, p = _i64(lens)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().tf_paged_mla_attend(pool.handle, cache, _ptr(pt), max_pages, p, S, R, H, _ptr(q), float(scale),
                                     _ptr(out), _ptr(lse), _ptr(ws), ws_bytes, _stream(stream)),
           "tf_paged_mla_attend")


TF_STATIC_WS_BYTES = 64 << 20


def tf_paged_mla_attend_static(pool: KVPool, cache: int, pt, max_pages: int, lens, q, scale: float, out, lse=None,
                               stream=None) -> None:
    """tf_paged_mla_attend without a workspace: for callers that cannot allocate device memory."""
    S, R, H = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
    a, p = _i64(lens)
    _check(lib().tf_paged_mla_attend_static(pool.handle, cache, _ptr(pt), max_pages, p, S, R, H, _ptr(q),
                                            float(scale), _ptr(out), _ptr(lse), _stream(stream)),
           "tf_paged_mla_attend_static")


def _i32(a):
    if not (isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous):
        a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data


def tf_paged_mla_sparse_workspace_bytes(pool, S: int, H: int, nidx) -> int:
    a, p = _i32(nidx)
    return int(lib().tf_paged_mla_sparse_workspace_bytes(pool.handle if pool is not None else None, S, H, p))


def tf_paged_mla_attend_sparse(pool: KVPool, cache: int, pt, max_pages: int, lens, idx, nidx, q, scale: float, out,
                               lse=None, ws=None, stream=None) -> None:
    """idx: int32 CUDA tensor [S][max_idx] of listed rows; nidx: host counts [S]; q: bf16 [S][H][576] (or
    [S][1][H][576]); out: bf16 [S][H][512] (same leading shape as q); lse: fp32 [S][H] or None."""
    S, H = int(q.shape[0]), int(q.shape[-2])
    a, p = _i64(lens)
    b, pn = _i32(nidx)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().tf_paged_mla_attend_sparse(pool.handle, cache, _ptr(pt), max_pages, p, _ptr(idx), int(idx.shape[1]),
                                            pn, S, H, _ptr(q), float(scale), _ptr(out), _ptr(lse), _ptr(ws), ws_bytes,
                                            _stream(stream)),
           "tf_paged_mla_attend_sparse")


def tf_state_copy_rows(pool: KVPool, cache: int, src_pages, dst_pages, at: int, stream=None) -> None:
    """src_pages / dst_pages: int32 CUDA tensors of ceil(at / 512) page ids."""
    _check(lib().tf_state_copy_rows(pool.handle, cache, _ptr(src_pages), _ptr(dst_pages), int(at),
                                    _stream(stream)), "tf_state_copy_rows")


def tf_diag_wait_timeout(pool: KVPool, limit_cycles: int, stream=None) -> None:
    _check(lib().tf_diag_wait_timeout(pool.handle, int(limit_cycles), _stream(stream)), "tf_diag_wait_timeout")


def tf_topk_workspace_bytes(rows: int, n: int, k: int) -> int:
    return int(lib().tf_topk_workspace_bytes(int(rows), int(n), int(k)))


def tf_topk_blocked(logits, k: int, idx, val, lens=None, n: int | None = None, ws=None, stream=None) -> None:
    """logits: fp32 CUDA tensor [rows][ld] (row stride ld, a multiple of 4); n: columns in play
    (default ld); lens: int32 CUDA tensor [rows] or None; idx: int32 [rows][k]; val: fp32 [rows][k]."""
    rows, ld = int(logits.shape[0]), int(logits.stride(0)) if logits.dim() == 2 else 0
    n = int(logits.shape[1]) if n is None else int(n)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().tf_topk_blocked(_ptr(logits), rows, n, ld, _ptr(lens), int(k), _ptr(idx), _ptr(val), _ptr(ws),
                                 ws_bytes, _stream(stream)), "tf_topk_blocked")


def tf_paged_mla_plan_info(S: int, R: int, H: int, lens, sms: int = 0, invariant: bool = False) -> dict:
    """The attention's work plan for these lengths (host arithmetic, nothing launched): mode,
    ctas, nranges, groups, work, slots, and the range bounds (modes 0 and 1) or each stream's
    split keys (mode 2) as int64 arrays."""
    a, p = _i64(lens)
    info = tf_attend_plan()
    bounds = np.zeros(TF_PLAN_MAX_RANGES + 1, np.int64)
    splits = np.zeros(max(S, 1), np.int64)
    _check(lib().tf_paged_mla_plan_info(S, R, H, p, sms, 1 if invariant else 0, ctypes.byref(info),
                                        bounds.ctypes.data_as(ctypes.c_void_p),
                                        splits.ctypes.data_as(ctypes.c_void_p)), "tf_paged_mla_plan_info")
    out = {f: int(getattr(info, f)) for f, _ in tf_attend_plan._fields_}
    out["bounds"] = bounds[:out["nranges"] + 1] if out["mode"] in (0, 1) else None
    out["split_keys"] = splits[:S] if out["mode"] == 2 else None
    return out


def tf_launch_count() -> int:
    return int(lib().tf_launch_count())
