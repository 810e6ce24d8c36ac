"""Top-k of a row of fp32 logits, unblocked and blocked -- TEST INFRASTRUCTURE ONLY.

Follows "Running CHUNKED_PREFILL_SIZE above 1024 without the long-prompt memory problem",
section 2.3: score a row block by block, keep each block's top-k (values and columns), then
take the top-k of the concatenated candidates; that equals the top-k of the whole row.

The page does not say how equal values are ranked.  Read here as: larger value first under the
IEEE total order of fp32 (+0 above -0, every NaN below every number, -inf included), equal
values by the smaller column.  Under that order the top-k is unique, which is what lets the
blocked and unblocked forms agree exactly.

`topk` is the plain definition (one library sort of the whole row); `topk_blocked` is the
page's blocked form built on it; `rank_by_count` is a second, independent formulation used
only by the pins (each key's place = how many keys beat it).
"""
from __future__ import annotations

import math

import numpy as np

PAD_COL = -1
PAD_VAL = -math.inf


def _order_keys(v: np.ndarray, cols: np.ndarray):
    """Sort keys for np.lexsort (last key primary): not-NaN first, value descending, +0 before
    -0, column ascending."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    nan = np.isnan(v)
    neg = np.where(nan, 0.0, -v)
    zero_sign = np.where(v == 0.0, np.signbit(v).astype(np.int8), 0)
    return (cols, zero_sign, neg, nan.astype(np.int8))


def topk(v, k: int, cols=None):
    """The k best entries of one row: (columns int64[k], values float32[k]), best first.
    A row with fewer than k entries is filled with column -1 and value -inf."""
    v = np.asarray(v, dtype=np.float32)
    cols = np.arange(v.size, dtype=np.int64) if cols is None else np.asarray(cols, dtype=np.int64)
    order = np.lexsort(_order_keys(v, cols))[:k]
    oc = np.full(k, PAD_COL, dtype=np.int64)
    ov = np.full(k, PAD_VAL, dtype=np.float32)
    oc[: order.size] = cols[order]
    ov[: order.size] = v[order]
    return oc, ov


def topk_blocked(v, k: int, block: int):
    """Section 2.3's blocked form: each block of `block` columns keeps its top-k, then the
    top-k of all the kept candidates."""
    v = np.asarray(v, dtype=np.float32)
    cand_c, cand_v = [], []
    for b0 in range(0, v.size, block):
        c, x = topk(v[b0:b0 + block], k, cols=np.arange(b0, min(b0 + block, v.size)))
        keep = c != PAD_COL
        cand_c.append(c[keep])
        cand_v.append(x[keep])
    if not cand_c:
        return topk(v, k)
    return topk(np.concatenate(cand_v), k, cols=np.concatenate(cand_c))


def topk_rows(logits: np.ndarray, k: int, lens=None):
    """topk of every row r over its first lens[r] columns: (int32[rows][k], float32[rows][k])."""
    logits = np.asarray(logits, dtype=np.float32)
    rows = logits.shape[0]
    oi = np.empty((rows, k), dtype=np.int32)
    ov = np.empty((rows, k), dtype=np.float32)
    for r in range(rows):
        n = logits.shape[1] if lens is None else max(0, min(int(lens[r]), logits.shape[1]))
        c, x = topk(logits[r, :n], k)
        oi[r] = c
        ov[r] = x
    return oi, ov


def _beats(a: float, ca: int, b: float, cb: int) -> bool:
    """True when (a, column ca) ranks before (b, column cb)."""
    an, bn = math.isnan(a), math.isnan(b)
    if an != bn:
        return bn
    if not an and a != b:
        return a > b
    if not an and a == 0.0 and math.copysign(1.0, a) != math.copysign(1.0, b):
        return math.copysign(1.0, a) > 0
    return ca < cb


def rank_by_count(v) -> list:
    """Columns in rank order, each placed by counting the keys that beat it (tiny rows only)."""
    v = [float(x) for x in np.asarray(v, dtype=np.float32)]
    place = [sum(_beats(v[j], j, v[i], i) for j in range(len(v))) for i in range(len(v))]
    out = [0] * len(v)
    for i, p in enumerate(place):
        out[p] = i
    return out
