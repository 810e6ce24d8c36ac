"""Pins for the top-k oracle (blocked top-k with an exact merge, chunked-prefill note section 2.3).

The oracle's `topk` is one library sort; these pins hold it to things fixed independently of
it: hand-ranked special values, a count-of-better-keys ranking on tiny rows, numpy's stable
argsort where the two orders coincide, and the page's identity between the blocked and the
unblocked forms.
"""
import math

import numpy as np
import pytest

from oracle import topk as T
from paged_mla_kv_gb300 import synth


def test_special_values_hand_ranked():
    # +1 twice (columns 4, 5), +0 above -0, -inf, then NaN last
    v = np.array([0.0, -0.0, np.nan, -np.inf, 1.0, 1.0], dtype=np.float32)
    c, x = T.topk(v, 6)
    assert c.tolist() == [4, 5, 0, 1, 3, 2]
    assert x[:4].tolist() == [1.0, 1.0, 0.0, 0.0]
    assert math.copysign(1.0, x[2]) > 0 and math.copysign(1.0, x[3]) < 0
    assert x[4] == -np.inf and np.isnan(x[5])


def test_short_row_filled():
    c, x = T.topk(np.array([2.0, 3.0], dtype=np.float32), 4)
    assert c.tolist() == [1, 0, -1, -1]
    assert x[2] == -np.inf and x[3] == -np.inf
    c, x = T.topk(np.zeros(0, dtype=np.float32), 2)
    assert c.tolist() == [-1, -1]


@pytest.mark.parametrize("seed", range(12))
def test_matches_count_of_better_keys(seed):
    g = np.random.default_rng(seed)
    n = int(g.integers(1, 40))
    pool = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 1.5, -1.5, 2.0], dtype=np.float32)
    v = np.where(g.random(n) < 0.5, g.choice(pool, n), np.round(g.standard_normal(n) * 2) / 2).astype(np.float32)
    ranked = T.rank_by_count(v)
    for k in (1, max(1, n // 3), n, n + 3):
        c, x = T.topk(v, k)
        m = min(k, n)
        assert c[:m].tolist() == ranked[:m]
        assert (c[m:] == -1).all()
        assert np.array_equal(x[:m].view(np.uint32), v[ranked[:m]].view(np.uint32))


@pytest.mark.parametrize("seed", range(6))
def test_matches_stable_argsort_without_nan_or_signed_zero(seed):
    g = np.random.default_rng(100 + seed)
    v = (g.integers(-20, 20, 5000) / 4.0).astype(np.float32)   # many equal values
    v[v == 0] = 0.25
    for k in (1, 17, 512, 5000):
        c, _ = T.topk(v, k)
        assert c.tolist() == np.argsort(-v, kind="stable")[:k].tolist()


@pytest.mark.parametrize("seed", range(8))
def test_blocked_equals_unblocked(seed):
    g = np.random.default_rng(200 + seed)
    n = int(g.integers(1, 3000))
    v = (np.round(g.standard_normal(n) * 3) / 3).astype(np.float32)   # heavy ties across blocks
    v[g.random(n) < 0.02] = np.nan
    v[g.random(n) < 0.02] = -0.0
    for k in (1, 5, 64, 700):
        ref = T.topk(v, k)
        for block in (1, 3, 64, 1000, n):
            got = T.topk_blocked(v, k, block)
            assert np.array_equal(got[0], ref[0]), (k, block)
            assert np.array_equal(got[1].view(np.uint32), ref[1].view(np.uint32))


def test_block_rule_needs_smallest_columns_among_ties():
    # If a block kept its last equal keys instead of its first, the merge would lose column 1.
    v = np.array([5.0, 5.0, 5.0, 5.0], dtype=np.float32)
    assert T.topk_blocked(v, 2, 2)[0].tolist() == [0, 1]
    c, _ = T.topk(v[2:], 1, cols=np.array([2, 3]))
    assert c.tolist() == [2]


def test_rows_and_lengths():
    x = synth.topk_logits(3, [0, 1, 2], 50)
    lens = np.array([50, 7, 0])
    oi, ov = T.topk_rows(x, 10, lens)
    assert oi[0].tolist() == T.topk(x[0], 10)[0].tolist()
    assert oi[1, :7].tolist() == T.topk(x[1, :7], 10)[0][:7].tolist() and (oi[1, 7:] == -1).all()
    assert (oi[2] == -1).all() and (ov[2] == -np.inf).all()


def test_synthetic_logits_depend_on_row_only():
    a = synth.topk_logits(9, [4, 5], 300)
    b = synth.topk_logits(9, [5], 300)
    assert np.array_equal(a[1], b[0])
    assert np.all(np.round(a * 64) == a * 64)
