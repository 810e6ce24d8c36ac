"""Pins of the paged-image oracle (append, kept-state copy) by brute force on tiny pools."""
import numpy as np

from oracle import paged as G
from paged_mla_kv_gb300 import synth as Y


def rows(seed, S, n):
    g = np.random.default_rng(seed)
    return (g.integers(0, 0x7F00, (S, n, 512)).astype(np.uint16),
            g.integers(0, 0x7F00, (S, n, 64)).astype(np.uint16))


def test_page_geometry():
    assert G.PAGE_WORDS * 2 == 589824 == 512 * Y.ROW_BYTES
    assert G.ROPE_OFF * 2 == 524288


def test_append_hand_addresses():
    pool = G.new_pool(1, 4)
    lat, rope = rows(1, 1, 3)
    pt = np.array([[2, 0]], np.int32)
    G.append(pool, 0, pt, 2, [511], lat, rope)          # rows 511, 512, 513
    # row 511 -> logical page 0 -> pool page 2, row 511
    assert np.array_equal(pool[0, 2, 511 * 512:512 * 512], lat[0, 0])
    assert np.array_equal(pool[0, 2, 262144 + 511 * 64:262144 + 512 * 64], rope[0, 0])
    # rows 512, 513 -> logical page 1 -> pool page 0, rows 0 and 1
    assert np.array_equal(pool[0, 0, 0:512], lat[0, 1])
    assert np.array_equal(pool[0, 0, 512:1024], lat[0, 2])
    assert np.array_equal(pool[0, 0, 262144 + 64:262144 + 128], rope[0, 2])
    # nothing else changed
    touched = np.zeros_like(pool, bool)
    touched[0, 2, 511 * 512:512 * 512] = True
    touched[0, 2, 262144 + 511 * 64:262144 + 512 * 64] = True
    touched[0, 0, 0:1024] = True
    touched[0, 0, 262144:262144 + 128] = True
    assert np.all(pool[~touched] == 0x7FC0)


def test_append_then_gather_round_trip_and_window_equals_identity_table():
    S, n, maxp = 3, 700, 2
    lat, rope = rows(2, S, n)
    perm = np.random.default_rng(3).permutation(S * maxp).astype(np.int32).reshape(S, maxp)
    a = G.new_pool(1, S * maxp)
    G.append(a, 0, perm, maxp, [0] * S, lat, rope)
    b = G.new_pool(1, S * maxp)
    G.append(b, 0, None, maxp, [0] * S, lat, rope)
    c = G.new_pool(1, S * maxp)
    G.append(c, 0, np.arange(S * maxp, dtype=np.int32).reshape(S, maxp), maxp, [0] * S, lat, rope)
    assert np.array_equal(b, c)                         # a null table is pages in order
    for s in range(S):
        la, ra = G.gather_rows(a, 0, perm, s, maxp, n)
        assert np.array_equal(la, lat[s]) and np.array_equal(ra, rope[s])


def test_state_copy_moves_only_rows_below_at():
    pool = G.new_pool(2, 6)
    lat, rope = rows(4, 1, 1024)
    src = np.array([[4, 1]], np.int32)
    for c in range(2):
        G.append(pool, c, src, 2, [0], lat, rope)
    before = pool.copy()
    G.state_copy_rows(pool, -1, src[0], [0, 5], 600)
    for c in range(2):
        l0, r0 = G.gather_rows(pool, c, np.array([[0, 5]]), 0, 2, 1024)
        assert np.array_equal(l0[:600], lat[0, :600]) and np.array_equal(r0[:600], rope[0, :600])
        assert np.all(l0[600:] == 0x7FC0) and np.all(r0[600:] == 0x7FC0)
    # source pages untouched
    assert np.array_equal(pool[:, [4, 1]], before[:, [4, 1]])
    # one cache only
    p2 = before.copy()
    G.state_copy_rows(p2, 1, src[0], [0, 5], 10)
    assert np.array_equal(p2[0], before[0])
