"""Pins of the fp64 attention oracle against closed forms, library routines and invariants.

Each pin is chosen so that a plausible slip in the oracle -- a dropped rope
term, a wrong sign, an off-by-one causal limit, a transposed operand, a wrong
query row or head -- fails at least one test.
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle.attend import attend_sparse, attend_stream
from paged_mla_kv_gb300 import synth as Y


def bf(x):
    return Y.f32_to_bf16_bits(np.asarray(x, np.float32))


def wide(b):
    return Y.bf16_bits_to_f32(b).astype(np.float64)


def rand_case(seed, n, R, H, std=0.5, qstd=0.5):
    g = np.random.default_rng(seed)
    lat = bf(g.normal(0, std, (n, 512)))
    rope = bf(g.normal(0, std, (n, 64)))
    q = bf(g.normal(0, qstd, (R, H, 576)))
    return q, lat, rope


def test_single_key_returns_its_latent_and_score():
    q, lat, rope = rand_case(1, 1, 1, 3)
    scale = 0.37
    out, lse = attend_stream(q, lat, rope, scale)
    for h in range(3):
        assert np.array_equal(out[h], wide(lat[0]))          # weight exactly 1
        terms = [float(a) * float(b) for a, b in zip(wide(q[0, h, :512]), wide(lat[0]))]
        terms += [float(a) * float(b) for a, b in zip(wide(q[0, h, 512:]), wide(rope[0]))]
        assert lse[h] == pytest.approx(scale * math.fsum(terms), rel=1e-12, abs=1e-12)


def test_zero_query_gives_mean_and_log_count():
    n, R, H = 77, 2, 2
    _, lat, rope = rand_case(2, n, R, H)
    q = np.zeros((R, H, 576), np.uint16)                     # bf16 +0.0
    out, lse = attend_stream(q, lat, rope, 0.5)
    L = wide(lat)
    for r in range(R):
        nk = n - R + r + 1                                   # row r sees keys 0..n-R+r
        for h in range(H):
            i = r * H + h
            np.testing.assert_allclose(out[i], L[:nk].mean(axis=0), rtol=1e-12, atol=1e-14)
            assert lse[i] == pytest.approx(math.log(nk), rel=1e-13)


def test_two_keys_closed_form_sign():
    # scores s0 = scale * a, s1 = scale * b through the rope part only
    lat = bf(np.array([[1.0] * 512, [-2.0] * 512]))
    rope = np.zeros((2, 64), np.uint16)
    rope[0, 5] = bf([3.0])[0]
    rope[1, 5] = bf([-1.0])[0]
    q = np.zeros((1, 1, 576), np.uint16)
    q[0, 0, 512 + 5] = bf([0.75])[0]
    scale = 0.5
    out, lse = attend_stream(q, lat, rope, scale)
    s0, s1 = scale * 0.75 * 3.0, scale * 0.75 * -1.0
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    np.testing.assert_allclose(out[0], (1 - w1) * 1.0 + w1 * -2.0, rtol=1e-13)
    assert lse[0] == pytest.approx(math.log(math.exp(s0) + math.exp(s1)), rel=1e-13)


@pytest.mark.parametrize("seed", [3, 4, 5])
def test_matches_scipy_softmax_for_the_last_row(seed):
    # the last row of the last head sees every key: a plain softmax-weighted average
    n, R, H = 123, 3, 4
    q, lat, rope = rand_case(seed, n, R, H)
    scale = 1 / math.sqrt(576)
    out, lse = attend_stream(q, lat, rope, scale)
    K = np.concatenate([wide(lat), wide(rope)], axis=1)      # [n][576]
    for r in range(R):
        nk = n - R + r + 1
        for h in range(H):
            s = scale * (K[:nk] @ wide(q[r, h]))
            np.testing.assert_allclose(out[r * H + h], softmax(s) @ wide(lat)[:nk], rtol=1e-10, atol=1e-12)
            assert lse[r * H + h] == pytest.approx(logsumexp(s), rel=1e-12)


def test_matches_a_40_digit_evaluation_of_the_definition():
    """Every output of a tiny causal case (two rows, two heads, 19 keys) against the definition
    evaluated in 40-digit arithmetic with mpmath, no numpy on that side: scores as the two dot
    products, max-shifted exponentials, their sum, the weighted latent mean and the log-sum-exp.
    The fp64 oracle must agree to 1e-12 of the output's size, far inside any kernel tolerance."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    n, R, H = 19, 2, 2
    q, lat, rope = rand_case(11, n, R, H, std=1.0, qstd=1.0)
    scale = 1 / math.sqrt(576)
    out, lse = attend_stream(q, lat, rope, scale)
    C = [[mp.mpf(float(v)) for v in row] for row in wide(lat)]
    Kr = [[mp.mpf(float(v)) for v in row] for row in wide(rope)]
    sc = mp.mpf(scale)                       # the same double the oracle is given
    for r in range(R):
        p_ = n - R + r                        # the row's position: it sees keys 0 .. p_
        for h in range(H):
            qq = [mp.mpf(float(v)) for v in wide(q[r, h])]
            s = [sc * (mp.fsum(qq[d] * C[j][d] for d in range(512)) +
                       mp.fsum(qq[512 + e] * Kr[j][e] for e in range(64))) for j in range(p_ + 1)]
            m = max(s)
            ex = [mp.exp(x - m) for x in s]
            Z = mp.fsum(ex)
            want = [float(mp.fsum(ex[j] * C[j][d] for j in range(p_ + 1)) / Z) for d in range(512)]
            got = out[r * H + h]
            size = max(1.0, max(abs(w) for w in want))
            assert max(abs(w - g) for w, g in zip(want, got)) <= 1e-12 * size, (r, h)
            assert abs(float(m + mp.log(Z)) - lse[r * H + h]) <= 1e-12 * max(1.0, abs(float(m))), (r, h)


def test_items_select_row_and_head():
    n, R, H = 40, 2, 3
    q, lat, rope = rand_case(6, n, R, H)
    full, fl = attend_stream(q, lat, rope, 0.2)
    items = [5, 0, 3]
    part, pl = attend_stream(q, lat, rope, 0.2, items=items)
    for k, i in enumerate(items):
        assert np.array_equal(part[k], full[i]) and pl[k] == fl[i]
    # different heads give different answers (a head index that is ignored fails this)
    assert not np.allclose(full[0], full[1])


def test_causal_limit_and_draft_equals_plain():
    n = 50
    q, lat, rope = rand_case(7, n, 2, 2)
    two, lse2 = attend_stream(q, lat, rope, 0.3)
    # row 0 of an R=2 pass at len n equals an R=1 pass at len n-1 with the same query
    one, lse1 = attend_stream(q[:1], lat[:n - 1], rope[:n - 1], 0.3)
    np.testing.assert_array_equal(two[:2], one)
    # changing the newest key leaves row 0 alone and moves row 1
    lat2, rope2 = lat.copy(), rope.copy()
    lat2[n - 1] = bf(np.full(512, 3.0))
    rope2[n - 1] = bf(np.full(64, 3.0))
    three, _ = attend_stream(q, lat2, rope2, 0.3)
    np.testing.assert_array_equal(three[:2], two[:2])
    assert not np.allclose(three[2:], two[2:])


def test_key_order_does_not_matter_and_dominant_key_wins():
    n = 64
    q, lat, rope = rand_case(8, n, 1, 1)
    perm = np.random.default_rng(0).permutation(n)
    a, la = attend_stream(q, lat, rope, 0.25)
    b, lb = attend_stream(q, lat[perm], rope[perm], 0.25)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)
    assert la[0] == pytest.approx(lb[0], rel=1e-13)
    # plant a key aligned with the query: its latent dominates
    lat3, rope3 = lat.copy(), rope.copy()
    lat3[17] = q[0, 0, :512]
    rope3[17] = q[0, 0, 512:]
    c, _ = attend_stream(q, lat3, rope3, 200.0)
    np.testing.assert_allclose(c[0], wide(lat3[17]), atol=1e-6)


def test_shift_of_all_scores_moves_only_lse():
    n = 30
    q, lat, rope = rand_case(9, n, 1, 2)
    a, la = attend_stream(q, lat, rope, 0.5)
    rope2 = rope.copy()
    rope2[:, 63] = bf([1.0])[0]                # every key gets the same extra component
    q2 = q.copy()
    q2[0, :, 576 - 1] = bf([2.0])[0]
    base = q.copy()
    base[0, :, 575] = 0
    b0, lb0 = attend_stream(base, lat, rope2, 0.5)
    b1, lb1 = attend_stream(q2, lat, rope2, 0.5)
    np.testing.assert_allclose(b1, b0, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lb1 - lb0, 0.5 * 2.0 * 1.0, rtol=1e-12)


def test_rope_term_is_not_dropped():
    # two keys equal in the latent, different in the rope part: weights must differ from 1/2
    lat = bf(np.array([[0.5] * 512, [0.5] * 512]))
    rope = bf(np.array([[1.0] * 64, [-1.0] * 64]))
    q = np.zeros((1, 1, 576), np.uint16)
    q[0, 0, 512:] = bf(np.full(64, 0.25))
    out, lse = attend_stream(q, lat, rope, 1.0)
    s0, s1 = 16.0, -16.0
    assert lse[0] == pytest.approx(math.log(math.exp(s0) + math.exp(s1)), rel=1e-13)


def test_rejects_rows_without_keys():
    q, lat, rope = rand_case(10, 1, 2, 1)
    with pytest.raises(ValueError):
        attend_stream(q, lat, rope, 1.0)


def test_rejects_items_outside_the_rows_and_heads():
    q, lat, rope = rand_case(10, 8, 2, 3)
    for bad in (-1, 6):                       # r*H + h must lie in [0, R*H)
        with pytest.raises(ValueError):
            attend_stream(q, lat, rope, 1.0, items=[0, bad])


# ---------------------------------------------------------------- listed rows (sparse)


def test_sparse_single_listed_row_is_that_row():
    q, lat, rope = rand_case(11, 300, 1, 4)
    out, lse = attend_sparse(q[0], lat, rope, [123], 0.3)
    for h in range(4):
        assert np.array_equal(out[h], wide(lat[123]))


def test_sparse_zero_query_is_the_mean_of_the_listed_rows():
    q, lat, rope = rand_case(12, 500, 1, 2)
    q[:] = 0
    idx = [7, 400, 3, 250, 7]                              # 7 is listed twice: counted twice
    out, lse = attend_sparse(q[0], lat, rope, idx, 0.5)
    want = np.mean([wide(lat[i]) for i in idx], axis=0)
    assert np.allclose(out[0], want, rtol=0, atol=1e-13)
    assert lse[0] == pytest.approx(math.log(len(idx)), abs=1e-12)


def test_sparse_every_row_listed_twice_moves_only_lse_by_log2():
    q, lat, rope = rand_case(13, 90, 1, 3)
    idx = np.random.default_rng(1).choice(90, 40, replace=False)
    o1, l1 = attend_sparse(q[0], lat, rope, idx, 0.2)
    o2, l2 = attend_sparse(q[0], lat, rope, np.concatenate([idx, idx]), 0.2)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12)
    assert np.allclose(l2 - l1, math.log(2.0), rtol=0, atol=1e-12)


def test_sparse_list_order_does_not_matter_and_unlisted_rows_do_not_count():
    q, lat, rope = rand_case(14, 200, 1, 3)
    g = np.random.default_rng(2)
    idx = g.choice(200, 64, replace=False)
    o1, l1 = attend_sparse(q[0], lat, rope, idx, 0.25)
    o2, l2 = attend_sparse(q[0], lat, rope, g.permutation(idx), 0.25)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)
    # poisoning a row that is not listed changes nothing
    lat2 = lat.copy()
    lat2[np.setdiff1d(np.arange(200), idx)[0]] = 0x7FC0
    o3, l3 = attend_sparse(q[0], lat2, rope, idx, 0.25)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)
    # and against scipy on the listed scores
    s = np.array([0.25 * (wide(q[0, 1, :512]) @ wide(lat[i]) + wide(q[0, 1, 512:]) @ wide(rope[i])) for i in idx])
    assert l1[1] == pytest.approx(float(logsumexp(s)), abs=1e-12)
    assert np.allclose(o1[1], softmax(s) @ np.array([wide(lat[i]) for i in idx]), rtol=0, atol=1e-12)


def test_the_draft_test_tolerance_catches_an_off_by_one_causal_limit():
    # The GPU test of the draft row (tests/test_gpu_parity.py, drafted == plain) bounds the
    # rel-L2 between the two outputs and to the oracle by 1e-2.  On its workload (3,333 rows of
    # N(0, 0.1) values, queries N(0, 0.1), scale 1/24) the weights are near uniform, so a draft
    # row that saw one key too many -- the planted off-by-one, here in the oracle's inputs --
    # moves by about 1/sqrt(3,333) = 1.7% in rel-L2 and fails that bound.
    w = Y.custom("draft", 45, lens=[3333], R=2, H=64)
    lat, rope = w.stream_rows(0, 0)
    q = w.q()[0][:1]                                     # the draft row's queries, [1][64][576]
    heads = np.arange(0, 64, 8, dtype=np.int32)          # eight heads keep this fast
    right, _ = attend_stream(q, lat[:3332], rope[:3332], w.scale, heads)
    wrong, _ = attend_stream(q, lat, rope, w.scale, heads)  # one key past the causal limit
    rel = np.linalg.norm(wrong - right) / np.linalg.norm(right)
    assert rel > 1e-2, rel
