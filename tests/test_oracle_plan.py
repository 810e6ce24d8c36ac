"""Pins of the plan oracle against the numbers the pages print (tests/golden/plan_worked_examples.json)."""
import json
import os

import pytest

from oracle import plan as P

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "plan_worked_examples.json")))
GiB, MiB = 1 << 30, 1 << 20
BPT = GOLD["bytes_per_token"]["value"]
FIXED = GOLD["fixed_mib"]["value"] * MiB
BUDGET = GOLD["cache_budget_gib"]["value"] * GiB


def room_tp2():
    # the 2.33 GiB left plus the engine's own 1M window, which is now pages
    return int(round(GOLD["left_gib_tp2_1m"]["value"] * GiB)) + 1048576 * BPT + FIXED


def mk(room, ctx, lanes, paged=False):
    return P.PlanIn(room_bytes=room, context_tokens=ctx, lanes=lanes, bytes_per_token=BPT,
                    fixed_bytes=FIXED, cache_budget_bytes=BUDGET, engine_paged=paged)


def test_byte_sizes():
    assert GOLD["caches"]["value"] * (1024 + 64) == BPT
    w = 1048576 * BPT + FIXED
    assert round(w / GiB, 2) == GOLD["window_gib_1m"]["value"]
    assert round(7 * w / GiB, 2) == GOLD["seven_windows_gib_1m"]["value"]


def test_tp2_1m_today_and_step1():
    g = GOLD["tp2_1m_p8"]["expect"]
    out = P.plan(mk(room_tp2(), 1048576, 8))
    assert out.window_pages == g["window_pages"]
    assert out.pool_pages == g["pool_pages"]
    assert out.pool_tokens == g["pool_tokens"]
    assert abs(out.cache_bytes / GiB - g["cache_gib_approx"]) < 0.05
    assert P.windows_served(room_tp2(), 1048576, BPT, FIXED) == g["windows_served"]
    s1 = P.plan(mk(room_tp2(), 1048576, 8, paged=True))
    assert s1.n_windows == g["step1_n"]
    assert s1.pool_pages == g["pool_pages"]


def _room_today(pages_today, ctx, lanes):
    """Smallest room at which today's order yields `pages_today` pages with a full cache."""
    page = 512 * BPT
    wp = -(-(ctx + 1) // 512)
    stream = wp + lanes - 1
    return stream * page + (lanes - 1) * FIXED + BUDGET + (pages_today - stream) * page


def test_tp3_1m_step1():
    g = GOLD["tp3_1m_p8"]
    room = _room_today(g["today_pages"], 1048576, 8)
    today = P.plan(mk(room, 1048576, 8))
    assert today.pool_pages == g["today_pages"] and today.cache_bytes == BUDGET
    s1 = P.plan(mk(room, 1048576, 8, paged=True))
    assert s1.n_windows == g["expect"]["step1_n"]
    assert s1.stream_pages == g["expect"]["step1_stream_pages"]
    assert round(s1.cache_bytes / GiB, 1) == g["expect"]["step1_cache_gib_approx"]


def test_tp2_256k():
    g = GOLD["tp2_256k_p8"]["expect"]
    out = P.plan(mk(room_tp2(), 262144, 8))
    assert out.pool_pages == g["pool_pages"] and out.pool_tokens == g["pool_tokens"]
    assert P.windows_served(room_tp2(), 262144, BPT, FIXED) == g["windows_served"]
    # step 1 never holds fewer rows than windows in the same room
    s1 = P.plan(mk(room_tp2(), 262144, 8, paged=True))
    assert s1.n_windows == g["windows_served"]
    assert s1.pool_tokens >= g["windows_served"] * 262144


def test_tp2_128k_p4_queues_today():
    g = GOLD["tp2_128k_p4"]
    room = int(g["room_gib"] * GiB)
    today = P.plan(mk(room, 131072, 4))
    assert (today.pool_tokens < 4 * 65536) == g["expect"]["queues_four_64k"]
    s1 = P.plan(mk(room, 131072, 4, paged=True))
    assert s1.n_windows == g["expect"]["step1_n"]
    assert s1.pool_tokens >= 4 * 131072


def test_refuses_when_room_too_small():
    assert P.plan(mk(1 * GiB, 1048576, 8)) is None


@pytest.mark.parametrize("lanes", [1, 2, 8, 64])
def test_step1_never_holds_fewer_rows_than_windows(lanes):
    # issue #1313 step 1: "never holding fewer rows than windows would"
    for room_gib in [4, 9.5, 15.256, 38.12, 80, 200]:
        room = int(room_gib * GiB)
        for ctx in [4096, 131072, 262144, 1048576]:
            s1 = P.plan(mk(room, ctx, lanes, paged=True))
            if s1 is None:
                continue
            served = min(lanes, P.windows_served(room, ctx, BPT, FIXED))
            assert s1.pool_tokens >= served * ctx
