"""The kv_pool plan arithmetic in integers -- TEST INFRASTRUCTURE ONLY.

Follows issue #1313 ("Why", third bullet; "Proposal, in two steps", step 1.1):

* the engine's own sequence gets one window of pages first:
  window_pages = ceil((context + lookahead) / page_rows)        (2,049 at 1M)
* today's order then funds a page a stream for the other lanes - 1 streams
  and each of those streams' fixed part, then the prompt cache (up to its
  budget), then the other pages from whatever room is left;
* step 1 ("engine_paged") sets aside, before the cache, the pages of
  n = min(lanes, 1 + (room - window_bytes) / (window_bytes + fixed)) windows
  (integer division, at least one window); the streams then hold
  max(n windows, one window plus a page for each other stream).

Readings where the text is silent:
* "180 MiB fixed" is charged once for each of the lanes - 1 other streams;
* every quantity is in bytes; `/` is integer division;
* the plan refuses (None) when the room cannot hold the streams' pages and
  fixed parts.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class PlanIn:
    room_bytes: int
    context_tokens: int
    lanes: int
    bytes_per_token: int
    fixed_bytes: int
    cache_budget_bytes: int
    page_rows: int = 512
    lookahead: int = 1
    engine_paged: bool = False


@dataclass(frozen=True)
class PlanOut:
    n_windows: int
    window_pages: int
    stream_pages: int
    cache_bytes: int
    other_pages: int
    pool_pages: int
    pool_tokens: int


def plan(p: PlanIn):
    page_bytes = p.page_rows * p.bytes_per_token
    window_pages = -(-(p.context_tokens + p.lookahead) // p.page_rows)
    window_bytes = window_pages * page_bytes
    if p.engine_paged:
        spare = p.room_bytes - window_bytes
        n = 1 + (spare // (window_bytes + p.fixed_bytes) if spare > 0 else 0)
        n = max(1, min(p.lanes, n))
    else:
        n = 1
    stream_pages = max(n * window_pages, window_pages + (p.lanes - 1))
    charged = stream_pages * page_bytes + (p.lanes - 1) * p.fixed_bytes
    if charged > p.room_bytes:
        return None
    cache = min(p.cache_budget_bytes, p.room_bytes - charged)
    other = (p.room_bytes - charged - cache) // page_bytes
    pool_pages = stream_pages + other
    return PlanOut(n, window_pages, stream_pages, cache, other, pool_pages, pool_pages * p.page_rows)


def windows_served(room_bytes: int, context_tokens: int, bytes_per_token: int, fixed_bytes: int) -> int:
    """Streams that whole windows (no pages) fit in a room: each costs context x bytes + fixed
    (issue #1313 opening: seven more 1M windows need 90.48 GiB)."""
    return room_bytes // (context_tokens * bytes_per_token + fixed_bytes)
