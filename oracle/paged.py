"""Expected pool images for paged appends and kept-state copies -- TEST INFRASTRUCTURE ONLY.

The pool is modelled as a uint16 array [caches][pages][PAGE_WORDS]: one page of
one cache is a latent block (512 rows x 512 bf16) followed by a rope block
(512 rows x 64 bf16).  Row `pos` of a stream lives in logical page pos // 512
at row pos % 512, and the logical page maps to a pool page through the
stream's page table, the way issue #1142 ("GLM declares a kv_pool.Layout")
has the cache kernels take a page table plus the elements between pages.  A
missing table keeps contiguous rows (same passage): stream s then owns pool
pages s*max_pages .. s*max_pages + max_pages - 1, a window laid out as pages in
order (issue #1313, step 1.3).

A kept state copies each cache's first `at` rows and nothing past them
(issue #1142, piece 1: keepAs / restoreState copy the first `at` rows; rows
past `at` are never read).
"""
from __future__ import annotations

import numpy as np

PAGE_ROWS = 512
LAT = 512
ROPE = 64
PAGE_WORDS = PAGE_ROWS * (LAT + ROPE)
ROPE_OFF = PAGE_ROWS * LAT


def new_pool(caches: int, pages: int, fill: int = 0x7FC0) -> np.ndarray:
    return np.full((caches, pages, PAGE_WORDS), fill, np.uint16)


def pool_page(page_table, s: int, logical_page: int, max_pages: int) -> int:
    if page_table is None:
        return s * max_pages + logical_page
    return int(page_table[s][logical_page])


def append(pool: np.ndarray, cache: int, page_table, max_pages: int, pos0, latent, rope) -> None:
    """Write rows pos0[s] + i (i < n) of every stream s into their pages.

    latent: [S][n][512], rope: [S][n][64] bf16 bits.
    """
    S, n = latent.shape[0], latent.shape[1]
    for s in range(S):
        for i in range(n):
            pos = int(pos0[s]) + i
            page = pool_page(page_table, s, pos // PAGE_ROWS, max_pages)
            row = pos % PAGE_ROWS
            pool[cache, page, row * LAT:(row + 1) * LAT] = latent[s, i]
            pool[cache, page, ROPE_OFF + row * ROPE:ROPE_OFF + (row + 1) * ROPE] = rope[s, i]


def state_copy_rows(pool: np.ndarray, cache: int, src_pages, dst_pages, at: int) -> None:
    """Copy rows [0, at) of one cache (or every cache when cache < 0) from src to dst pages."""
    caches = range(pool.shape[0]) if cache < 0 else [cache]
    for c in caches:
        for j in range(at):
            sp, dp, row = int(src_pages[j // PAGE_ROWS]), int(dst_pages[j // PAGE_ROWS]), j % PAGE_ROWS
            pool[c, dp, row * LAT:(row + 1) * LAT] = pool[c, sp, row * LAT:(row + 1) * LAT]
            pool[c, dp, ROPE_OFF + row * ROPE:ROPE_OFF + (row + 1) * ROPE] = \
                pool[c, sp, ROPE_OFF + row * ROPE:ROPE_OFF + (row + 1) * ROPE]


def gather_rows(pool: np.ndarray, cache: int, page_table, s: int, max_pages: int, n: int):
    """Read a stream's logical rows [0, n) back out of the pool: (latent [n][512], rope [n][64])."""
    lat = np.empty((n, LAT), np.uint16)
    rope = np.empty((n, ROPE), np.uint16)
    for pos in range(n):
        page = pool_page(page_table, s, pos // PAGE_ROWS, max_pages)
        row = pos % PAGE_ROWS
        lat[pos] = pool[cache, page, row * LAT:(row + 1) * LAT]
        rope[pos] = pool[cache, page, ROPE_OFF + row * ROPE:ROPE_OFF + (row + 1) * ROPE]
    return lat, rope
