"""Seeded synthetic inputs for the paged latent-cache workloads.

This module is shared by the CPU oracle and by the CUDA path, so it holds none
of the attention arithmetic: only random draws, their bf16 encoding, the length
mixes and the prefix-sharing structure of the workloads described on the
TensorFold pages (issues #1313 and #1142, PR #1732) and on the chunked-prefill
memory note (section 1, the T x L pairs).

Every array of values is drawn from a counter-keyed PCG64 stream, so a page's
rows depend only on (seed, cache, owning stream, logical page) and never on the
order in which a harness asks for them.  A stream that shares a prefix reads
the owning stream's pages, exactly as a radix prompt store's kept pages would
be adopted at the head of a new stream's lease (PR #1732, "What this changes").
"""
from __future__ import annotations

from dataclasses import dataclass, field
import numpy as np

LATENT = 512          # latent values a row (bf16)
ROPE = 64             # rope-key values a row (bf16)
DK = LATENT + ROPE    # query width a head: absorbed latent part + rope part
PAGE_ROWS = 512       # rows a page (issue #1313 step 1.3; issue #1142 question 2)
ROW_BYTES = DK * 2    # 1,152 bytes a row and cache as stored here


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


BF16_NAN = np.uint16(0x7FC0)   # the poison pattern for taken-but-unwritten rows


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(k) & 0xFFFFFFFF for k in key]))


@dataclass
class Workload:
    """One batch of streams over a paged latent cache.

    lens[s] counts rows after the current R rows are appended; query row r of
    stream s sits at position lens[s] - R + r and sees keys 0..that position.
    share[s] = (src, n) means stream s's first n logical pages are stream src's
    first n pages (held by reference); n = 0 means no sharing.
    """
    name: str
    seed: int
    S: int
    R: int
    H: int
    lens: np.ndarray
    share: list
    pool_pages: int
    num_caches: int = 1
    scale: float = 1.0 / np.sqrt(DK)
    value_std: float = 0.1
    q_std: float = 0.1
    ramp: float = 0.0          # > 0: rope column 0 grows with position (forces running-max updates)
    notes: str = ""
    extra: dict = field(default_factory=dict)

    # ---- sizes -------------------------------------------------------------
    def pages_of(self, s: int) -> int:
        return -(-int(self.lens[s]) // PAGE_ROWS)

    def shared_pages(self, s: int) -> int:
        return int(self.share[s][1])

    def own_pages(self, s: int) -> int:
        return self.pages_of(s) - self.shared_pages(s)

    @property
    def max_pages(self) -> int:
        return max(self.pages_of(s) for s in range(self.S))

    def pages_needed(self) -> int:
        return sum(self.own_pages(s) for s in range(self.S))

    def kv_bytes(self) -> int:
        """Key/value bytes read once a stream (shared pages counted per reader)."""
        return int(np.sum(self.lens)) * ROW_BYTES

    # ---- values ------------------------------------------------------------
    def _owner(self, s: int, page: int) -> int:
        src, n = self.share[s]
        while n and page < n:
            s = src
            src, n = self.share[s]
        return s

    def page_rows(self, cache: int, s: int, page: int):
        """Full 512-row content of logical page `page` of stream s: (latent, rope) bf16 bits."""
        owner = self._owner(s, page)
        g = _rng(self.seed, 7919, cache, owner, page)
        lat = f32_to_bf16_bits(g.standard_normal((PAGE_ROWS, LATENT), dtype=np.float32) * np.float32(self.value_std))
        rope = g.standard_normal((PAGE_ROWS, ROPE), dtype=np.float32) * np.float32(self.value_std)
        if self.ramp > 0.0:
            pos = np.arange(page * PAGE_ROWS, (page + 1) * PAGE_ROWS, dtype=np.float64)
            rope[:, 0] = (self.ramp * pos / max(1, int(self.lens.max()))).astype(np.float32)
        return lat, f32_to_bf16_bits(rope)

    def stream_rows(self, cache: int, s: int, lo: int = 0, hi: int | None = None):
        """Contiguous logical rows [lo, hi) of stream s: (latent [n][512], rope [n][64]) bf16 bits."""
        n = int(self.lens[s])
        hi = n if hi is None else min(hi, n)
        lat = np.empty((max(0, hi - lo), LATENT), np.uint16)
        rope = np.empty((max(0, hi - lo), ROPE), np.uint16)
        p0, p1 = lo // PAGE_ROWS, -(-hi // PAGE_ROWS)
        for p in range(p0, p1):
            a, b = max(lo, p * PAGE_ROWS), min(hi, (p + 1) * PAGE_ROWS)
            if a >= b:
                continue
            pl, pr = self.page_rows(cache, s, p)
            lat[a - lo:b - lo] = pl[a - p * PAGE_ROWS:b - p * PAGE_ROWS]
            rope[a - lo:b - lo] = pr[a - p * PAGE_ROWS:b - p * PAGE_ROWS]
        return lat, rope

    def q(self, cache: int = 0) -> np.ndarray:
        """Absorbed queries, bf16 bits [S][R][H][576]."""
        g = _rng(self.seed, 104729, cache)
        q = g.standard_normal((self.S, self.R, self.H, DK), dtype=np.float32) * np.float32(self.q_std)
        if self.ramp > 0.0:
            q[..., LATENT] = 1.0
        return f32_to_bf16_bits(q)


def _lens(rng: np.random.Generator, n: int, lo: int, hi: int) -> np.ndarray:
    return rng.integers(lo, hi + 1, size=n).astype(np.int64)


def tiny_decode(seed: int = 1) -> Workload:
    """1 stream, 16 heads, 1 query row, 2,048 rows = 4 pages in a 16-page pool."""
    return Workload("tiny_decode", seed, S=1, R=1, H=16, lens=np.array([2048], np.int64),
                    share=[(-1, 0)], pool_pages=16,
                    notes="4 pages placed by a seeded permutation of a 16-page pool")


def decode_batch(seed: int = 2, S: int = 8, H: int = 64, lo: int = 4096, hi: int = 65536,
                 n_shared: int = 4, shared_pages: int = 16, spare_frac: float = 0.10) -> Workload:
    """8 streams, 64 heads, 1 row; lengths U[4,096, 65,536]; streams 0-3 share 8,192 rows of pages."""
    g = _rng(seed, 17)
    lens = _lens(g, S, lo, hi)
    share = [(-1, 0)] * S
    for s in range(1, min(n_shared, S)):
        share[s] = (0, min(shared_pages, (int(lens[s]) - 1) // PAGE_ROWS, (int(lens[0]) - 1) // PAGE_ROWS))
    w = Workload("decode_batch", seed, S=S, R=1, H=H, lens=lens, share=share, pool_pages=0)
    need = w.pages_needed()
    w.pool_pages = need + max(1, int(round(spare_frac * need)))
    w.notes = "pool shuffled by a seeded permutation; spare pages poisoned"
    return w


def long_window(seed: int = 3, S: int = 8, H: int = 64, long_len: int = 1048576, short_hi: int = 8192,
                pool_pages: int = 2056) -> Workload:
    """Stream 0 at 1,048,576 rows, 7 streams at U[2, 8,192] reading stream 0's pages; 2 causal rows."""
    g = _rng(seed, 17)
    lens = np.concatenate([[long_len], _lens(g, S - 1, 2, short_hi)]).astype(np.int64)
    share = [(-1, 0)] + [(0, (int(n) - 1) // PAGE_ROWS) for n in lens[1:]]
    w = Workload("long_window", seed, S=S, R=2, H=H, lens=lens, share=share, pool_pages=pool_pages,
                 notes="streams 1-7 read stream 0's first floor((len-1)/512) pages and own one tail page")
    assert w.pages_needed() <= pool_pages, (w.pages_needed(), pool_pages)
    return w


def chunked_prefill(seed: int = 4, T: int = 2048, L: int = 100000, H: int = 64) -> Workload:
    """One stream: a T-row chunk at positions L..L+T-1 against its L-row prefix plus the causal triangle."""
    lens = np.array([L + T], np.int64)
    w = Workload(f"prefill_T{T}_L{L}", seed, S=1, R=T, H=H, lens=lens, share=[(-1, 0)], pool_pages=0)
    w.pool_pages = w.pages_needed() + 1
    return w


def full_model(seed: int = 5, caches: int = 12, S: int = 16, H: int = 64, window: int = 40960,
               at: int = 32768) -> Workload:
    """12 caches, 16 streams at a full 40,960-row window, one row a step, then a 32,768-row state copy."""
    lens = np.full(S, window, np.int64)
    w = Workload("full_model", seed, S=S, R=1, H=H, lens=lens, share=[(-1, 0)] * S, pool_pages=0,
                 num_caches=caches)
    w.pool_pages = w.pages_needed() + -(-at // PAGE_ROWS)
    w.extra["at"] = at
    return w


def custom(name: str, seed: int, lens, R: int, H: int, share=None, pool_pages: int | None = None,
           num_caches: int = 1, **kw) -> Workload:
    lens = np.asarray(lens, np.int64)
    S = len(lens)
    share = share if share is not None else [(-1, 0)] * S
    w = Workload(name, seed, S=S, R=R, H=H, lens=lens, share=share, pool_pages=0, num_caches=num_caches, **kw)
    w.pool_pages = pool_pages if pool_pages is not None else w.pages_needed() + 2
    return w


def listed_rows(seed: int, lens, n: int, repeats: bool = False) -> list:
    """Seeded lists of rows for attention over listed rows: for stream s, min(n, len_s)
    distinct rows of [0, len_s) in a random order (or n rows drawn with repeats)."""
    g = _rng(seed, 4099)
    out = []
    for L in np.asarray(lens, np.int64):
        L = int(L)
        if repeats:
            out.append(g.integers(0, L, n).astype(np.int32))
        else:
            out.append(g.choice(L, min(n, L), replace=False).astype(np.int32))
    return out


def sparse_decode(seed: int = 6, S: int = 64, H: int = 64, lo: int = 4096, hi: int = 65536,
                  n: int = 2048) -> Workload:
    """64 streams, 64 heads, 1 row, lengths U[4,096, 65,536]; each attends 2,048 listed rows."""
    g = _rng(seed, 17)
    lens = _lens(g, S, lo, hi)
    w = Workload("sparse_decode", seed, S=S, R=1, H=H, lens=lens, share=[(-1, 0)] * S, pool_pages=0)
    w.pool_pages = w.pages_needed() + 2
    w.extra = dict(w.extra or {}, nidx=n)
    w.notes = "keys: 2,048 seeded distinct rows of each stream (listed_rows), in a random order"
    return w


def fp8_decode(seed: int = 2) -> Workload:
    """The decode batch (same lengths, sharing and rows) held on FP8 pages."""
    w = decode_batch(seed)
    w.name = "fp8_decode"
    w.extra = dict(w.extra or {}, fp8=True)
    w.notes = "decode_batch's rows, stored as E4M3 codes with one fp32 scale a row"
    return w


def sparse_fp8_decode(seed: int = 6) -> Workload:
    """The listed-row decode (same streams, rows and lists) held on FP8 pages."""
    w = sparse_decode(seed)
    w.name = "sparse_fp8_decode"
    w.extra = dict(w.extra or {}, fp8=True)
    w.notes += "; rows stored as E4M3 codes with one fp32 scale a row"
    return w


def permutation(seed: int, n: int) -> np.ndarray:
    """A seeded permutation of n pool pages (int32)."""
    return _rng(seed, 31337).permutation(n).astype(np.int32)


@dataclass
class TopkWorkload:
    """Rows of indexer logits for the blocked top-k: row t has lens[t] keys in play."""
    name: str
    seed: int
    rows: int
    n: int
    k: int
    lens: np.ndarray
    grid: float
    notes: str = ""


def topk_logits(seed: int, row_ids, n: int, grid: float = 1.0 / 64) -> np.ndarray:
    """float32 [len(row_ids)][n]: standard normal scores rounded to multiples of `grid`, so equal
    scores are common (the indexer's scores come out of low-precision products); row r depends
    only on (seed, r)."""
    out = np.empty((len(row_ids), n), dtype=np.float32)
    for i, r in enumerate(row_ids):
        x = _rng(seed, 7919, int(r)).standard_normal(n, dtype=np.float32)
        out[i] = np.round(x / grid) * grid if grid else x
    return out


def topk_prefill(seed: int = 7, T: int = 2048, L: int = 100000, k: int = 512) -> TopkWorkload:
    """A 2,048-row chunk over a 100,000-key prefix (the chunked-prefill note, section 1); row t
    sees L - T + 1 + t keys (causal); the top-512 of each row (section 2.3)."""
    lens = (L - T + 1 + np.arange(T)).astype(np.int32)
    return TopkWorkload("topk_prefill", seed, T, L, k, lens, 1.0 / 64,
                        "scores N(0,1) rounded to 1/64; causal row lengths")


TOPK_WORKLOADS = {"topk_prefill": topk_prefill}


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "decode_batch": decode_batch,
    "long_window": long_window,
    "prefill_100k": lambda seed=4: chunked_prefill(seed, 2048, 100000),
    "prefill_208k": lambda seed=4: chunked_prefill(seed, 1024, 208000),
    "full_model": full_model,
    "sparse_decode": sparse_decode,
    "fp8_decode": fp8_decode,
    "sparse_fp8_decode": sparse_fp8_decode,
}
