"""Make a workload resident on the GPU through the library's own calls.

Given a synth.Workload this takes pages from a tf_kvpool (sharing prefix pages
by reference, as kept prompt states are adopted at the head of a new stream's
lease in PR #1732), builds the per-stream page tables, and writes every row with
tf_paged_append.  With windowed=True it uses the null table instead: stream s
owns pool pages s*max_pages .. s*max_pages + max_pages - 1, pages in order.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from . import synth as Y


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


class Resident:
    def __init__(self, w: Y.Workload, poison: bool = True, pool_seed: int | None = None, windowed: bool = False,
                 caches=None, chunk_rows: int = 65536, device="cuda", extra_pages: int = 0,
                 invariant: bool = False, fp8: bool = False):
        self.w = w
        self.windowed = windowed
        self.device = device
        self.max_pages = w.max_pages
        npages = (w.S * self.max_pages if windowed else w.pool_pages) + extra_pages
        seed = (w.seed * 1000003 + 7) if pool_seed is None else pool_seed
        self.pool = B.KVPool(w.num_caches, npages, poison=poison, seed=seed, device=device, invariant=invariant,
                             fp8=fp8)
        self.caches = list(range(w.num_caches)) if caches is None else list(caches)
        pt = np.full((w.S, self.max_pages), -1, np.int32)
        if windowed:
            ids = self.pool.take(w.S * self.max_pages)   # poisons every page, as a take does
            pt[:] = np.arange(w.S * self.max_pages, dtype=np.int32).reshape(w.S, self.max_pages)
            self.pt = None
        else:
            for s in range(w.S):
                src, n = w.share[s]
                if n:
                    pt[s, :n] = pt[src, :n]
                    self.pool.ref(pt[src, :n])
                own = w.own_pages(s)
                pt[s, n:n + own] = self.pool.take(own)
            self.pt = torch.from_numpy(pt).to(device)
        self.pt_host = pt
        self.lens = np.asarray(w.lens, np.int64)
        for c in self.caches:
            for s in range(w.S):
                lo = 0 if windowed else w.shared_pages(s) * Y.PAGE_ROWS
                self.append_rows(c, s, lo, int(w.lens[s]), chunk_rows)
        torch.cuda.synchronize()

    def stream_pt(self, s: int):
        return None if self.pt is None else self.pt[s:s + 1]

    def append_rows(self, cache: int, s: int, lo: int, hi: int, chunk_rows: int = 65536) -> None:
        """Write logical rows [lo, hi) of stream s into its pages."""
        for a in range(lo, hi, chunk_rows):
            b = min(hi, a + chunk_rows)
            lat, rope = self.w.stream_rows(cache, s, a, b)
            tl = bf16_tensor(lat, self.device).view(1, b - a, 512)
            tr = bf16_tensor(rope, self.device).view(1, b - a, 64)
            if self.pt is None:
                # windowed: one stream at a time through a null table needs S == 1 addressing;
                # its window starts at page s * max_pages, so shift by whole windows
                pos = np.array([s * self.max_pages * Y.PAGE_ROWS + a], np.int64)
                B.tf_paged_append(self.pool, cache, None, self.max_pages * self.w.S, pos, tl, tr)
            else:
                B.tf_paged_append(self.pool, cache, self.stream_pt(s), self.max_pages, np.array([a], np.int64),
                                  tl, tr)

    def current_rows(self, cache: int):
        """The rows each stream appends this step (its last R rows), as device tensors [S][R][...]."""
        R = self.w.R
        lat = np.stack([self.w.stream_rows(cache, s, int(self.lens[s]) - R, int(self.lens[s]))[0]
                        for s in range(self.w.S)])
        rope = np.stack([self.w.stream_rows(cache, s, int(self.lens[s]) - R, int(self.lens[s]))[1]
                         for s in range(self.w.S)])
        return bf16_tensor(lat, self.device), bf16_tensor(rope, self.device)

    def append_current(self, cache: int, lat, rope) -> None:
        B.tf_paged_append(self.pool, cache, self.pt, self.max_pages, self.lens - self.w.R, lat, rope)

    def q(self, cache: int = 0) -> torch.Tensor:
        return bf16_tensor(self.w.q(cache), self.device)

    def workspace(self) -> torch.Tensor | None:
        n = B.tf_paged_mla_workspace_bytes(self.pool, self.w.S, self.w.R, self.w.H, self.lens)
        return torch.empty(max(n, 256), dtype=torch.uint8, device=self.device) if n else None

    def attend(self, q, cache: int = 0, out=None, lse=None, ws=None, scale=None):
        w = self.w
        if out is None:
            out = torch.empty((w.S, w.R, w.H, 512), dtype=torch.bfloat16, device=self.device)
        if lse is None:
            lse = torch.empty((w.S, w.R, w.H), dtype=torch.float32, device=self.device)
        if ws is None:
            ws = self.workspace()
        B.tf_paged_mla_attend(self.pool, cache, self.pt, self.max_pages, self.lens, q,
                              w.scale if scale is None else scale, out, lse, ws)
        return out, lse
