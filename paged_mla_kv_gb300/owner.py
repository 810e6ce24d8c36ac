"""Owner decode across ranks: the host side of the latent split (issue #1313, step 2).

A conversation's latent pages all live on one rank, its owner.  Heads are split across
ranks (tensor parallel), so a decode step moves queries instead of rows:
- every rank sends the absorbed queries of its head slice, for the rows other ranks own,
  to their owners;
- each owner runs attention for every head of the rows it owns, over its own pages,
  with the same attention call a single rank would make;
- each owner returns to every rank the outputs of that rank's heads.
Every (row, head) output thus comes from the same call over the same bytes as on one
rank, so every rank's outputs equal the unsharded engine's bit for bit.

This module is the routing only: who owns what, what moves where, and in which order.
The attention itself is a callable the caller passes in (on a GPU, the library's
tf_paged_mla_attend over the owner's pool); nothing here computes scores.  Messages go
over torch.distributed point-to-point calls, so any backend with send/recv serves.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


def choose_owners(free_pages, pages_needed) -> list:
    """Owner of each conversation, in admission order.

    The "Owner" bullet of issue #1313, step 2: a conversation goes to the rank with the
    most free latent pages at its admission (ties to the lowest rank), and that rank's
    free count drops by the conversation's pages.  Every rank computes the same answer
    from the same book, so no message is needed.  Raises ValueError when no rank can
    hold a conversation.
    """
    free = [int(x) for x in free_pages]
    owners = []
    for need in pages_needed:
        r = max(range(len(free)), key=lambda i: (free[i], -i))
        if free[r] < int(need):
            raise ValueError(f"no rank has {int(need)} free latent pages (most: {free[r]})")
        free[r] -= int(need)
        owners.append(r)
    return owners


def head_slice(H: int, world: int, rank: int) -> slice:
    """The heads a rank holds queries and outputs for (H divisible by the world size)."""
    if H % world:
        raise ValueError(f"{H} heads do not split over {world} ranks")
    n = H // world
    return slice(rank * n, (rank + 1) * n)


@dataclass
class StepBytes:
    sent_queries: int = 0
    sent_outputs: int = 0


class OwnerDecode:
    """One rank's side of owner decode for a fixed set of conversations.

    owners: owner rank of every conversation (choose_owners).  H: heads of the model;
    this rank holds heads head_slice(H, world, rank) of every row.
    """

    def __init__(self, dist, owners, H: int):
        self.dist = dist
        self.world = dist.get_world_size()
        self.rank = dist.get_rank()
        self.owners = [int(o) for o in owners]
        self.H = H
        self.hs = head_slice(H, self.world, self.rank)
        self.owned = [s for s, o in enumerate(self.owners) if o == self.rank]
        self.bytes = StepBytes()

    def step(self, q_local: torch.Tensor, attend) -> torch.Tensor:
        """One decode step.

        q_local: [S][R][H/W][576] bf16 (CPU): this rank's heads of every conversation.
        attend(streams, q): attention of the listed conversations, all heads, over this
        rank's pages; q is [len(streams)][R][H][576]; returns [len(streams)][R][H][512].
        Returns [S][R][H/W][512]: this rank's heads of every conversation's output.
        """
        d, W, me = self.dist, self.world, self.rank
        S, R, hw, dk = q_local.shape
        assert S == len(self.owners) and hw * W == self.H
        # 1. queries of rows owned elsewhere go to their owners; an owner assembles all heads
        full = torch.empty((len(self.owned), R, self.H, dk), dtype=q_local.dtype)
        slot = {s: i for i, s in enumerate(self.owned)}
        for i, s in enumerate(self.owned):
            full[i, :, self.hs] = q_local[s]
        self.bytes = StepBytes()
        for src in range(W):
            for dst in range(W):
                if src == dst:
                    continue
                rows = [s for s in range(S) if self.owners[s] == dst]
                if not rows:
                    continue
                if me == src:
                    msg = q_local[rows].contiguous()
                    d.send(msg, dst)
                    self.bytes.sent_queries += msg.numel() * msg.element_size()
                elif me == dst:
                    msg = torch.empty((len(rows), R, hw, dk), dtype=q_local.dtype)
                    d.recv(msg, src)
                    hs = head_slice(self.H, W, src)
                    for j, s in enumerate(rows):
                        full[slot[s], :, hs] = msg[j]
        # 2. the owner computes every head of its rows, as a single rank would
        out_owned = attend(self.owned, full) if self.owned else None
        # 3. every rank receives the outputs of its own heads
        out = torch.empty((S, R, hw, 512), dtype=q_local.dtype)
        for i, s in enumerate(self.owned):
            out[s] = out_owned[i, :, self.hs]
        for src in range(W):
            for dst in range(W):
                if src == dst:
                    continue
                rows = [s for s in range(S) if self.owners[s] == src]
                if not rows:
                    continue
                if me == src:
                    hs = head_slice(self.H, W, dst)
                    msg = torch.stack([out_owned[slot[s], :, hs] for s in rows]).contiguous()
                    d.send(msg, dst)
                    self.bytes.sent_outputs += msg.numel() * msg.element_size()
                elif me == dst:
                    msg = torch.empty((len(rows), R, hw, 512), dtype=q_local.dtype)
                    d.recv(msg, src)
                    for j, s in enumerate(rows):
                        out[s] = msg[j]
        return out


def expected_step_bytes(owners, rank: int, world: int, R: int, H: int, dk: int = 576) -> StepBytes:
    """What one rank sends in a step: its head slice of the queries of every row owned
    elsewhere (R x H/W x 576 bf16 a row: the page's R x heads/W x 512 plus the rope
    part the scores need) and, as an owner, every other rank's heads of its rows' outputs."""
    hw = H // world
    elsewhere = sum(1 for o in owners if o != rank)
    mine = sum(1 for o in owners if o == rank)
    return StepBytes(sent_queries=elsewhere * R * hw * dk * 2, sent_outputs=mine * (world - 1) * R * hw * 512 * 2)


def pages_of(lens, page_rows: int = 512) -> np.ndarray:
    return (np.asarray(lens, np.int64) + page_rows - 1) // page_rows
