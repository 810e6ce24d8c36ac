"""Owner decode across CPU ranks (gloo): queries move to each conversation's owner, the
owner computes every head, outputs come back, and every rank's heads equal the
single-rank engine's bit for bit (issue #1313, step 2, "Owner" and "Decode").  The
attention each owner runs here is the fp64 oracle rounded to bf16 -- the same callable
the single-rank reference uses -- so the test checks the routing, not the kernel."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_mla_kv_gb300 import owner as OW
from paged_mla_kv_gb300 import synth as Y


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _case():
    lens = [3000, 700, 5200, 64, 1500, 2600, 900]
    return Y.custom("owner", 91, lens=lens, R=2, H=12)


def _attend_fn(w, allowed):
    """Oracle attention of the listed conversations, all heads, as bf16 tensors."""
    from oracle import attend as OA

    def attend(streams, q):
        res = []
        for i, s in enumerate(streams):
            assert s in allowed, f"conversation {s} is not owned here"
            lat, rope = w.stream_rows(0, s)
            qb = q[i].contiguous().view(torch.int16).numpy().view(np.uint16)
            o, _ = OA.attend_stream(qb, lat, rope, w.scale, threads=1)
            res.append(torch.from_numpy(o.astype(np.float32)).to(torch.bfloat16).reshape(w.R, w.H, 512))
        return torch.stack(res)
    return attend


def _worker(rank, world, port, free, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = _case()
    owners = OW.choose_owners(free, OW.pages_of(w.lens))
    od = OW.OwnerDecode(dist, owners, w.H)
    qall = torch.from_numpy(w.q(0).view(np.int16)).view(torch.bfloat16)        # [S][R][H][576]
    q_local = qall[:, :, od.hs].contiguous()
    out = od.step(q_local, _attend_fn(w, set(od.owned)))
    q.put((rank, owners, out.view(torch.int16).numpy().copy(), od.bytes.sent_queries, od.bytes.sent_outputs))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,free", [(2, [40, 40]), (3, [9, 30, 20])])
def test_owner_decode_equals_single_rank_bit_for_bit(world, free):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, free, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=180) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    w = _case()
    owners = got[0][1]
    assert all(g[1] == owners for g in got)                  # every rank derived the same book
    assert sorted(set(owners)) != [0] or world == 1           # the rows really are spread
    # the single-rank engine: every conversation, every head, on one rank
    qall = torch.from_numpy(w.q(0).view(np.int16)).view(torch.bfloat16)
    ref = _attend_fn(w, set(range(w.S)))(list(range(w.S)), qall).view(torch.int16).numpy()
    for rank, _, out, sq, so in got:
        hs = OW.head_slice(w.H, world, rank)
        assert np.array_equal(out, ref[:, :, hs])
        exp = OW.expected_step_bytes(owners, rank, world, w.R, w.H)
        assert (sq, so) == (exp.sent_queries, exp.sent_outputs)


def test_owner_choice_follows_the_most_free_pages():
    assert OW.choose_owners([10, 12, 12], [5, 4, 8, 3]) == [1, 2, 0, 2]
    assert OW.choose_owners([5, 5], [1, 1, 1]) == [0, 1, 0]   # ties go to the lowest rank
    with pytest.raises(ValueError):
        OW.choose_owners([3, 2], [4])
    with pytest.raises(ValueError):
        OW.head_slice(64, 3, 0)
    # the page's TP=2 cost: R x 32 heads x 512 bf16 = R x 32 KiB of latent query a row; the
    # rope part the scores also need adds 64 values a head
    b = OW.expected_step_bytes([1], 0, 2, R=1, H=64)
    assert b.sent_queries == 32 * 576 * 2 and b.sent_outputs == 0
