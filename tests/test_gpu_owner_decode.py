"""Owner decode with the library's attention on the GPU: two ranks (processes on the one
GPU, gloo for the messages; their kernels never wait on each other), each holding only
the pages of the conversations it owns in a batch-invariant pool.  Every rank's heads
equal the single-rank engine's bit for bit (issue #1313, step 2, "Decode"), which needs
the batch-invariant split plan: an owner attends a different batch than one rank would."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _case():
    from paged_mla_kv_gb300 import synth as Y
    lens = [3000, 700, 9000, 64, 20000, 2600]
    return Y.custom("owner_gpu", 93, lens=lens, R=2, H=64)


def _sub(w, streams):
    """The conversations `streams` of w as their own workload (same rows, same queries)."""
    from paged_mla_kv_gb300 import synth as Y
    ws = Y.custom(w.name + "_sub", w.seed, lens=[int(w.lens[s]) for s in streams], R=w.R, H=w.H)
    ws.page_rows = lambda c, ss, p: w.page_rows(c, streams[ss], p)
    return ws


def _gpu_attend(w, streams):
    from paged_mla_kv_gb300 import binding as B
    from paged_mla_kv_gb300.harness import Resident
    ws = _sub(w, streams)
    res = Resident(ws, invariant=True)

    def attend(listed, q):
        assert list(listed) == list(streams)
        qd = q.cuda()
        out = torch.empty((len(streams), w.R, w.H, 512), dtype=torch.bfloat16, device="cuda")
        B.tf_paged_mla_attend(res.pool, 0, res.pt, res.max_pages, res.lens, qd, w.scale, out, None, res.workspace())
        torch.cuda.synchronize()
        rc, _ = res.pool.last_error()
        assert rc == 0
        return out.cpu()
    return attend


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    from paged_mla_kv_gb300 import build as BUILD
    from paged_mla_kv_gb300 import owner as OW
    BUILD.build()
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = _case()
    owners = OW.choose_owners([60, 60], OW.pages_of(w.lens))
    od = OW.OwnerDecode(dist, owners, w.H)
    attend = _gpu_attend(w, od.owned) if od.owned else None
    qall = torch.from_numpy(w.q(0).view(np.int16)).view(torch.bfloat16)
    out = od.step(qall[:, :, od.hs].contiguous(), attend)
    q.put((rank, owners, out.view(torch.int16).numpy().copy()))
    dist.barrier()
    dist.destroy_process_group()


def test_owner_decode_on_the_gpu_equals_one_rank_bit_for_bit():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=600) for _ in range(2)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    from paged_mla_kv_gb300 import build as BUILD
    from paged_mla_kv_gb300 import owner as OW
    BUILD.build()
    w = _case()
    owners = got[0][1]
    assert sorted(set(owners)) == [0, 1]
    qall = torch.from_numpy(w.q(0).view(np.int16)).view(torch.bfloat16)
    ref = _gpu_attend(w, list(range(w.S)))(list(range(w.S)), qall).view(torch.int16).numpy()
    for rank, _, out in got:
        assert np.array_equal(out, ref[:, :, OW.head_slice(w.H, 2, rank)])
