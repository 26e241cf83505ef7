"""The N > 1 path on the CPU: two gloo ranks, no GPU.

Under torchrun each rank of ``bench.py`` runs the owner step of its own share of the owner plan
(MatrixFSDP §3: every matrix is whole on exactly one owner, so the shares are disjoint and need
no collective); the only cross-rank operation is the max of the timed region.  Here each rank
derives its share with the library's planner exactly as ``bench.py`` does, the shares are
gathered and checked to be disjoint and to cover the plan's ranks, and the max-reduction of a
rank-dependent time is checked.
"""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from matrix_optimizer_owner_gb300 import owner_step
        from workloads import get_config
        wl = get_config(2)
        params = [(p.rows, p.cols, p.block, p.is_matrix) for p in wl.params]
        shares = []
        for shift in range(rank, wl.world_size, world):      # this rank's plan ranks
            owner_rank = (wl.rank + shift) % wl.world_size    # as bench.Workload does
            lay = owner_step.owned_layout(params, wl.world_size, owner_rank)
            shares.append((owner_rank, tuple(lay.matrices), tuple(lay.tails)))
        gathered = [None] * world
        dist.all_gather_object(gathered, shares)
        t = torch.tensor([10.0 + rank])
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        q.put((rank, gathered, float(t.item())))
    finally:
        dist.destroy_process_group()


def test_two_ranks_own_disjoint_shares_and_reduce_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, gathered, tmax in results:
        assert tmax == 11.0
        all_shares = [s for rank_shares in gathered for s in rank_shares]
        ranks = sorted(s[0] for s in all_shares)
        assert ranks == list(range(8))
        mats = [m for s in all_shares for m in s[1]]
        tails = [t for s in all_shares for t in s[2]]
        assert len(mats) == len(set(mats)) == 224        # every Llama-3-8B matrix, once
        assert len(tails) == len(set(tails)) == 64       # every RMSNorm vector, once
