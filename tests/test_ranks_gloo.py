"""Multi-rank host logic on CPU (gloo, world size 2): seeds, barrier, max-over-ranks rate."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    from dynamic_tree_speculative_gb300 import ranks as R
    info = R.rank_info()
    R.init(info, "gloo")
    R.barrier(info)
    # rank r "processed" 64 trees in (1 + r) seconds: whole-job rate = 128 / 2
    rate = R.whole_job_rate(64, 1.0 + rank, info)
    q.put((rank, R.rank_seed(5, rank), rate, R.max_over_ranks(rank * 3.0, info)))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0][1] == 5 and out[1][1] != 5
    assert out[0][2] == out[1][2] == 64.0
    assert out[0][3] == out[1][3] == 3.0
