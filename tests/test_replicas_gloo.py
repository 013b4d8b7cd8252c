"""The replica path of the multi-GPU bench, on CPU with the gloo backend.

Two processes (world size 2, 127.0.0.1): each rank draws its own token rows,
reports a different step time; max_over_ranks must give both ranks the slowest
time, the whole-job rate must count both ranks' tokens over it, and the ranks'
rows must differ (independent replicas, no shared data).
"""

import socket

import torch.multiprocessing as mp

from pretraining_step_03_b300 import replicas, synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import os
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w, lr = replicas.rank_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    tok, _ = synth.zipf_rows(2, 16, 512, seed=replicas.data_seed(r))
    dist.barrier()
    ms = 10.0 + 2.0 * r                      # rank 1 is the slow one
    slowest = replicas.max_over_ranks(ms, dist)
    rate = replicas.job_rate(w, 2 * 16, slowest * 1e-3)
    out.put((r, w, lr, slowest, rate, tok.tobytes()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_count_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 and x[2] == x[0] for x in res)
    assert all(x[3] == 12.0 for x in res)                      # max over ranks
    assert all(abs(x[4] - 2 * 32 / 0.012) < 1e-6 for x in res)  # both ranks' tokens / slowest time
    assert res[0][5] != res[1][5]                               # independent data per rank


def test_single_process_defaults():
    assert replicas.max_over_ranks(3.5) == 3.5
    assert replicas.job_rate(1, 65536, 0.25) == 262144.0
    assert replicas.data_seed(0) != replicas.data_seed(1)
