"""The benchmark's multi-rank logic on CPU with the gloo backend (world size
2): every rank is an independent replica of the layer with its own token
rows, and the job's time is the slowest rank's (max over ranks)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    bench.barrier(w)
    t = bench.max_over_ranks(1.5 + r, w)
    spec = synth.WORKLOADS["decode-t1"]
    x = synth.activations(spec, T=spec.T, start=r * spec.T)
    q.put((r, w, lr, t, x.float().sum().item()))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_distinct_rows():
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
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    assert all(o[3] == 2.5 for o in out)
    assert out[0][4] != out[1][4]  # replicas process different token rows
