"""Multi-rank host logic of bench.py on CPU: two gloo ranks (no GPU). Each rank draws
its own batch (distinct seeds: weak scaling, no data-path collective) and the timed
region is the max over ranks."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        bench.barrier(ws)
        t_max = bench.reduce_max(1.5 + rank, ws)
        q.put((r, local, ws, bench.shard_seed(3, r), t_max))
    finally:
        dist.destroy_process_group()


def test_two_rank_host_logic():
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
    assert [r[0] for r in res] == [0, 1] and [r[1] for r in res] == [0, 1] and all(r[2] == 2 for r in res)
    assert res[0][3] != res[1][3]  # each rank draws its own batch
    assert all(r[4] == 2.5 for r in res)  # max over ranks


def test_single_rank_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.reduce_max(3.25, 1) == 3.25


def test_kernel_work_matches_config_flops():
    import dit_inputs as di
    cfg = di.CONFIGS["1024px"]
    work = bench.kernel_work(cfg)
    flops = sum(a for b, a, u in work.values() if u == "flops")
    assert abs(flops - di.config_flops(cfg)) / di.config_flops(cfg) < 1e-12
    assert abs(di.config_flops(cfg) - 2.551e12) / 2.551e12 < 1e-3


def test_warmup_minimum_enforced():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "1"])
