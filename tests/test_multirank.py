"""The N > 1 path of bench.py on CPU: two gloo ranks run independent replicas
and the whole-job figures take the slowest rank's time and the sum of the
work (weak scaling; no collective touches the data path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    agg = bench.aggregate_ranks([2.0, 3.0][rank], kv_bytes=1_000_000, requests=8)
    q.put((rank, agg, bench.dist_info()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, agg, info in out:
        assert info == (rank, 2, 0)
        assert agg["ms_per_step"] == 3.0                      # slowest rank
        assert agg["value_gbs"] == pytest.approx(2_000_000 / 3e-3 / 1e9)
        assert agg["tokens_per_s"] == pytest.approx(16 / 3e-3)


def test_single_process_aggregation_is_identity():
    import bench
    agg = bench.aggregate_ranks(4.0, kv_bytes=4_000_000, requests=8)
    assert agg["ms_per_step"] == 4.0 and agg["value_gbs"] == pytest.approx(1.0)
