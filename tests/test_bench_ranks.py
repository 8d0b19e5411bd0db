"""The multi-replica path of bench.py on CPU: two gloo ranks agree on the
slowest replica's step time and on the whole-job throughput."""
import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    step_ms = 0.30 + 0.05 * rank             # rank 1 is the slow replica
    mx = bench.max_over_ranks(step_ms)
    out[rank] = (mx, bench.job_rows_per_s(8, world, mx))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]
    mx, value = res[0]
    assert abs(mx - 0.35) < 1e-12
    assert abs(value - 2 * 8 / 0.35e-3) < 1e-6


def test_single_process_passthrough():
    import bench
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.job_rows_per_s(8, 1, 0.25) == 32000.0
