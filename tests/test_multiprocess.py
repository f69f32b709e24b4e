"""The N > 1 host logic of bench.py on CPU: two gloo ranks (world size 2,
rendezvous on 127.0.0.1) reduce their step times to the slowest rank's and
report whole-job throughput with weak scaling (each rank runs its own copy of
the workload).  On GPUs the same functions run over NCCL; here no GPU is used."""
import os
import queue
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world, init_method=f"tcp://127.0.0.1:{port}")
    try:
        w, r, _ = bench.dist_setup()
        ms = bench.max_over_ranks(times[rank], dist, "cpu")
        out.put((r, w, ms, bench.job_tflops(w, 1e12, ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    times = [12.5, 20.0]   # ms per step seen by rank 0 and rank 1
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = []
    try:
        for _ in procs:
            results.append(out.get(timeout=120))
    except queue.Empty:
        pass
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    assert sorted(r for r, *_ in results) == [0, 1]
    for _, w, ms, tflops in results:
        assert w == 2
        assert ms == 20.0                                   # the slowest rank sets the job's time
        assert abs(tflops - 2 * 1e12 / 0.020 / 1e12) < 1e-9  # both ranks' work in that time


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(7.5) == 7.5
    assert abs(bench.job_tflops(1, 492.6e12, 430.0) - 492.6 / 0.430) < 1e-6
