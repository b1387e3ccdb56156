"""The multi-rank host logic of bench.py on two gloo ranks (CPU): rank setup
from the launcher's environment, the barrier, the maximum over ranks that
times the job, the whole-job throughput, and the reference arm leaving its
work to rank 0.  Replicas share nothing on the data path, so this is all the
N > 1 path adds."""
import importlib.util
import multiprocessing as mp
import os
import socket

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, port, q):
    os.environ.update(WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    import torch.distributed as dist
    b = _bench()
    world, r, _ = b.dist_setup()
    b.barrier(world)
    slowest = b.max_over_ranks(world, 100.0 + 50.0 * r)     # rank 1 is the slower one
    skipped = b.run_reference(None, None, world, r) if r == 1 else None
    q.put((r, world, slowest, b.job_throughput(world, 64, 10, slowest), skipped))
    b.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, slowest, value, skipped) in enumerate(out):
        assert rank == r and world == 2
        assert slowest == 150.0                  # both ranks see the slowest time
        assert value == 2 * 64 * 10 / 0.150     # all ranks' tokens over that time
    assert out[1][4] == 0                        # the reference arm's rank 1 exits without work
