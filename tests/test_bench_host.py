"""Host logic of bench.py's multi-GPU mode (replicas only), on CPU with the gloo backend and
two ranks: the timing barrier, the max over ranks of the step time, and that under torchrun
only rank 0 prints the JSON line (the reference arm's other ranks exit without work)."""
import io
import json
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    mx = bench.max_over_ranks(1.5 + rank, w)  # per-rank step times 1.5 ms and 2.5 ms
    # the reference arm under torchrun: rank 0 alone works and prints
    calls = []
    bench.run_reference = lambda args, rank_, world_, local_: calls.append(rank_) or {"impl": "reference", "rank": rank_}
    buf = io.StringIO()
    argv = sys.argv
    sys.argv = ["bench.py", "--impl", "reference", "--gpus", str(world), "--steps", "1", "--warmup", "3"]
    try:
        with redirect_stdout(buf):
            bench.main()
    finally:
        sys.argv = argv
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((rank, mx, calls, buf.getvalue()))


def test_two_gloo_ranks_barrier_max_and_rank0_output():
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
    (r0, mx0, calls0, out0), (r1, mx1, calls1, out1) = res
    assert mx0 == mx1 == 2.5  # whole-job time is the slowest rank's
    assert calls0 == [0] and calls1 == []
    assert json.loads(out0.strip()) == {"impl": "reference", "rank": 0}
    assert out1 == ""


