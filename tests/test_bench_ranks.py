"""The multi-rank logic of bench.py on two CPU ranks (gloo).

Each rank verifies its own batch (weak scaling): the timed region is closed by
the slowest rank, whole-job throughput counts every rank's rows, and only rank
0 prints.  The GPU work itself needs one GPU per rank and is not run here.
"""

import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        elapsed = [0.25, 0.75][rank]  # rank 1 is the slow one
        slowest = bench.max_over_ranks(elapsed, w, "cpu")
        rate = bench.job_rate(w, 2048, 10, slowest)
        # the reference arm: only rank 0 runs and prints
        args = bench.argparse.Namespace(steps=1, warmup=0, gpus=w, batch=4, reference_seqs=1)
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_reference(args)
        # the oracle arms of the other measured operations behave the same way
        ops = {}
        for op in ("overlap", "typical", "rerank"):
            oargs = bench.argparse.Namespace(steps=1, warmup=0, gpus=w, batch=2, op=op,
                                             impl="reference")
            obuf = io.StringIO()
            with redirect_stdout(obuf):
                if op == "rerank":
                    bench.run_rerank(oargs)
                else:
                    bench.run_rowop_reference(oargs)
            ops[op] = obuf.getvalue()
        out.put((rank, w, r, local, slowest, rate, buf.getvalue(), ops))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_rows():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, w, r, local, slowest, rate, printed, _ in res:
        assert (w, r, local) == (2, rank, rank)
        assert slowest == 0.75
        assert rate == 2 * 2048 * 10 / 0.75
    assert res[1][6] == ""  # rank 1 prints nothing
    line = json.loads(res[0][6].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["scaling"] == "weak"
    assert line["cpu_baseline"]["kind"] == "oracle"
    for op in ("overlap", "typical", "rerank"):
        assert res[1][7][op] == ""
        line = json.loads(res[0][7][op].strip().splitlines()[-1])
        assert line["impl"] == "reference" and line["value"] > 0
        assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_one_rank_is_its_own_maximum():
    assert bench.max_over_ranks(1.5, 1, "cpu") == 1.5
    assert bench.job_rate(1, 2048, 2, 0.5) == 8192
