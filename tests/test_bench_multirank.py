"""bench.py's multi-rank plumbing on the CPU: two gloo ranks (the launch the
bench gets under torchrun for N > 1), rendezvous on 127.0.0.1.

Checks the pieces the N-GPU run relies on: the rank setup, the barrier, the
max over ranks of a time, and that only rank 0 of the reference arm works
and prints its one JSON line (the other ranks exit without work)."""
import contextlib
import io
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    import torch.distributed as dist

    r, ws, local = bench.dist_setup()
    res = {"rank": r, "ws": ws, "local": local}
    bench.barrier(ws)
    res["max"] = bench.max_over_ranks(10.0 + r, ws, "cpu")
    bench.barrier(ws)
    # the reference arm on a tiny pattern: rank 0 alone runs and prints
    wl = workloads.custom("tiny", "bf16", 1, 1, 256, 64, 16, (1,), False, (0,), None, seed=1)

    class Args:
        steps, warmup = 1, 0

    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(Args, wl)
    res["printed"] = buf.getvalue()
    with open(os.path.join(outdir, "rank%d.json" % r), "w") as f:
        json.dump(res, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(2)]
    assert [x["rank"] for x in res] == [0, 1]
    assert all(x["ws"] == 2 for x in res)
    assert all(x["max"] == 11.0 for x in res)  # the max of 10 + rank over both ranks
    assert res[1]["printed"] == ""               # rank 1: no work, no output
    lines = [ln for ln in res[0]["printed"].splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
