"""The multi-rank bench path on the CPU: two `gloo` ranks on 127.0.0.1.

bench.py runs one independent replica per GPU (the method needs no exchange
on one device); what is shared between ranks is the timing protocol: a
barrier around the timed region, the slowest rank's time taken with a MAX
all-reduce, the whole-job rate = units of all ranks / that time, and only
rank 0 printing (the reference arm's other ranks exit without work).
"""

import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local, dist = bench._dist_setup(world, backend="gloo")
    local_ms = 10.0 + 5.0 * r                    # rank 1 is the slower one
    dist.barrier()
    slowest = bench._max_over_ranks(local_ms, dist, "cpu")
    rate = bench._job_rate(w, 1e12, 3, slowest)
    # the reference arm: ranks other than 0 return at once without work
    ref_rc = None
    if r != 0:
        from sequence_exact_attention_gb300.workloads import WORKLOADS
        args = type("A", (), dict(gpus=world, steps=1, warmup=0, ref_rows=4))()
        ref_rc = bench.run_reference(args, WORKLOADS["fp32_s256"])
    dist.barrier()
    dist.destroy_process_group()
    out.put((r, w, local, slowest, rate, ref_rc))


def test_two_gloo_ranks_share_the_timing_protocol():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1]
    for rank, world, local, slowest, rate, ref_rc in res:
        assert world == 2 and local == rank
        assert slowest == 15.0                       # MAX over ranks
        assert rate == pytest.approx(2 * 1e12 * 3 / 0.015)
    assert res[1][5] == 0                            # rank 1 of the reference arm: no work


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench._dist_setup(1) == (1, 0, 0, None)
    assert bench._max_over_ranks(7.5, None, "cpu") == 7.5
    assert bench._job_rate(1, 100.0, 4, 2.0) == pytest.approx(200000.0)
