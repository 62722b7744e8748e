"""Two-rank host logic of the benchmark on CPU (gloo, world size 2): rank
discovery from the launcher's environment, the barrier, the max-over-ranks
step time, the weak-scaling aggregate, independent pairs per rank, and a
reference arm that runs on rank 0 only."""
import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import sys
    import torch
    sys.path.insert(0, ROOT)
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    from voxel_grid_sampler_gb300 import synth
    torch.distributed.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        w, r, loc = bench._dist()
        bench._barrier(w)
        step_ms = bench._max_over_ranks(2.0 + rank, w, "cpu")  # the slowest rank's time
        value = bench._aggregate_gvox(1000, w, step_ms)
        pair = synth.make_pair(1, device="cpu", shape=(8, 9, 10), seed=1000 + 1 + 100 * r)
        checksum = float(pair.F.double().sum() + pair.u.double().sum())

        class Args:
            workload, steps, warmup, ref_step_s = 4, 1, 0, 1.0

        ref_returned = None
        if r != 0:  # must return at once, without work or output
            bench.run_reference(Args(), w, r, loc)
            ref_returned = True
        q.put((rank, w, r, loc, step_ms, value, checksum, ref_returned))
    finally:
        torch.distributed.destroy_process_group()


def test_two_ranks_on_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(2):
        item = q.get(timeout=240)
        out[item[0]] = item
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        rank, w, rr, loc, step_ms, value, checksum, ref_returned = out[r]
        assert (w, rr, loc) == (2, r, r)
        assert step_ms == 3.0  # max over ranks
        assert value == pytest.approx(1000 * 2 / 3e-3 / 1e9)
    assert out[0][6] != out[1][6]  # each rank evaluates its own pair
    assert out[1][7] is True
