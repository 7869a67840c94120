"""bench.py's multi-GPU path on CPU: N independent replicas (one process per
GPU, no collective on the data path), a barrier around the timed region, the
job time = the slowest rank's, and the whole-job value = all ranks' work over
that time.  Two gloo ranks stand in for two GPUs."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys

    import torch.distributed as dist

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    # rank r "took" 100 + 50 r ms for 1e12 units of work
    value, total_ms = bench.replica_value(1.0e12, 100.0 + 50.0 * rank, world)
    bench.barrier(world)
    out[rank] = (value, total_ms)
    dist.destroy_process_group()


def test_two_replicas_on_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        value, total_ms = res[r]
        assert total_ms == pytest.approx(150.0)  # the slowest rank
        assert value == pytest.approx(2 * 1.0e12 / 0.150)  # both ranks' work over that time


def test_single_replica_needs_no_process_group():
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    value, total_ms = bench.replica_value(3.0e12, 200.0, 1)
    assert total_ms == 200.0 and value == pytest.approx(1.5e13)


def test_bench_entry_points_resolve():
    """Every mode bench.py's command line dispatches to exists (the profiling
    recipes under profiles/ call ``--case``)."""
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    for name in ("run_case", "run_reference", "run_ours", "main"):
        assert callable(getattr(bench, name, None)), name


def test_chunk_flop_convention_adds_up_to_the_full_prefill():
    """Chunks of one context count exactly the full prefill's work."""
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    full = bench.prefill_flops(1, 32, 128, 131072)
    assert bench.chunk_prefill_flops(1, 32, 128, 131072, 0) == full
    parts = [(0, 50000), (50000, 8192), (58192, 131072 - 58192)]
    assert sum(bench.chunk_prefill_flops(1, 32, 128, s_new, n_past) for n_past, s_new in parts) == full
