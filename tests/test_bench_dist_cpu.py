"""Host-side multi-rank logic of bench.py on CPU (gloo, world size 2).

One rank per GPU, each on its own batch (no collective on the data path);
the only collectives are the barrier around the timed region and the max of
the per-rank times.  Here two CPU processes exercise exactly those pieces.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    w, r, lr = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    # the slowest rank sets the job time
    got = bench.max_over_ranks(10.0 + rank, w, torch.device("cpu"))
    # the reference arm runs on rank 0 only; other ranks return at once
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    other = None
    if rank == 1:
        other = bench.run_reference(args)
    bench.barrier(w)
    torch.distributed.destroy_process_group()
    queue.put((rank, w, r, got, other))


def test_two_rank_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in results] == [0, 1]
    for rank, world, r, got, other in results:
        assert world == 2 and r == rank
        assert got == 11.0
        assert other is None


def test_byte_counts_of_the_step():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    h, t = 8192, 8
    assert bench.fwd_bytes_per_token(t, h, 1) == 23 * h + 8 == 188_424
    assert bench.bwd_bytes_per_token(h, 1) == 9 * h + 8 == 73_736
    assert (bench.fwd_bytes_per_token(t, h, 1) + bench.bwd_bytes_per_token(h, 1)) * 16384 \
        == 4_295_229_440
    assert bench.fwd_bytes_per_token(t, h, t) == 2 * t * h + 5 * h + 2 * h * t + 8
    assert bench.bwd_bytes_per_token(h, 1, "rmsnorm") == 9 * h + 4


def test_clock_rejection_rules():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.clocks_rejected({"reasons": ["hw_slowdown"], "sm_mhz": 2000, "sm_max_mhz": 2070})
    assert bench.clocks_rejected({"reasons": [], "sm_mhz": 900, "sm_max_mhz": 2070})
    assert not bench.clocks_rejected({"reasons": ["sw_power_cap"], "sm_mhz": 1500,
                                      "sm_max_mhz": 2070})
    assert not bench.clocks_rejected({"reasons": [], "sm_mhz": 2070, "sm_max_mhz": 2070})


def test_backward_through_g_byte_counts():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    h, t = 8192, 8
    assert bench.bwd_g_bytes_per_token(t, h, 1, fused=True) == 23 * h + 8
    assert bench.bwd_g_bytes_per_token(t, h, 1, fused=False) == 27 * h + 8
    # reduce-scatter 18h, shard norm 9h + 8, all-gather 4h
    assert bench.unfused_fwd_bytes_per_token(t, h, 1) == 31 * h + 8


def test_recorded_traffic_only_on_the_profiled_workload():
    """roofline.traffic comes from the ncu summary of the default line; any
    other workload, size or norm reports null."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args([])
    assert bench.profiled_workload(args)
    for extra in (["--h", "5120"], ["--s", "4096"], ["--norm", "rmsnorm"], ["--p", "0"],
                  ["--n-gather", "8"], ["--workload", "ragged"], ["--workload", "trace4k"]):
        assert not bench.profiled_workload(bench.parse_args(extra)), extra
    assert bench.profiled_workload(bench.parse_args(["--norm", "layernorm"]))
