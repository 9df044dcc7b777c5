"""bench.py's multi-rank path on the CPU: two gloo ranks run independent replicas;
the timed region is bracketed by barriers and the reported time is the slowest
rank's (max over ranks).  No collective touches the data path.  A rank that fails
between steps is detected on the host: the surviving rank's next barrier raises
instead of waiting forever."""

import os
import socket
import time

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world)
    # rank 1 is the slow replica: 4 steps of 50 ms against 4 of 10 ms
    delay = 0.05 if rank == 1 else 0.01
    t = {}

    def start():
        t["t0"] = time.perf_counter()

    def stop():
        return time.perf_counter() - t["t0"]

    secs = bench.timed_steps(lambda: time.sleep(delay), 4, world, None, None, (start, stop))
    own = bench.max_over_ranks(delay * 4, 1)   # world 1: identity
    q.put((rank, secs, own))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(world))
    secs = [s for _, s, _ in res]
    assert secs[0] == pytest.approx(secs[1])          # both ranks report the same (max) time
    assert secs[0] >= 0.2                             # the slow rank's 4 x 50 ms
    assert res[0][2] == pytest.approx(0.04)


def test_clock_rows_parse():
    import bench
    rows = [["2026/12/03 07:30:11.100", "0", "1965 MHz", "2070 MHz", "1200.5 W", "0x0", "Not Active",
             "Not Active", "Not Active", "Active"],
            ["2026/12/03 07:30:11.120", "0", "1980 MHz", "2070 MHz", "1250.0 W", "0x0", "Not Active",
             "Not Active", "Not Active", "Not Active"],
            ["2026/12/03 07:30:11.140", "0", "345 MHz", "2070 MHz", "150.0 W", "0x0", "Not Active",
             "Not Active", "Not Active", "Not Active"]]
    c = bench.parse_clock_rows(rows)
    assert c["sm_mhz"] == pytest.approx(1972.5)       # idle sample left out
    assert c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]
    assert c["samples"] == 3 and c["window"] == "whole sampling"
    # only the samples stamped inside the timed region (plus the sampling period) count
    t = bench._stamp("2026/12/03 07:30:11.115")
    c = bench.parse_clock_rows(rows, t, t + 0.02, 0.0)
    assert c["samples"] == 1 and c["sm_mhz"] == 1980 and c["reasons"] == []
    assert c["window"] == "timed region"
    # no stamp inside the region: every row counts
    c = bench.parse_clock_rows(rows, t + 100.0, t + 101.0, 0.02)
    assert c["samples"] == 3 and c["window"] == "whole sampling"


def test_kernel_flops_sum_to_the_block_minus_rank_work():
    import bench
    import synth
    cfg = synth.MLP_CONFIGS["llama7b"]
    f = bench.kernel_flops(cfg)
    base = 12.0 * cfg.M * cfg.h * cfg.i
    assert sum(f.values()) > base
    assert sum(f.values()) < cfg.flops()


def _failing_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    bench.dist_init("gloo", timeout_s=10.0)
    bench.barrier(world)                       # both ranks joined
    if rank == 1:
        os._exit(3)                            # dies between steps, nothing in flight
    t0 = time.perf_counter()
    try:
        bench.timed_steps(lambda: time.sleep(0.01), 4, world, None, None,
                          (lambda: None, lambda: 0.0))
        q.put((rank, "no error", time.perf_counter() - t0))
    except Exception as e:                     # noqa: BLE001 - any error is the detection
        q.put((rank, type(e).__name__, time.perf_counter() - t0))


def test_a_dead_rank_is_detected_not_waited_for():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_failing_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert procs[1].exitcode == 3
    assert procs[0].exitcode is not None, "the surviving rank is still waiting"
    rank, what, secs = q.get()
    assert rank == 0 and what != "no error"
    assert secs < 60.0
