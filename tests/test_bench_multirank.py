"""The N>1 path of bench.py on CPU: world_size-2 gloo ranks, each timing a
different replica; every rank must see the slowest time and the job
throughput must count all ranks' tokens."""
import os
import socket

import torch.multiprocessing as mp
import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
    q.put((rank, ms, bench.job_tokens_per_s(8192, world, ms)))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
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
    assert [r[1] for r in res] == [15.0, 15.0]
    assert res[0][2] == pytest.approx(2 * 8192 / 0.015)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.job_tokens_per_s(100, 1, 10.0) == pytest.approx(10000.0)


def test_clock_samples_outside_the_timed_window_are_ignored():
    """The clock record keeps only nvidia-smi samples taken inside the timed
    window (host wall clock), and falls back to the first sample after the
    window began when the window is shorter than the sampling period."""
    import datetime
    import bench

    def line(t, mhz, cap="Not Active"):
        ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, 0, {mhz}, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, {cap}\n"

    t0 = 1_800_000_000.0
    s = bench.ClockSampler(0)
    with open(s.tmp.name, "w") as f:
        f.write(line(t0 - 0.2, 345))                    # idle, before the window
        f.write(line(t0 + 0.05, 1950, cap="Active"))
        f.write(line(t0 + 0.10, 1965))
        f.write(line(t0 + 0.40, 400))                    # after the window
    s.proc = type("P", (), {"terminate": lambda self: None, "wait": lambda self, timeout=None: 0})()
    s.mark(t0, t0 + 0.2)
    c = s.stop()
    assert c["samples"] == 2 and c["sm_mhz"] == 1957.5 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]

    s = bench.ClockSampler(0)
    with open(s.tmp.name, "w") as f:
        f.write(line(t0 - 0.2, 345))
        f.write(line(t0 + 0.03, 1980))
    s.proc = type("P", (), {"terminate": lambda self: None, "wait": lambda self, timeout=None: 0})()
    s.mark(t0, t0 + 0.01)
    c = s.stop()
    assert c["samples"] == 1 and c["sm_mhz"] == 1980.0
