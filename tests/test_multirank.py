"""Host logic of running the benchmark on several GPUs as independent
replicas: rank setup, the barrier around the timed region, the max of the
ranks' times and the whole-job figures — world size 2 on the gloo backend,
CPU only (no data-path collective exists to test: the replicas share nothing).
"""
import math
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch.distributed as tdist
    got_ws, got_rank, local = bench.dist_setup()
    try:
        assert (got_ws, got_rank, local) == (ws, rank, rank)
        assert tdist.get_backend() == "gloo"
        bench.barrier(got_ws)
        m = bench.max_over_ranks(times[rank], got_ws)
        bench.barrier(got_ws)
        out.put((rank, m))
    finally:
        tdist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ws, port = 2, _free_port()
    times = [12.5, 17.25]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, times, out)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(out.get(timeout=10) for _ in range(ws))
    assert res == {0: 17.25, 1: 17.25}


def test_single_rank_needs_no_process_group():
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_setup() == (1, 0, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_job_figures_weak_scaling():
    # each replica: 100 steps of 24 layers in 410 ms, 870.75 MB selected per layer
    sel, pred = 870_752_256, 123_072_000
    one = bench.job_figures(410.0, 100, 24, 1, sel, pred)
    two = bench.job_figures(410.0, 100, 24, 2, sel, pred)
    assert one["us_layer_replica"] == pytest.approx(410.0e3 / 100 / 24)
    assert one["us_layer_job"] == pytest.approx(one["us_layer_replica"])
    # twice the layers in the same time: half the job time per layer, twice the bytes/s
    assert two["us_layer_job"] == pytest.approx(one["us_layer_job"] / 2)
    assert two["gbs_selected"] == pytest.approx(2 * one["gbs_selected"])
    assert two["layers_per_s"] == pytest.approx(2 * one["layers_per_s"])
    assert one["gbs_selected"] == pytest.approx(sel / (410.0e-3 / 2400) / 1e9)
    assert one["gbs_all"] == pytest.approx((sel + pred) / (410.0e-3 / 2400) / 1e9)


def test_measured_crossing_of_the_gate_sweep():
    # bench.py's App. E interpolation of two modes' sweep times
    ctx = [2048, 4096, 8192, 16384]
    assert bench._measured_crossing(ctx, [10, 12, 16, 24], [13, 13.5, 14, 14.5]) == 4096 + 1.5 / 3.5 * 4096
    # b leads first, a takes over between 4096 and 8192 (differences 6 -> -0.5)
    assert math.isclose(bench._measured_crossing(ctx, [20, 18, 16, 14], [10, 12, 16.5, 20]),
                        4096 + 6 / 6.5 * 4096)
    assert bench._measured_crossing(ctx, [1, 1, 1, 1], [2, 2, 2, 2]) is None
