"""Host logic of bench.py (no GPU): the work model against the oracle's
definition on small cases, and the multi-rank timing reduction (max over
ranks, whole-job throughput) with two gloo ranks on CPU."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
import oracle as ora
import workloads


def test_landed_pairs_matches_brute_force():
    rng = np.random.default_rng(0)
    for _ in range(300):
        L, k, s, d = (int(rng.integers(1, 20)), int(rng.integers(1, 6)), int(rng.integers(1, 4)),
                      int(rng.integers(1, 4)))
        p = int(rng.integers(0, 4))
        op = int(rng.integers(0, max(s, d)))
        Lo = ora.out_len(L, k, s, p, op, d)
        if Lo < 1:
            continue
        brute = sum(1 for i in range(L) for kk in range(k) if 0 <= i * s - p + kk * d < Lo)
        assert bench.landed_pairs(L, k, s, p, op, d) == brute


def test_work_model_flops_equal_oracle_tap_count():
    """FLOPs of the work model = 2 x the multiply-adds the oracle performs:
    with all-ones inputs the oracle's output sums to exactly that count / 2."""
    for name in ("convT1d_tiny",):
        cfg = workloads.CONFIGS[name]
        x = np.ones((cfg["N"], cfg["C_in"]) + tuple(cfg["L_in"]))
        w = np.ones((cfg["C_in"], cfg["C_out"] // cfg["groups"]) + tuple(cfg["k"]))
        y = ora.conv_transpose(x, w, None, cfg["stride"], cfg["padding"], cfg["output_padding"],
                               cfg["dilation"], cfg["groups"])
        assert 2 * int(y.sum()) == bench.work_model(cfg)["flops"]
    cfg = dict(workloads.CONFIGS["convT3d_grouped"])
    cfg["L_in"] = (3, 4, 5)
    cfg["N"] = 1
    x = np.ones((1, cfg["C_in"]) + tuple(cfg["L_in"]))
    w = np.ones((cfg["C_in"], cfg["C_out"] // cfg["groups"]) + tuple(cfg["k"]))
    y = ora.conv_transpose(x, w, None, cfg["stride"], cfg["padding"], cfg["output_padding"],
                           cfg["dilation"], cfg["groups"])
    assert 2 * int(y.sum()) == bench.work_model(cfg)["flops"]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank "measured" a different time; the job time is the slowest
        t = 0.5 + rank
        bench.barrier(world)
        tmax = bench.reduce_max(t, world)
        units_per_rank = 100.0
        out[rank] = (tmax, bench.aggregate(units_per_rank * world, tmax))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert set(out.keys()) == {0, 1}
    for r in range(world):
        tmax, thr = out[r]
        assert tmax == pytest.approx(1.5)
        assert thr == pytest.approx(200.0 / 1.5)


def test_single_rank_is_identity():
    assert bench.reduce_max(3.0, 1) == 3.0
    assert bench.aggregate(10.0, 2.0) == 5.0
