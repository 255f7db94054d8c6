"""Replica (data-parallel) path of the bench, world_size 2 on the gloo
backend on CPU: requests are independent, so each rank verifies its own
seeded batch and the only collectives are the timing reductions (max of the
elapsed time, min of the end-to-end rate) and the barrier around the timed
region. No collective touches the verify data."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from oracle import spec_oracle as O

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(WORLD))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        cfg = dict(kind="greedy", B=4, K=4, V=32, dtype="fp32", p_match=0.8, seed=7200)
        x = bench.make_inputs(cfg, bench.rank_seed(cfg["seed"], rank), "cpu")
        # each rank verifies its own batch with the oracle (no exchange)
        h = bench.host_copy(x)
        res = O.verify_greedy(h["target"], h["draft_tokens"])
        dist.barrier()
        elapsed = [3.0, 5.0][rank]               # rank 1 is the slow one
        e2e_rate = [200.0, 150.0][rank]
        emax = bench.reduce_over_ranks(elapsed, "max", "cpu", WORLD)
        emin = bench.reduce_over_ranks(e2e_rate, "min", "cpu", WORLD)
        dist.barrier()
        np.savez(os.path.join(result_dir, f"r{rank}.npz"), target=h["target"],
                 n=res["num_accepted"], emax=emax, emin=emin)
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    d = str(tmp_path_factory.mktemp("gloo"))
    mp.start_processes(_worker, args=(_free_port(), d), nprocs=WORLD, start_method="spawn", join=True)
    return [np.load(os.path.join(d, f"r{r}.npz")) for r in range(WORLD)]


def test_ranks_draw_distinct_requests(results):
    assert bench.rank_seed(7200, 0) != bench.rank_seed(7200, 1)
    assert not np.array_equal(results[0]["target"], results[1]["target"])


def test_every_rank_sees_the_slowest_time_and_rate(results):
    for r in results:
        assert float(r["emax"]) == 5.0
        assert float(r["emin"]) == 150.0


def test_whole_job_rate_is_from_the_slowest_rank():
    # 2 ranks x 10 steps x 160 rows in 5 ms (the max over ranks) = 640,000 rows/s
    assert bench.aggregate(5.0, 160, 10, WORLD) == pytest.approx(640000.0)
    assert bench.aggregate(5.0, 160, 10, 1) == pytest.approx(320000.0)


def test_single_rank_reduction_is_identity():
    assert bench.reduce_over_ranks(4.5, "max", "cpu", 1) == 4.5


def test_bench_describes_every_workload():
    """Host-side helpers of bench.py hold for every workload it can time (no
    GPU): launch counts, kernel description, algorithmic bytes, config."""
    import bench
    for name, cfg in bench.CONFIGS.items():
        n = bench.launches_per_call(cfg)
        assert 1 <= n <= 4, name
        assert bench.kernel_desc(cfg), name
        rows, alg = bench.algorithmic_bytes(cfg)
        assert rows > 0 and alg > 0, name
        assert bench.config_dict(cfg, name, 1)["name"] == name
    # stochastic tree workloads run on the cluster path: row pass + one kernel
    assert bench.launches_per_call(bench.CONFIGS["eagle_tree_power"]) == 2
    assert bench.launches_per_call(bench.CONFIGS["eagle_tree_greedy"]) == 2
