"""The multi-rank path of the benchmark on CPU ranks (gloo, world size 2).

Each rank scores its own layer (weak scaling, no data-path collective); the
only collectives are the timing barrier and the max-reduction of the step
time, and the job's throughput counts every rank's units.  These tests run
the same helpers bench.py uses, on two gloo processes, with the oracle
standing in for the GPU path (no GPU needed)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from kv_cache_eviction_dropkv_gb300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_env()
        assert (r, w) == (rank, world)
        # each rank's own layer, as bench.py seeds it
        spec = synth.WORKLOADS["tiny_d16_n128"]
        wl = synth.make_workload(spec.name, seed=bench.rank_seed(spec, rank))
        import oracle
        ref = oracle.run_path(wl.q, wl.k, wl.v, wl.lengths, wl.evict_k, spec.pool_kernel, spec.protect, nthreads=1)
        np.save(os.path.join(out_dir, "final_%d.npy" % rank), ref["final"])
        # the slowest rank sets the step time; throughput counts all ranks
        local_ms = 1.0 + rank                      # rank 1 is the slow one
        dist.barrier()
        step_ms = bench.reduce_max(local_ms, world)
        units = int(wl.lengths.sum())
        value = bench.job_throughput(units, world, step_ms)
        with open(os.path.join(out_dir, "agg_%d.txt" % rank), "w") as f:
            f.write("%r %r %d" % (step_ms, value, units))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    aggs = [open(tmp_path / ("agg_%d.txt" % r)).read().split() for r in range(world)]
    for step_ms, value, units in aggs:
        assert float(step_ms) == 2.0                              # max over ranks
        assert float(value) == pytest.approx(int(units) * world / 2e-3)
    assert aggs[0] == aggs[1]                                    # every rank agrees
    f0, f1 = (np.load(tmp_path / ("final_%d.npy" % r)) for r in range(world))
    assert not np.allclose(f0, f1, equal_nan=True)               # independent layers per rank


def test_single_rank_helpers_need_no_process_group():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.job_throughput(1000, 1, 2.0) == pytest.approx(5e5)
    spec = synth.WORKLOADS["llama8b_gqa_d128_n128k"]
    assert [bench.rank_seed(spec, r) for r in range(3)] == [spec.seed, spec.seed + 1, spec.seed + 2]
