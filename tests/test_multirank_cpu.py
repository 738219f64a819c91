"""Host side of the multi-rank bench path, run as two gloo ranks on the CPU.

With N ranks every rank processes its own batch (heads are independent, there
is no exchange on the data path); only the timing is combined: the whole-job
time is the maximum over ranks and the throughput counts the units of all
ranks. The ranks here stand in for GPUs: each evaluates its shard with the
oracle (the forward of its own seeded batch), which must not depend on the
other rank, and the timing helpers of bench.py combine their times over gloo.
"""
import importlib.util
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _shard_output(rank):
    import oracle
    from workloads import make_qkv, to_f64
    bench = _bench()
    q, k, v = make_qkv(1, 2, 48, 8, "f32", seed=bench.replica_seed(rank, 0))
    return oracle.recurrent(to_f64(q), to_f64(k), to_f64(v), causal=True)


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        o = _shard_output(rank)
        # A rank-dependent time: the job time is the largest.
        ms = bench.job_ms(10.0 + 5.0 * rank, dist, torch.device("cpu"))
        rate = bench.job_rate(1000, world, ms)
        np.save(os.path.join(out_dir, f"o{rank}.npy"), o)
        with open(os.path.join(out_dir, f"t{rank}.txt"), "w") as f:
            f.write(f"{ms} {rate}")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_shard_independently_and_time_by_max(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for rank in range(world):
        got = np.load(tmp_path / f"o{rank}.npy")
        # The shard equals the same batch computed alone: no cross-rank dependency.
        np.testing.assert_array_equal(got, _shard_output(rank))
        ms, rate = map(float, (tmp_path / f"t{rank}.txt").read_text().split())
        assert ms == pytest.approx(15.0)                 # max over ranks (10 and 15)
        assert rate == pytest.approx(1000 * world / 15e-3)
    # Different ranks draw different batches.
    assert not np.array_equal(np.load(tmp_path / "o0.npy"), np.load(tmp_path / "o1.npy"))


def test_single_rank_helpers_are_identity():
    bench = _bench()
    assert bench.job_ms(3.5, None, None) == 3.5
    assert bench.job_rate(10, 1, 2.0) == pytest.approx(5000.0)
    assert bench.replica_seed(0, 3) != bench.replica_seed(1, 3)
