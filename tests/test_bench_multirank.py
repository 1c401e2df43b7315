"""Multi-rank host logic of bench.py on CPU: two gloo ranks check the max-over-ranks
reduction, the aggregate rate and that each rank's shard of the synthetic workload is
its own slice of the global batch."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    from workloads import byte_stream, qkv_bits, workload
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.rank_info() == (rank, world, rank)
        max_over = bench.make_max_over_ranks(dist, torch.device("cpu"))
        local_ms = 3.0 + rank            # rank 1 is the slower one
        slowest = max_over(local_ms)
        cfg = workload("tiny_topk", batch=2)
        seqs = bench.shard_sequences(rank, cfg["batch"])
        shard = byte_stream(cfg, seq_offset=seqs.start)
        q, _, _ = qkv_bits(cfg, seed_offset=1000 * rank)
        dist.barrier()
        np.save(os.path.join(out_dir, f"r{rank}.npy"), shard)
        np.save(os.path.join(out_dir, f"q{rank}.npy"), q[:, :4])
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{slowest} {bench.aggregate_rate(world, 10.0, slowest)} {seqs.start} {seqs.stop}")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [open(tmp_path / f"r{r}.txt").read().split() for r in range(world)]
    for r in range(world):
        slowest, rate, lo, hi = map(float, res[r])
        assert slowest == 4.0                              # max over ranks, seen by every rank
        assert rate == pytest.approx(2 * 10.0 / 4.0)       # whole-job work over the slowest time
        assert (lo, hi) == (2.0 * r, 2.0 * r + 2)          # disjoint, contiguous shards
    from workloads import byte_stream, workload
    whole = byte_stream(workload("tiny_topk", batch=4))
    shards = np.concatenate([np.load(tmp_path / f"r{r}.npy") for r in range(world)])
    assert np.array_equal(shards, whole)                   # the shards tile the global batch
    q0, q1 = (np.load(tmp_path / f"q{r}.npy") for r in range(world))
    assert not np.array_equal(q0, q1)                      # ranks draw their own Q/K/V
