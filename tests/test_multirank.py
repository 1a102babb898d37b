"""The N > 1 benchmark path on CPU: two gloo ranks shard rows with no data-path collective and
agree on the max time over ranks."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, wsize, local = bench.dist_env()
    assert (r, wsize, local) == (rank, world, rank)
    w = synth.WORKLOADS["fp32_64x1024"]
    row0 = bench.shard_row0(r, w.M)
    shard = synth.generate(w, row0=row0, nrows=w.M)
    np.save(os.path.join(out_dir, f"shard{rank}.npy"), shard)
    t = bench.reduce_max(1.5 + rank, wsize)  # each rank's "elapsed time"
    bench.barrier(wsize)
    with open(os.path.join(out_dir, f"max{rank}.txt"), "w") as fh:
        fh.write(repr(t))
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    maxes = [float(open(tmp_path / f"max{r}.txt").read()) for r in range(world)]
    assert maxes == [2.5, 2.5]
    shards = [np.load(tmp_path / f"shard{r}.npy") for r in range(world)]
    w = synth.WORKLOADS["fp32_64x1024"].with_rows(128)
    whole = synth.generate(w)
    assert np.array_equal(np.concatenate(shards), whole)  # disjoint shards of one seeded matrix
    assert not np.array_equal(shards[0], shards[1])
