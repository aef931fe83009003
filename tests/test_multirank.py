"""The N > 1 path on the CPU with gloo, world size 2.

Images are independent (every route of every image starts from the same
memories0), so the batch shards across ranks with no exchange on the data
path: two ranks each computing their own images give exactly the single
process result.  The benchmark's cross-rank reduction takes the slowest
rank's time and counts every rank's tokens."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    from visual_backbone_gb300 import synth
    wl = synth.Workload("mr", 4, 5, 6, 2, 8, 0, "f32", seed=31, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    mine = list(range(rank, wl.B, world))          # this rank's images
    out = oracle.forward(inp.x64[mine], inp.mem0, wl.H, wl.W, wl.nh, wl.d,
                         params=oracle.OracleParams(alpha_init=wl.alpha_init))
    np.save(os.path.join(outdir, f"out{rank}.npy"), out)
    # timing reduction: each rank reports a different time; all must see the max
    t = bench.max_over_ranks([1.0 + rank, 5.0 - rank])
    np.save(os.path.join(outdir, f"t{rank}.npy"), np.array(t))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_shard_images_without_exchange(tmp_path, orc):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    from visual_backbone_gb300 import synth
    wl = synth.Workload("mr", 4, 5, 6, 2, 8, 0, "f32", seed=31, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    full = orc.forward(inp.x64, inp.mem0, wl.H, wl.W, wl.nh, wl.d,
                       params=orc.OracleParams(alpha_init=wl.alpha_init))
    for rank in range(world):
        part = np.load(tmp_path / f"out{rank}.npy")
        np.testing.assert_array_equal(part, full[rank::world])
        assert np.load(tmp_path / f"t{rank}.npy").tolist() == [2.0, 5.0]


def test_job_throughput_counts_all_ranks():
    import bench
    assert bench.job_throughput(100, 10, 4, 2.0) == pytest.approx(2000.0)
