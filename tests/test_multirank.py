"""The N > 1 path on the CPU with gloo, world size 2.

Images are independent (every route of every image starts from the same memories0), so
the job's batch shards across ranks with no exchange on the data path.  Each rank takes
its images with the library's own mapping (``vh.shard_images``, the one ``bench.py``
uses) and draws exactly those images (``synth.make_inputs(first_image=...)``).  The
ranks here scan their shards with the oracle (there is no GPU on this host); the test
checks that the shards cover the job's batch with every image exactly once, that each
rank's inputs are the job's images, and that the gathered outputs equal the single
process result.  The benchmark's cross-rank reduction takes the slowest rank's time and
counts every rank's tokens."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

WL_ARGS = ("mr", 5, 5, 6, 2, 8, 0, "f32")
WL_KW = dict(seed=31, alpha_init=0.999)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _check_cover(shards, global_batch):
    """Every image of the batch in exactly one shard, in order within each shard."""
    seen = [i for sh in shards for i in sh]
    assert sorted(seen) == list(range(global_batch)), f"images dropped or duplicated: {shards}"
    for sh in shards:
        assert list(sh) == sorted(sh)


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
    import visual_backbone_gb300 as vh
    from visual_backbone_gb300 import synth
    wl = synth.Workload(*WL_ARGS, **WL_KW)
    mine = vh.shard_images(wl.B, world, rank)       # this rank's images of the job
    inp = synth.make_inputs(wl, batch=len(mine), first_image=mine.start)
    out = oracle.forward(inp.x64, inp.mem0, wl.H, wl.W, wl.nh, wl.d,
                         params=oracle.OracleParams(alpha_init=wl.alpha_init))
    np.save(os.path.join(outdir, f"idx{rank}.npy"), np.array(list(mine)))
    np.save(os.path.join(outdir, f"x{rank}.npy"), inp.x_store)
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
    wl = synth.Workload(*WL_ARGS, **WL_KW)
    inp = synth.make_inputs(wl)
    full = orc.forward(inp.x64, inp.mem0, wl.H, wl.W, wl.nh, wl.d,
                       params=orc.OracleParams(alpha_init=wl.alpha_init))
    shards = [np.load(tmp_path / f"idx{r}.npy").tolist() for r in range(world)]
    _check_cover(shards, wl.B)
    for rank in range(world):
        idx = shards[rank]
        np.testing.assert_array_equal(np.load(tmp_path / f"x{rank}.npy"), inp.x_store[idx])
        np.testing.assert_array_equal(np.load(tmp_path / f"out{rank}.npy"), full[idx])
        assert np.load(tmp_path / f"t{rank}.npy").tolist() == [2.0, 5.0]


@pytest.mark.parametrize("global_batch", [0, 1, 5, 32, 33, 256])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_shard_images_cover_once(global_batch, world):
    import visual_backbone_gb300 as vh
    shards = [vh.shard_images(global_batch, world, r) for r in range(world)]
    _check_cover(shards, global_batch)
    sizes = [len(s) for s in shards]
    assert max(sizes) - min(sizes) <= 1


def test_cover_check_catches_bad_shards():
    """The coverage check the gloo test relies on fails for a dropped or a duplicated image."""
    with pytest.raises(AssertionError):
        _check_cover([range(0, 2), range(3, 5)], 5)       # image 2 dropped
    with pytest.raises(AssertionError):
        _check_cover([range(0, 3), range(2, 5)], 5)       # image 2 twice


def test_shard_images_rejects_bad_ranks():
    import visual_backbone_gb300 as vh
    for args in ((4, 0, 0), (4, 2, 2), (4, 2, -1), (-1, 2, 0)):
        with pytest.raises(ValueError):
            vh.shard_images(*args)


def test_job_throughput_counts_all_ranks():
    import bench
    assert bench.job_throughput(100, 10, 4, 2.0) == pytest.approx(2000.0)
