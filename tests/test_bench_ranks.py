"""The multi-process parts of bench.py on CPU (gloo, world size 2): time is the max
over ranks, and only rank 0 of the reference arm does work and prints."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q.put((rank, bench.max_over_ranks(1.5 + rank, "cpu")))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get() for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, "cpu") == 3.25


def test_reference_arm_non_zero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def _shard_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import sift_synth
    import top_ratio_test_gb300 as serac
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sizes = [tuple(int(v) for v in x) for x in sift_synth.ragged_sizes(0)]
    mine = serac.shard_pairs(sizes, world)[rank]
    # every rank computes the same partition; gather what each rank takes
    got = [None] * world
    dist.all_gather_object(got, mine)
    load = torch.tensor([float(sum(sizes[k][0] * sizes[k][1] for k in mine))])
    loads = [torch.zeros(1) for _ in range(world)]
    dist.all_gather(loads, load)
    q.put((rank, got, [float(x) for x in loads]))
    dist.barrier()
    dist.destroy_process_group()


def test_shard_pairs_gloo():
    """The 256-pair ragged batch split over two gloo ranks: the ranks agree on the
    partition, every pair goes to exactly one rank, and the costs are balanced."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict((r, (g, l)) for r, g, l in (q.get() for _ in range(2)))
    assert res[0][0] == res[1][0]
    shards = res[0][0]
    assert sorted(shards[0] + shards[1]) == list(range(256))
    loads = res[0][1]
    assert max(loads) / (sum(loads) / 2) < 1.01


def test_shard_pairs_edge_cases():
    sys.path.insert(0, ROOT)
    import top_ratio_test_gb300 as serac
    assert serac.shard_pairs([], 3) == [[], [], []]
    assert serac.shard_pairs([(5, 5)], 1) == [[0]]
    assert serac.shard_pairs([(10, 10), (1, 1), (10, 10)], 2) == [[0, 1], [2]]


class _FakeOut:
    """Stands in for a MatchOutput on CPU: result() gives the pair's match list."""

    def __init__(self, k):
        import torch
        self.m = torch.tensor([[k, 1000 + k], [k + 1, 2000 + k]], dtype=torch.int32)[: 1 + k % 2]

    def result(self):
        return self.m


def _gather_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import sift_synth
    import top_ratio_test_gb300 as serac
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sizes = [tuple(int(v) for v in x) for x in sift_synth.ragged_sizes(0)]
    mine = serac.shard_pairs(sizes, world)[rank]
    outs = [_FakeOut(k) for k in mine]
    got = serac.gather_matches(mine, outs, len(sizes))
    q.put((rank, None if got is None else [m.tolist() for m in got]))
    dist.barrier()
    dist.destroy_process_group()


def test_gather_matches_gloo():
    """The host-side collection of a sharded batch over two gloo ranks: rank 0 gets
    every pair's match list, in pair order, each from the rank that matched it."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert res[1] is None
    assert res[0] == [_FakeOut(k).m.tolist() for k in range(256)]
