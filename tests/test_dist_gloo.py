"""The benchmark's multi-rank host logic on CPU ranks (gloo, world size 2):
each rank gets its own batch of the same shape, and the reported time is the
slowest rank's.  The data path has no collective, so this is the whole of the
multi-GPU logic."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from block_sparse_paged_score_gb300 import workloads as W
    spec = bench.rank_workload_spec(2, rank)
    w = W.Workload(spec)
    slowest = bench.max_over_ranks(10.0 + rank)
    q.put((rank, spec["seed"], int(w.decode_lens.sum()), w.num_decode, w.max_pages, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_batches_and_take_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, n0, d0, m0, t0), (r1, s1, n1, d1, m1, t1) = out
    assert s0 != s1 and n0 != n1          # different batches ...
    assert d0 == d1 == 32                  # ... of the same shape
    assert t0 == t1 == 11.0                # both report the slowest rank
