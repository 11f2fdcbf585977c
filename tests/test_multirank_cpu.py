"""N > 1 bench path on the CPU with gloo, world size 2.

The decode work shards by sequence with no collective on the data path: each
rank decodes its own batch (weak scaling) and only the timing is reduced
(max over ranks) and the work summed.  This runs those pieces as two real
processes.
"""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads
        import oracle
        m = bench.max_over_ranks(float(10 * (rank + 1)), world)
        s = bench.sum_over_ranks(float(rank + 1), world)
        # each rank owns a different seeded batch of the same shape
        b = workloads.make_batch("tiny", seed=1000 * rank)
        v = workloads.host_values(b, seed=1000 * rank, nan_tails=False)
        ref = oracle.paged_decode_attention(v["q"], v["k_cache"], v["v_cache"], b.block_tables, b.seq_lens,
                                            b.scale, b.block_size)
        # contiguous split of a global batch (strong-scaling helper) covers every sequence once
        lo, hi = workloads.shard_sequences(10, rank, world)
        t = torch.tensor([hi - lo], dtype=torch.int64)
        dist.all_reduce(t)
        out_q.put((rank, m, s, b.seq_lens.tolist(), float(np.abs(ref).sum()), int(t.item())))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_weak_scaling_path():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, m0, s0, lens0, a0, n0), (r1, m1, s1, lens1, a1, n1) = res
    assert m0 == m1 == 20.0            # max over ranks
    assert s0 == s1 == 3.0             # sum over ranks
    assert len(lens0) == len(lens1) and lens0 != lens1   # same shape, independent batches
    assert a0 != a1
    assert n0 == n1 == 10
