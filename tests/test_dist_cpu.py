"""The multi-rank pieces of bench.py on CPU with the gloo backend (world size 2): the
max-over-ranks timing reduction and the sharding of independent units. The path itself
needs no collective (state tiles are independent), so these are the only cross-rank
operations."""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(1.5 + rank, world)
        lo, hi = bench.shard_units(4096, world, rank)
        bench.barrier(world)
        q.put((rank, m, lo, hi))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_sharding_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]
    assert res[0][2:] == (0, 2048) and res[1][2:] == (2048, 4096)


@pytest.mark.parametrize("total,world", [(10, 3), (4096, 8), (1, 2)])
def test_shard_units_cover_exactly(total, world):
    sys.path.insert(0, ROOT)
    import bench
    seen = []
    for r in range(world):
        lo, hi = bench.shard_units(total, world, r)
        seen.extend(range(lo, hi))
    assert seen == list(range(total))


def _shard_worker(rank, world, port, q):
    """One rank of the bench's multi-rank split: heads shard_units(H, world, rank) of every
    slot, its own pool of those heads, the call run on them (here by the fp64 oracle), no
    collective on the data path; only the timing reduction crosses ranks."""
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    from linear_attention_state_recurrent_gb300 import workloads as wl
    from oracle import kda_oracle as ko
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = wl.decode_case(6, 5, 32, 32, seed=41, lower_bound=-5.0, index_stride=3, num_slots=16,
                           pool_std=0.1, name="tp_decode")
        lo, hi = bench.shard_units(w.H, world, rank)
        ref = ko.run(wl.shard_heads(w, lo, hi))
        bench.max_over_ranks(float(rank), world)
        q.put((rank, lo, hi, ref.out, ref.final_states, ref.err_flags))
    finally:
        dist.destroy_process_group()


def test_head_sharded_ranks_reassemble_the_call_gloo():
    sys.path.insert(0, ROOT)
    import numpy as np
    from linear_attention_state_recurrent_gb300 import workloads as wl
    from oracle import kda_oracle as ko
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 30500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in range(2)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = wl.decode_case(6, 5, 32, 32, seed=41, lower_bound=-5.0, index_stride=3, num_slots=16,
                       pool_std=0.1, name="tp_decode")
    full = ko.run(w)
    assert [(r[1], r[2]) for r in res] == [(0, 3), (3, 5)]
    out = np.concatenate([r[3] for r in res], axis=1)
    states = np.concatenate([r[4] for r in res], axis=1)
    assert np.array_equal(out, full.out)
    assert np.array_equal(states, full.final_states)
    assert all(r[5] == full.err_flags for r in res)
