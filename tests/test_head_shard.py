"""The head partition for several GPUs, on CPU: two gloo ranks each run the
oracle on their share of the heads, and the gathered result equals the
single-process oracle result; the shards cover every head exactly once."""
import os
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("H,world", [(16, 2), (16, 8), (5, 2), (3, 4), (1, 1)])
def test_shards_cover_every_head_once(H, world):
    sys.path.insert(0, ROOT)
    from variable_length_prefill_gb300 import head_shard
    owner = np.full(H, -1)
    for r in range(world):
        b, c = head_shard(H, r, world)
        assert c >= 0 and 0 <= b and b + c <= H
        assert (owner[b:b + c] == -1).all()
        owner[b:b + c] = r
    assert (owner >= 0).all()
    counts = [head_shard(H, r, world)[1] for r in range(world)]
    assert max(counts) - min(counts) <= 1


def test_bad_shard_requests():
    sys.path.insert(0, ROOT)
    from variable_length_prefill_gb300 import head_shard
    for args in ((4, 2, 2), (4, -1, 2), (4, 0, 0), (-1, 0, 1)):
        with pytest.raises(ValueError):
            head_shard(*args)


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle
    from variable_length_prefill_gb300 import head_shard
    from workloads import Workload, make_inputs
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = Workload("shard", (37, 0, 150, 1), 5, 72, seed=91, seq_lens_k=(60, 3, 150, 9))
        x = make_inputs(w)
        b, c = head_shard(w.num_heads, rank, world)
        part = oracle.attn_varlen(x["q"][:, b:b + c], x["k"][:, b:b + c], x["v"][:, b:b + c],
                                  x["cu_q"], x["cu_k"], fill=0.0)
        # gather the shards (padded to the largest count) and reassemble heads
        cmax = max(head_shard(w.num_heads, r, world)[1] for r in range(world))
        buf = torch.zeros((part.shape[0], cmax, part.shape[2]), dtype=torch.float64)
        buf[:, :c] = torch.from_numpy(part)
        got = [torch.zeros_like(buf) for _ in range(world)]
        dist.all_gather(got, buf)
        if rank == 0:
            whole = np.concatenate(
                [got[r].numpy()[:, :head_shard(w.num_heads, r, world)[1]] for r in range(world)],
                axis=1)
            ref = oracle.attn_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], fill=0.0)
            q.put(("cmp", bool(np.array_equal(whole, ref)), whole.shape))
        q.put(("ok", rank))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reassemble_the_single_rank_result():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29600 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    msgs = [q.get(timeout=10) for _ in range(3)]
    cmp = [m for m in msgs if m[0] == "cmp"]
    assert cmp and cmp[0][1], cmp
    assert sorted(m[1] for m in msgs if m[0] == "ok") == [0, 1]
