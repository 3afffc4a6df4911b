"""The N > 1 host logic on CPU: two gloo ranks (127.0.0.1), barrier and max over ranks, and
the split of independent (batch, head) sequences between ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from ssm_sequence_layer_gb300.replicas import max_over_ranks, shard_sequences


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    from ssm_sequence_layer_gb300.replicas import barrier, max_over_ranks, shard_sequences
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    barrier(world)
    m = max_over_ranks(1.5 + rank, world)
    lo, hi = shard_sequences(3, 5, world, rank)
    barrier(world)
    dist.destroy_process_group()
    q.put((rank, m, lo, hi))


def test_two_gloo_ranks_agree_on_the_max_and_cover_all_sequences():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]
    covered = []
    for _, _, lo, hi in res:
        covered.extend(range(lo, hi))
    assert covered == list(range(15))


@pytest.mark.parametrize("B,H,world", [(1, 1, 1), (2, 4, 3), (1, 16, 8), (4, 8, 5), (1, 3, 4)])
def test_shards_partition_the_sequences(B, H, world):
    seen = []
    sizes = []
    for r in range(world):
        lo, hi = shard_sequences(B, H, world, r)
        seen.extend(range(lo, hi))
        sizes.append(hi - lo)
    assert seen == list(range(B * H))
    assert max(sizes) - min(sizes) <= 1


def test_single_rank_max_is_identity():
    assert max_over_ranks(3.25, 1) == 3.25
    with pytest.raises(ValueError):
        shard_sequences(1, 1, 2, 2)
