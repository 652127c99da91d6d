"""The Ring P2P exchange on CPU, with ``gloo`` process groups: the schedule
gives every device each K/V shard exactly once, :func:`ring.hop` delivers the
shard that the schedule says, and accumulators travelling with the K/V
shards arrive back at their owner after ``world`` hops with every device's
contribution.  No GPU and no attention arithmetic: this is the host logic of
the ring (the per-device computation is covered by test_gpu_ring)."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _ring():
    sys.path.insert(0, ROOT)
    from long_context_masked_mask_gb300 import ring
    return ring


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_schedule_visits_every_shard_once():
    ring = _ring()
    for world in (1, 2, 3, 5, 8):
        for r in range(world):
            sched = ring.schedule(r, world)
            assert sched[0] == r and sorted(sched) == list(range(world))
        # in every round the devices hold distinct shards (a permutation)
        for t in range(world):
            assert sorted(ring.kv_shard_at(r, t, world) for r in range(world)) == list(range(world))
    assert ring.shard_starts(10, 3) == [0, 3, 6, 10]
    with pytest.raises(ValueError):
        ring.shard_starts(2, 3)


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    ring = _ring()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        kv = torch.full((4,), float(rank))           # the K/V shard this device owns
        acc = torch.zeros(4)                          # its travelling dK/dV accumulator
        seen = []
        for t in range(world):
            held = int(kv[0].item())
            assert held == ring.kv_shard_at(rank, t, world)
            seen.append(held)
            acc += 10.0 ** rank                       # this device's contribution to shard `held`
            if t < world - 1:
                kv, acc = ring.hop([kv, acc], rank, world)
            else:
                (acc,) = ring.hop([acc], rank, world)  # the last hop takes the accumulator home
        q.put((rank, seen, acc.tolist()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_hop_with_gloo_ranks(world):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    total = sum(10.0 ** r for r in range(world))
    for rank, seen, acc in out:
        assert seen == [(rank - t) % world for t in range(world)]
        assert acc == [total] * 4                    # every device added to the owner's shard


def test_zigzag_chunks_cover_the_sequence_and_balance_causal_work():
    """Zigzag shards: every position in exactly one chunk; under CAUSAL every
    device does the same work (allowed pairs of its query chunks against all
    keys) to within 1% (chunk lengths differ by one row), while contiguous shards differ by about
    2 * world - 1 between the first and the last device."""
    import numpy as np
    import oracle
    from synthetic import MaskSpec
    ring = _ring()
    N = 999
    for world in (2, 3, 4):
        for layout in ("contiguous", "zigzag"):
            sh = ring.shard_chunks(N, world, layout)
            cover = np.zeros(N, int)
            for chunks in sh:
                for a, n in chunks:
                    cover[a:a + n] += 1
            assert (cover == 1).all()
        M = oracle.allowed(MaskSpec("CAUSAL"), N, np.arange(N))
        work = {lay: [sum(int(M[a:a + n].sum()) for a, n in chunks) for chunks in ring.shard_chunks(N, world, lay)]
                for lay in ("contiguous", "zigzag")}
        z = work["zigzag"]
        assert max(z) <= 1.01 * min(z)                             # equal up to chunk rounding
        c = work["contiguous"]
        assert c[-1] / c[0] > 2 * world - 2                        # the imbalance zigzag removes
    with pytest.raises(ValueError):
        ring.shard_chunks(5, 3, "zigzag")
