"""Multi-GPU host logic, checked with two gloo ranks on CPU.

bench.py runs one pool replica per rank (weak scaling) with no data-path
collective; the only cross-rank step is the max of the timings.  A slot
partition (gated_deltanet_recurrent_gb300.shard) gives each rank one
contiguous range of the slot space: two ranks that decode only the requests
routed to them, on the oracle, must reproduce one pool decoding everything,
bit for bit."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp
import numpy as np

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 10.0 - rank, 0.5 * (rank + 1)]
        out[rank] = bench.max_over_ranks(mine, dist, torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    for r in range(world):
        assert got[r] == [2.0, 10.0, 1.0]


# ---- slot partition: two ranks, each owning half of the slot space

from gated_deltanet_recurrent_gb300 import shard, synth  # noqa: E402
from oracle import gdn_oracle as O  # noqa: E402

N_SLOTS, STEPS = 9, 3
SHAPE = synth.LayerShape(2, 1, 8, 8, 4, 4)


def _batch(step):
    rng = np.random.default_rng(100 + step)
    ids = rng.choice(N_SLOTS, 6, replace=False)
    return ids, synth.token_inputs(rng, len(ids), SHAPE, "f32")


def _initial_states():
    return synth.random_states(np.random.default_rng(99), N_SLOTS, SHAPE)


def _shard_worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lo, hi = shard.slot_range(rank, world, N_SLOTS)
        pool = O.OraclePool(1, hi - lo, SHAPE.h_v, SHAPE.h_k, SHAPE.dk, SHAPE.dv, 4, 4)
        pool.S[0] = _initial_states()[lo:hi]
        outs = []
        for step in range(STEPS):
            ids, tok = _batch(step)
            pos, local = shard.route(ids, world, N_SLOTS)[rank]
            o = np.zeros((len(ids), SHAPE.h_v, SHAPE.dv))
            if len(pos):
                o[pos] = pool.decode_step(0, local, *(tok[n][pos] for n in
                                                      ("q", "k", "v", "g", "beta")))
            # gather: every rank contributes its entries (zeros elsewhere)
            t = torch.from_numpy(o)
            dist.all_reduce(t)
            outs.append(t.numpy().copy())
        out[rank] = (np.stack(outs), pool.S[0].copy(), lo, hi)
    finally:
        dist.destroy_process_group()


def test_slot_partition_over_two_gloo_ranks_equals_one_pool():
    """Each rank owns a contiguous half of the slots and decodes only the
    requests routed to it; the gathered outputs and the union of the ranks'
    states equal one pool decoding everything, bit for bit."""
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_shard_worker, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    ref = O.OraclePool(1, N_SLOTS, SHAPE.h_v, SHAPE.h_k, SHAPE.dk, SHAPE.dv, 4, 4)
    ref.S[0] = _initial_states()
    ref_o = []
    for step in range(STEPS):
        ids, tok = _batch(step)
        ref_o.append(ref.decode_step(0, ids, *(tok[n] for n in ("q", "k", "v", "g", "beta"))))
    for r in range(world):
        o, S, lo, hi = got[r]
        np.testing.assert_array_equal(o, np.stack(ref_o))
        np.testing.assert_array_equal(S, ref.S[0, lo:hi])


def test_slot_range_and_route_cover_the_slots_once():
    for n_slots, world in ((9, 2), (512, 8), (5, 4), (3, 3)):
        ranges = [shard.slot_range(r, world, n_slots) for r in range(world)]
        assert ranges[0][0] == 0 and ranges[-1][1] == n_slots
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
        for s in range(n_slots):
            r = shard.owner(s, world, n_slots)
            assert ranges[r][0] <= s < ranges[r][1]
        ids = np.random.default_rng(n_slots).permutation(n_slots)[: max(1, n_slots // 2)]
        parts = shard.route(ids, world, n_slots)
        seen = np.concatenate([p for p, _ in parts])
        assert sorted(seen.tolist()) == list(range(len(ids)))
        for r, (pos, local) in enumerate(parts):
            np.testing.assert_array_equal(local + ranges[r][0], ids[pos])
