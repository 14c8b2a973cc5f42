"""Multi-rank host logic on the CPU (gloo, world size 2).

Jagged attention partitions into independent sequences, so N GPUs run N
replicas with no data-path collective. This checks, with two CPU ranks:
  * partitioning the sequences of a batch across ranks and reassembling the
    per-rank results gives exactly the full-batch result (fp64 oracle);
  * bench.py's max / sum over ranks (the timing and throughput reductions).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import sys
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        sys.path.insert(0, root)
        import oracle.attention as orc
        import bench

        rng = np.random.default_rng(0)  # every rank draws the same full batch
        lengths = [5, 17, 1, 9, 30, 2, 11]
        H, d = 2, 8
        off = np.concatenate([[0], np.cumsum(lengths)])
        T = int(off[-1])
        q, k, v, do = (rng.standard_normal((T, H, d)) for _ in range(4))
        # this rank's sequences: b = rank, rank + world, ...
        mine = list(range(rank, len(lengths), world))
        o_part = np.zeros((T, H, d))
        dq_part = np.zeros((T, H, d))
        for b in mine:
            s0, s1 = int(off[b]), int(off[b + 1])
            one = np.array([0, s1 - s0])
            O, _ = orc.attention_forward(q[s0:s1], k[s0:s1], v[s0:s1], one, 0.5)
            dQ, _, _, _ = orc.attention_backward(q[s0:s1], k[s0:s1], v[s0:s1], do[s0:s1], one, 0.5)
            o_part[s0:s1] = O
            dq_part[s0:s1] = dQ
        # reassemble: each row is owned by exactly one rank, the others contribute zeros
        t_o = torch.from_numpy(o_part)
        t_dq = torch.from_numpy(dq_part)
        dist.all_reduce(t_o)
        dist.all_reduce(t_dq)
        O_full, _ = orc.attention_forward(q, k, v, off, 0.5)
        dQ_full, _, _, _ = orc.attention_backward(q, k, v, do, off, 0.5)
        err = max(float(np.max(np.abs(t_o.numpy() - O_full))), float(np.max(np.abs(t_dq.numpy() - dQ_full))))
        mx = bench.max_over_ranks(dist, float(rank + 1) * 1.5, "cpu")
        sm = bench.sum_over_ranks(dist, float(rank + 1), "cpu")
        out_q.put((rank, err, mx, sm))
    finally:
        dist.destroy_process_group()


def test_two_rank_partition_and_reductions():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, err, mx, sm in results:
        assert err < 1e-13, (rank, err)
        assert mx == 3.0 and sm == 3.0


def _bcast_worker(rank, world, port, out_q):
    """Broadcast-Q backward with the batch sharded: each rank takes whole
    sequences (longest-first greedy on the key lengths, as a balanced shard
    would), computes its partial dQ, and one all-reduce (sum) gives the dQ of
    the whole batch; dK / dV rows belong to one rank each."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import sys
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        sys.path.insert(0, root)
        import oracle.attention as orc

        rng = np.random.default_rng(1)
        k_lengths = [7, 0, 23, 3, 12, 1, 18]
        Lq, H, d = 5, 2, 8
        off = np.concatenate([[0], np.cumsum(k_lengths)])
        T = int(off[-1])
        q = rng.standard_normal((Lq, H, d))
        k, v = (rng.standard_normal((T, H, d)) for _ in range(2))
        do = rng.standard_normal((len(k_lengths), Lq, H, d))
        load = [0] * world
        owner = {}
        for b in sorted(range(len(k_lengths)), key=lambda b: (-k_lengths[b], b)):
            r = min(range(world), key=lambda r: (load[r], r))
            owner[b] = r
            load[r] += k_lengths[b]
        mine = [b for b in range(len(k_lengths)) if owner[b] == rank]
        dq = np.zeros((Lq, H, d))
        dk = np.zeros((T, H, d))
        dv = np.zeros((T, H, d))
        for b in mine:
            s0, s1 = int(off[b]), int(off[b + 1])
            one = np.array([0, s1 - s0])
            a, kk, vv = orc.broadcast_backward(q, k[s0:s1], v[s0:s1], do[b:b + 1], one, 0.35)
            dq += a
            dk[s0:s1] = kk
            dv[s0:s1] = vv
        t = [torch.from_numpy(x) for x in (dq, dk, dv)]
        for x in t:
            dist.all_reduce(x)
        ref = orc.broadcast_backward(q, k, v, do, off, 0.35)
        err = max(float(np.max(np.abs(x.numpy() - r))) for x, r in zip(t, ref))
        out_q.put((rank, err, len(mine)))
    finally:
        dist.destroy_process_group()


def test_two_rank_broadcast_dq_all_reduce():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_bcast_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sum(n for _, _, n in results) == 7
    for rank, err, _ in results:
        assert err < 1e-12, (rank, err)
