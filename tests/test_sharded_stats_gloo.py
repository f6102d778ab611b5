"""Token-sharded replicas (world size 2, gloo on CPU).

With every expert resident on every GPU, each replica routes its own tokens
and the layer output needs no exchange. The load-balancing statistics are
global, though: summing per-rank expert counts and per-rank probability sums
with one all-reduce of 2E numbers must give the unsharded f, P and aux.
(The capacity rule stays per replica: C is computed from the local T.)"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import moe_oracle as O


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, logits, k, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T, E = logits.shape
        shard = np.array_split(np.arange(T), world)[rank]
        r = O.route_from_logits(logits[shard], k)
        counts = torch.from_numpy(np.bincount(r.idx.reshape(-1), minlength=E).astype(np.float64))
        psum = torch.from_numpy(r.p.sum(axis=0))
        ntok = torch.tensor([float(len(shard))], dtype=torch.float64)
        buf = torch.cat([counts, psum, ntok])
        dist.all_reduce(buf)
        cnt, ps, n = buf[:E].numpy(), buf[E:2 * E].numpy(), float(buf[-1])
        f = cnt / (n * k)
        P = ps / n
        q.put((rank, cnt, f, P, float(E * np.sum(f * P))))
    finally:
        dist.destroy_process_group()


def test_two_rank_stats_equal_unsharded():
    rng = np.random.default_rng(7)
    T, E, k = 301, 12, 3
    logits = (rng.standard_normal((T, E)) + np.linspace(1, -1, E)).astype(np.float32)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, logits, k, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    r = O.route_from_logits(logits, k)
    st = O.load_balance_stats(r.idx, r.p, E)
    for rank, cnt, f, P, aux in got:
        assert np.array_equal(cnt.astype(np.int64), st.routed)
        assert np.allclose(f, st.f, rtol=0, atol=1e-15)
        assert np.allclose(P, st.P, rtol=1e-13, atol=0)
        assert abs(aux - st.aux) < 1e-12
