"""Expert parallelism over two CPU ranks (gloo): the exchange protocol of
top_routing_expert_gb300.ep - gathering every rank's routed counts, the
counts all-to-all and the row all-to-alls out and back with uneven split
sizes - run for real, with each rank's compute done by the oracle.

Each rank holds half of the tokens (contiguous) and half of the experts.
With the global capacity (every expert serves the group's tokens in global
order) the two ranks' outputs must be exactly the oracle's single-device
layer over all tokens; with the per-rank capacity, each rank's outputs are
the oracle layer on its shard alone."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import moe_oracle as O

WORLD = 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _inputs():
    import workloads as W
    w = W.custom(240, 64, 8, 2, 64, 0.8, "zipf", name="ep_gloo")
    inp = W.make_inputs(w, seed=3)
    f64 = lambda t: t.float().numpy().astype(np.float64)
    return w, f64(inp["x"]), f64(inp["gate"]), inp["bias"].numpy(), f64(inp["W1"]), f64(inp["W2"])


def _regroup(counts, rows, to_expert_major):
    """Source-major <-> expert-major row order (as moe_ep_regroup)."""
    world, E_loc = counts.shape
    start = np.concatenate([[0], np.cumsum(counts.reshape(-1))])
    order = [i for e in range(E_loc) for r in range(world)
             for i in range(start[r * E_loc + e], start[r * E_loc + e + 1])]
    out = np.empty_like(rows)
    if to_expert_major:
        out[:] = rows[order]
    else:
        out[order] = rows
    return out


def _worker(rank, world, port, capacity, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from top_routing_expert_gb300 import ep
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, x_all, gate, bias, W1, W2 = _inputs()
        E, k, H = w.E, w.k, w.H
        E_loc = E // world
        sh = np.array_split(np.arange(w.T), world)[rank]
        x = x_all[sh]
        r = O.route_from_logits(O.router_logits(x, gate, bias), k)
        routed = torch.from_numpy(np.bincount(r.idx.reshape(-1), minlength=E).astype(np.int32))
        routed_all, T_global = ep.gather_routed(routed, len(sh))
        if capacity == "global":
            C = O.capacity(T_global, E, k, w.cf)
            before = routed_all[:rank].sum(dim=0).numpy().astype(np.int64)
            d = O.ep_dispatch_plan(r.idx, E, C, before)
        else:
            d = O.ep_dispatch_plan(r.idx, E, O.capacity(len(sh), E, k, w.cf))
        x_perm = O.permute(x, d)
        send = O.ep_send_counts(d.kept_counts, world)
        recv_counts = ep.exchange_counts(torch.from_numpy(d.kept_counts.astype(np.int32)), world)
        recv = recv_counts.sum(dim=1).tolist()
        x_recv = ep.exchange_rows(torch.from_numpy(x_perm), send, recv).numpy()
        cnt = recv_counts.numpy()
        x_loc = _regroup(cnt, x_recv, True)
        off = np.concatenate([[0], np.cumsum(cnt.sum(axis=0))])
        y_loc = O.expert_ffn(x_loc, off, W1[rank * E_loc:(rank + 1) * E_loc],
                             W2[rank * E_loc:(rank + 1) * E_loc])
        y_send = _regroup(cnt, y_loc, False)
        y_perm = ep.exchange_rows(torch.from_numpy(y_send), recv, send).numpy()
        y = O.combine(y_perm, d, r.w, H)
        q.put((rank, sh, y, d.dest_row >= 0, int(T_global), routed_all.numpy()))
    finally:
        dist.destroy_process_group()


def _run(capacity):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, WORLD, port, capacity, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    got = sorted([q.get(timeout=300) for _ in procs], key=lambda g: g[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return got


def test_two_rank_expert_parallel_layer_equals_single_device():
    got = _run("global")
    w, x, gate, bias, W1, W2 = _inputs()
    ref = O.layer_forward(x, gate, bias, W1, W2, w.k, w.cf)
    y = np.concatenate([g[2] for g in got])
    kept = np.concatenate([g[3] for g in got])
    assert got[0][4] == w.T
    assert np.array_equal(got[0][5], got[1][5])            # both ranks saw the same counts
    assert np.array_equal(kept, ref.dispatch.dest_row >= 0)
    assert (~kept).any()                                    # the case drops
    assert np.array_equal(y, ref.y)


def test_two_rank_per_rank_capacity_equals_each_shard():
    got = _run("per_rank")
    w, x, gate, bias, W1, W2 = _inputs()
    for rank, sh, y, kept, _, _ in got:
        ref = O.layer_forward(x[sh], gate, bias, W1, W2, w.k, w.cf)
        assert np.array_equal(kept, ref.dispatch.dest_row >= 0)
        assert np.array_equal(y, ref.y)
