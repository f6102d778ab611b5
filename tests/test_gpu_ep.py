"""Expert parallelism on one GPU: the per-rank steps (moe_ep_permute,
moe_ep_regroup, the rank's grouped GEMM, moe_combine) of a group of 2 or 4
ranks, run one rank after another on the same device, with the two
all-to-alls replaced by copies of row blocks between the ranks' buffers
(no kernel waits on another rank's kernel).

Checked against the oracle's expert-parallel dispatch (bit for bit: kept
counts, offsets, destinations, send counts, the rows each rank receives) and
against the single-device layer over all tokens (global capacity: identical
routing and drops, outputs within the FFN bars and mostly bit-identical);
the per-rank capacity mode against the oracle layer on each shard alone.
moe_ep_regroup alone against a host permutation."""
import numpy as np
import pytest
import torch

import top_routing_expert_gb300 as moe
import workloads as W
from oracle import moe_oracle as O
from tests._helpers import assert_ffn_close, np64, oracle_logits_chunked

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    moe.load_library()


def _z(shape, dt):
    return torch.zeros(shape, dtype=dt, device=DEV)


def _host_regroup(counts, rows, to_expert_major):
    """Row permutation between source-major and expert-major order."""
    world, E_loc = counts.shape
    src_blocks, pos = {}, 0
    for r in range(world):
        for e in range(E_loc):
            src_blocks[(r, e)] = (pos, int(counts[r, e]))
            pos += int(counts[r, e])
    order = [i for e in range(E_loc) for r in range(world)
             for i in range(src_blocks[(r, e)][0], sum(src_blocks[(r, e)]))]
    out = torch.empty_like(rows[:pos])
    if to_expert_major:
        out[:] = rows[order]
    else:
        out[order] = rows[:pos]
    return out


@pytest.mark.parametrize("world,E_loc,H,seed", [(2, 4, 64, 0), (4, 2, 192, 1), (8, 32, 64, 2),
                                                (1, 16, 128, 3)])
def test_regroup_is_the_host_permutation_and_inverts(world, E_loc, H, seed):
    gen = torch.Generator().manual_seed(seed)
    counts = torch.randint(0, 40, (world, E_loc), generator=gen, dtype=torch.int32)
    counts[0, 0] = 0                      # empty blocks, including the first
    counts[-1, -1] = 0
    n = int(counts.sum())
    rows = torch.randn((n, H), generator=gen).to(torch.bfloat16)
    fwd = _z((n, H), torch.bfloat16)
    off = _z(E_loc + 1, torch.int32)
    moe.moe_ep_regroup(world, E_loc, counts.to(DEV), rows.to(DEV), fwd, True, off)
    back = _z((n, H), torch.bfloat16)
    moe.moe_ep_regroup(world, E_loc, counts.to(DEV), fwd, back, False)
    torch.cuda.synchronize()
    ref = _host_regroup(counts, rows, True)
    assert torch.equal(fwd.cpu().view(torch.int16), ref.view(torch.int16))
    assert torch.equal(back.cpu().view(torch.int16), rows.view(torch.int16))
    per_e = counts.sum(0).numpy()
    assert np.array_equal(off.cpu().numpy(), np.concatenate([[0], np.cumsum(per_e)]))


def test_regroup_never_writes_past_the_buffer():
    counts = torch.tensor([[5, 7], [6, 2]], dtype=torch.int32)   # 20 rows sent
    rows = torch.randn((12, 64)).to(torch.bfloat16)
    dst = torch.full((14, 64), 3.0, dtype=torch.bfloat16, device=DEV)
    moe.moe_ep_regroup(2, 2, counts.to(DEV), rows.to(DEV), dst[:12], True)
    torch.cuda.synchronize()
    assert (dst[12:].float().cpu() == 3.0).all()


def _run_group(w, inp, world, capacity):
    """The expert-parallel layer of `world` ranks, each holding T/world
    contiguous tokens and E/world experts, run rank by rank on this GPU."""
    T, H, E, k, h = w.T, w.H, w.E, w.k, w.h
    E_loc, Tl = E // world, T // world
    d = {n: (v.to(DEV) if v is not None else None) for n, v in inp.items()}
    s = moe.MoeShape.make(Tl, H, E, k, h, w.cf)
    ranks = []
    for r in range(world):
        x = d["x"][r * Tl:(r + 1) * Tl].contiguous()
        st = dict(x=x, idx=_z((Tl, k), torch.int32), w=_z((Tl, k), torch.float32),
                  routed=_z(E, torch.int32), ws=moe.Workspace(s), status=_z(1, torch.int32))
        moe.moe_route(s, x, d["gate"], d["bias"], st["idx"], st["w"], st["routed"],
                      dev_status=st["status"], ws=st["ws"])
        ranks.append(st)
    routed_all = torch.stack([st["routed"] for st in ranks]).contiguous()   # the all-gather
    for r, st in enumerate(ranks):
        st.update(kept=_z(E, torch.int32), off=_z(E + 1, torch.int32),
                  dest=_z((Tl, k), torch.int32), src=_z(Tl * k, torch.int32),
                  xp=_z((Tl * k, H), torch.bfloat16), send=_z(world, torch.int32))
        moe.moe_ep_permute(s, world, r, st["x"], st["idx"], st["kept"], st["off"], st["dest"],
                           st["src"], st["xp"], st["send"],
                           routed_all=routed_all if capacity == "global" else None,
                           T_global=T, dev_status=st["status"], ws=st["ws"])
    torch.cuda.synchronize()
    # the counts exchange: rank g's row r = source r's kept counts of g's experts
    recv_counts = [torch.stack([ranks[r]["kept"][g * E_loc:(g + 1) * E_loc]
                                for r in range(world)]).contiguous() for g in range(world)]
    # the rows exchange: source r's block for g = its x_perm rows of g's experts
    blocks = [[None] * world for _ in range(world)]
    for r, st in enumerate(ranks):
        off = st["off"].cpu()
        for g in range(world):
            blocks[r][g] = st["xp"][int(off[g * E_loc]):int(off[(g + 1) * E_loc])]
    y_blocks = [[None] * world for _ in range(world)]
    for g in range(world):
        x_recv = torch.cat([blocks[r][g] for r in range(world)]).contiguous()
        n = x_recv.shape[0]
        x_loc, y_loc, y_send = (_z((max(n, 1), H), torch.bfloat16) for _ in range(3))
        act = _z((max(n, 1), h), torch.bfloat16)
        loff = _z(E_loc + 1, torch.int32)
        moe.moe_ep_regroup(world, E_loc, recv_counts[g], x_recv, x_loc[:n], True, loff)
        ranks[g]["recv_expert_major"] = x_loc[:n].clone()
        fs = moe.MoeShape.make(n, H, E_loc, 1, h, 1.0)
        moe.moe_expert_ffn(fs, x_loc, loff, d["W1"][g * E_loc:(g + 1) * E_loc].contiguous(),
                           d["W2"][g * E_loc:(g + 1) * E_loc].contiguous(), act, y_loc,
                           dev_status=ranks[g]["status"])
        moe.moe_ep_regroup(world, E_loc, recv_counts[g], y_loc[:n], y_send[:n], False)
        pos = 0
        for r in range(world):
            c = blocks[r][g].shape[0]
            y_blocks[r][g] = y_send[pos:pos + c]
            pos += c
    ys = []
    for r, st in enumerate(ranks):
        yp = _z((Tl * k, H), torch.bfloat16)
        yp[:sum(b.shape[0] for b in y_blocks[r])] = torch.cat(y_blocks[r])   # the return trip
        y = _z((Tl, H), torch.bfloat16)
        moe.moe_combine(s, yp, st["dest"], st["w"], y)
        ys.append(y)
    torch.cuda.synchronize()
    for st in ranks:
        assert int(st["status"].item()) == 0
    return ranks, torch.cat(ys).cpu()


@pytest.mark.parametrize("world,T,H,E,k,h,cf,bias", [
    (2, 2048, 256, 8, 2, 384, 0.8, "zipf"),     # drops, the CTA-pair GEMM on the full layer
    (4, 1000, 192, 12, 3, 320, 1.0, "zipf"),    # ragged, E/world = 3
    (4, 4096, 512, 16, 2, 256, 1.0, "zipf"),    # the imbalanced workload's routing shape
])
def test_ep_group_equals_the_single_device_layer(world, T, H, E, k, h, cf, bias):
    w = W.custom(T, H, E, k, h, cf, bias, name=f"ep{world}")
    inp = W.make_inputs(w, seed=world + T)
    ranks, y_ep = _run_group(w, inp, world, "global")
    # the single-device layer over all tokens
    s = moe.MoeShape.make(T, H, E, k, h, cf)
    d = {n: (v.to(DEV) if v is not None else None) for n, v in inp.items()}
    y = _z((T, H), torch.bfloat16)
    idx = _z((T, k), torch.int32)
    dest = _z((T, k), torch.int32)
    moe.moe_layer_fwd(s, d["x"], d["gate"], d["bias"], d["W1"], d["W2"], y, topk_idx=idx,
                      dest_row=dest, ws=moe.Workspace(s))
    torch.cuda.synchronize()
    Tl, E_loc = T // world, E // world
    gidx = idx.cpu().numpy()
    assert np.array_equal(np.concatenate([st["idx"].cpu().numpy() for st in ranks]), gidx)
    kept_ep = np.concatenate([st["dest"].cpu().numpy() >= 0 for st in ranks])
    assert np.array_equal(kept_ep, dest.cpu().numpy() >= 0)
    # the oracle's expert-parallel dispatch of the GPU's indices, bit for bit
    C = O.capacity(T, E, k, cf)
    before = np.zeros(E, np.int64)
    x_all = inp["x"].view(torch.int16)
    for r, st in enumerate(ranks):
        ir = gidx[r * Tl:(r + 1) * Tl]
        dp = O.ep_dispatch_plan(ir, E, C, before)
        assert np.array_equal(st["kept"].cpu().numpy(), dp.kept_counts)
        assert np.array_equal(st["off"].cpu().numpy(), dp.offsets)
        assert np.array_equal(st["dest"].cpu().numpy(), dp.dest_row)
        assert np.array_equal(st["send"].cpu().numpy(), O.ep_send_counts(dp.kept_counts, world))
        before += np.bincount(ir.reshape(-1), minlength=E)
    # rank g's regrouped rows are the single-device buffer's rows of its experts
    dd = O.dispatch_plan(gidx, E, C)
    for g, st in enumerate(ranks):
        a, b = int(dd.offsets[g * E_loc]), int(dd.offsets[(g + 1) * E_loc])
        want = x_all[torch.from_numpy(dd.src_token[a:b]).long()]
        assert torch.equal(st["recv_expert_major"].cpu().view(torch.int16), want)
    # outputs: the same rows through the same experts
    assert_ffn_close(np64(y_ep), np64(y.cpu()), "ep layer vs single-device layer")
    assert (y_ep.view(torch.int16) == y.cpu().view(torch.int16)).float().mean() > 0.99


def test_ep_per_rank_capacity_equals_each_shard_alone():
    """Capacity from each rank's own batch (the module notes' listing): rank
    r's outputs are the oracle layer's on its shard alone."""
    world = 2
    w = W.custom(1200, 128, 8, 2, 192, 0.7, "zipf", name="ep_local")
    inp = W.make_inputs(w, seed=5)
    ranks, y_ep = _run_group(w, inp, world, "per_rank")
    Tl = w.T // world
    for r, st in enumerate(ranks):
        sh = slice(r * Tl, (r + 1) * Tl)
        lg = oracle_logits_chunked(inp["x"][sh], inp["gate"], inp["bias"])
        rr = O.route_from_logits(lg, w.k)
        gidx = st["idx"].cpu().numpy()
        mism = (gidx != rr.idx).any(axis=1)
        assert not mism.any()   # these seeds have no near-ties
        dp = O.ep_dispatch_plan(gidx, w.E, O.capacity(Tl, w.E, w.k, w.cf))
        assert np.array_equal(st["dest"].cpu().numpy(), dp.dest_row)
        ref = O.token_outputs(np64(inp["x"][sh]), gidx, rr.w, dp.dest_row >= 0,
                              np64(inp["W1"]), np64(inp["W2"]))
        assert_ffn_close(np64(y_ep[sh]), ref, f"per-rank capacity rank {r}")


DRIVER_CHILD = r"""
import json, os, sys
sys.path.insert(0, ROOT)
import torch, torch.distributed as dist
import top_routing_expert_gb300 as moe
from top_routing_expert_gb300.ep import ExpertParallelMoE
import workloads as W
moe.build(); moe.load_library()
torch.cuda.set_device(0)
dist.init_process_group("nccl", init_method="tcp://127.0.0.1:PORT", rank=0, world_size=1)
out = {}
for cap in ("global", "per_rank"):
    w = W.custom(2048, 256, 8, 2, 384, 0.8, "zipf", name="ep_driver")
    inp = W.make_inputs(w, seed=9)
    d = {n: (v.cuda() if v is not None else None) for n, v in inp.items()}
    layer = ExpertParallelMoE(w.T, w.H, w.E, w.k, w.h, w.cf, capacity=cap)
    y = layer.forward(d["x"], d["gate"], d["bias"], d["W1"], d["W2"])
    s = moe.MoeShape.make(w.T, w.H, w.E, w.k, w.h, w.cf)
    y_ref = torch.empty_like(y)
    moe.moe_layer_fwd(s, d["x"], d["gate"], d["bias"], d["W1"], d["W2"], y_ref,
                      ws=moe.Workspace(s))
    torch.cuda.synchronize()
    out[cap] = {"equal": bool(torch.equal(y, y_ref)), "status": int(layer.status.item())}
dist.destroy_process_group()
print("EP_RESULT " + json.dumps(out), flush=True)
"""


def test_ep_driver_on_a_one_rank_group_equals_the_layer():
    """The driver (top_routing_expert_gb300.ep) with every collective issued
    for real on a one-rank NCCL group: all experts are local, so both
    capacity modes must give moe_layer_fwd's bits."""
    import json
    import os
    import socket
    import subprocess
    import sys
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = DRIVER_CHILD.replace("ROOT", repr(root)).replace("PORT", str(port))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, NCCL_NVLS_ENABLE="0"))
    assert r.returncode == 0, r.stderr[-3000:]
    # NCCL may print its own lines to stdout too, in either order
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("EP_RESULT ")]
    assert len(lines) == 1, r.stdout[-3000:]
    out = json.loads(lines[0][len("EP_RESULT "):])
    for cap, res in out.items():
        assert res["status"] == 0 and res["equal"], (cap, res)
