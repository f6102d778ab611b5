"""One rank of an expert-parallel MoE layer forward.

The experts are spread over the ranks of a process group, rank g holding the
E/world consecutive experts g*E/world .. (g+1)*E/world - 1 (W1/W2 of those
experts only). Each token's rows travel to the rank of its expert and back:
the dispatch and combine all-to-alls of the MoE comm bottleneck page,
section 1.1, whose bytes section 2.1 counts (B*k*H*dtype each way); the MoE
module notes' MoELayer listing, section 4.2, routes through the same
exchange (_all_to_all_routed). Every step that computes runs in the
library's kernels; this module only allocates buffers and issues the
exchanges as torch.distributed collectives (NCCL on GPUs; the exchange
helpers below also run on CPU tensors with gloo).

A forward on rank r:
  1. moe_route on the rank's tokens (top-k, weights, routed counts);
  2. [global capacity] all ranks' routed counts and token counts gathered;
  3. moe_ep_permute: capacity drops and the expert-major dispatch buffer,
     whose rows for each destination rank are contiguous (send_counts);
  4. counts exchange: each rank learns how many rows every source sends for
     each of its experts;
  5. rows exchange (all-to-all with those sizes: the split sizes are read
     back to the host once per layer);
  6. moe_ep_regroup to expert-major, moe_expert_ffn on the rank's experts,
     moe_ep_regroup back;
  7. the reverse all-to-all returns every row to its source rank, in the
     order it was sent, so it lands at the row moe_ep_permute gave it;
  8. moe_combine with the rank's own weights and destinations.
With the global capacity (the default), the layer's outputs equal those of
the single-device layer over all ranks' tokens taken in rank order.
"""
from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist

from . import (MoeShape, Workspace, moe_combine, moe_ep_permute, moe_ep_regroup,
               moe_expert_ffn, moe_route)


def gather_routed(routed: torch.Tensor, T_local: int, group=None):
    """Every rank's routed counts [world, E] (int32, on routed's device) and
    the group's token count."""
    world = dist.get_world_size(group)
    buf = torch.cat([routed.to(torch.int32).reshape(-1),
                     torch.tensor([int(T_local)], dtype=torch.int32, device=routed.device)])
    allc = torch.empty((world, buf.numel()), dtype=torch.int32, device=routed.device)
    dist.all_gather(list(allc.unbind(0)), buf, group=group)
    return allc[:, :-1].contiguous(), sum(int(v) for v in allc[:, -1].tolist())


def exchange_counts(kept_counts: torch.Tensor, world: int, group=None) -> torch.Tensor:
    """kept_counts [E] of this rank -> recv_counts [world, E/world]: row r
    holds how many rows source rank r sends for each of this rank's
    experts."""
    send = kept_counts.to(torch.int32).reshape(world, -1).contiguous()
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send, group=group)
    return recv


def exchange_rows(rows: torch.Tensor, send_sizes, recv_sizes, group=None,
                  out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """All-to-all of row blocks: send_sizes[g] rows of `rows` (in rank order)
    go to rank g; the sum(recv_sizes) rows received, source by source, are
    returned (written to the first rows of `out` if given). The same call
    with the sizes swapped returns rows to their sources."""
    send_sizes = [int(v) for v in send_sizes]
    recv_sizes = [int(v) for v in recv_sizes]
    n = sum(recv_sizes)
    if out is None:
        out = torch.empty((n,) + tuple(rows.shape[1:]), dtype=rows.dtype, device=rows.device)
    out = out[:n]
    dist.all_to_all_single(out, rows[:sum(send_sizes)], output_split_sizes=recv_sizes,
                           input_split_sizes=send_sizes, group=group)
    return out


class ExpertParallelMoE:
    """The layer forward on one rank of an expert-parallel group: T tokens
    per rank (the group's batch is the ranks' tokens in rank order), H, E
    experts in all, top_k, expert width h, capacity factor cf.
    capacity="global": each expert serves the group's tokens in global order
    against the group's capacity (equal to the single-device layer);
    "per_rank": each rank applies its own batch's capacity to its tokens,
    as the module notes' listing does."""

    def __init__(self, T, H, E, k, h, cf, group=None, capacity: str = "global",
                 device: Optional[torch.device] = None):
        if capacity not in ("global", "per_rank"):
            raise ValueError("capacity is 'global' or 'per_rank'")
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if E % self.world:
            raise ValueError("the number of experts must be a multiple of the group size")
        self.E_loc = E // self.world
        self.capacity = capacity
        self.dev = device or torch.device("cuda", torch.cuda.current_device())
        self.shape = MoeShape.make(T, H, E, k, h, cf)
        self.ws = Workspace(self.shape, device=self.dev)
        z = lambda shape, dt: torch.zeros(shape, dtype=dt, device=self.dev)
        A = T * k
        self.idx, self.w = z((T, k), torch.int32), z((T, k), torch.float32)
        self.routed, self.P, self.aux = z(E, torch.int32), z(E, torch.float32), z(1, torch.float32)
        self.kept, self.offsets = z(E, torch.int32), z(E + 1, torch.int32)
        self.dest = z((T, k), torch.int32)
        self.x_perm, self.y_perm = z((max(A, 1), H), torch.bfloat16), z((max(A, 1), H), torch.bfloat16)
        self.send_counts = z(self.world, torch.int32)
        self.status = z(1, torch.int32)

    def forward(self, x, gate, gate_bias, W1_local, W2_local, y=None):
        """y [T,H] bf16 for this rank's tokens x [T,H]; gate [H,E] (all
        experts), W1_local [E/world,H,h], W2_local [E/world,h,H] of this
        rank's experts. Returns y."""
        s, world, E_loc = self.shape, self.world, self.E_loc
        T, H, h = s.T, s.H, s.h
        y = torch.empty((T, H), dtype=torch.bfloat16, device=self.dev) if y is None else y
        moe_route(s, x, gate, gate_bias, self.idx, self.w, self.routed, self.P, self.aux,
                  dev_status=self.status, ws=self.ws)
        routed_all, T_global = None, 0
        if self.capacity == "global":
            routed_all, T_global = gather_routed(self.routed, T, self.group)
        moe_ep_permute(s, world, self.rank, x, self.idx, self.kept, self.offsets, self.dest, None,
                       self.x_perm, self.send_counts, routed_all=routed_all, T_global=T_global,
                       dev_status=self.status, ws=self.ws)
        recv_counts = exchange_counts(self.kept, world, self.group)
        # the split sizes of the row exchanges, read back once per layer
        send_sizes = self.send_counts.tolist()
        recv_sizes = [sum(r) for r in recv_counts.tolist()]
        x_recv = exchange_rows(self.x_perm, send_sizes, recv_sizes, self.group)
        n = x_recv.shape[0]
        y_send = torch.empty_like(x_recv)
        if n > 0:   # a rank whose experts received nothing has no FFN to run
            x_loc = torch.empty_like(x_recv)
            local_off = torch.zeros(E_loc + 1, dtype=torch.int32, device=self.dev)
            moe_ep_regroup(world, E_loc, recv_counts, x_recv, x_loc, True, local_off)
            act = torch.empty((n, h), dtype=torch.bfloat16, device=self.dev)
            y_loc = torch.empty_like(x_loc)
            ffn_shape = MoeShape.make(n, H, E_loc, 1, h, 1.0)
            moe_expert_ffn(ffn_shape, x_loc, local_off, W1_local, W2_local, act, y_loc,
                           dev_status=self.status)
            moe_ep_regroup(world, E_loc, recv_counts, y_loc, y_send, False)
        exchange_rows(y_send, recv_sizes, send_sizes, self.group, out=self.y_perm)
        moe_combine(s, self.y_perm, self.dest, self.w, y)
        return y
