"""Expert parallelism across GPUs: one MoE layer pass on one EP rank.

Blog post "专家并行(EP)": section 2.1 places the experts of block g (32 of
256, or 33 slots with a replica) on EP rank g and replicates the shared
experts; section 2.2 follows a token through the dispatch all-to-all (step 2),
the expert FFN on the owning rank (step 3) and the combine all-to-all back
(step 4); section 2.3 gives the volume, 2 x top-k x hidden x 2 bytes per token
each way; section 4.2 runs the all-to-alls through NCCL.

Every rank routes and dispatches its own tokens (the data-parallel part).  Its
dispatch buffer is grouped by slot, so the rows for rank g are block g's
contiguous segment.  The exchange is:

1. ``exchange_counts``: each rank sends rank g its per-slot counts of g's slots;
2. ``moe_ep_plan`` (libmoe, host): row counts of both all-to-alls and the
   permutations between the received (source-major) and the GEMM's
   (slot-major) layouts;
3. ``exchange_rows``: the dispatch all-to-all of token rows;
4. ``moe_gather_rows`` regroups them slot-major; the local experts' GEMMs run
   on them; ``moe_gather_rows`` puts the outputs back source-major;
5. ``return_rows``: the combine all-to-all, landing every output in the
   sender's dispatch-buffer order, where ``moe_combine`` finds it.

The collectives are torch.distributed calls (NCCL between GPUs); they carry
bytes and do no arithmetic.  Every arithmetic step is a libmoe kernel.  The
counts exchange needs the counts on the host for the plan: one
device-to-host copy of world x slots-per-rank integers per layer.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch
import torch.distributed as dist

from . import (MOE_FFN_AUTO, Shape, moe_combine, moe_dispatch, moe_ep_plan, moe_expert_ffn, moe_ffn_workspace_size,
               moe_gather_rows, moe_route, moe_route_workspace_size)


def exchange_counts(counts: torch.Tensor, world: int, spb: int, group=None) -> torch.Tensor:
    """All-to-all of per-slot counts: counts [world*spb (+1)] int32, this rank's
    dispatch counts; returns [world, spb] with row s = what rank s sends for
    this rank's slots."""
    send = counts[:world * spb].contiguous()
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send, group=group)
    return recv.view(world, spb)


def _as_bytes(t: torch.Tensor) -> torch.Tensor:
    """A row tensor viewed as rows of bytes (every backend moves uint8; gloo has no 16-bit types)."""
    return t.view(torch.uint8) if t.dtype != torch.uint8 else t


def exchange_rows(rows: torch.Tensor, send_rows, recv_rows, group=None) -> torch.Tensor:
    """Dispatch all-to-all: rows [sum(send_rows), ...] in rank-segment order ->
    [sum(recv_rows), ...] source-major."""
    out = torch.empty((int(np.sum(recv_rows)),) + tuple(rows.shape[1:]), dtype=rows.dtype, device=rows.device)
    dist.all_to_all_single(_as_bytes(out), _as_bytes(rows[:int(np.sum(send_rows))].contiguous()),
                           [int(v) for v in recv_rows], [int(v) for v in send_rows], group=group)
    return out


def return_rows(rows: torch.Tensor, send_rows, recv_rows, out: torch.Tensor, group=None) -> torch.Tensor:
    """Combine all-to-all, the reverse of exchange_rows: rows [sum(recv_rows), ...]
    source-major go back into out[:sum(send_rows)] (the sender's order)."""
    n = int(np.sum(send_rows))
    tmp = out[:n] if out[:n].is_contiguous() else torch.empty_like(out[:n])
    dist.all_to_all_single(_as_bytes(tmp), _as_bytes(rows.contiguous()), [int(v) for v in send_rows],
                           [int(v) for v in recv_rows], group=group)
    if tmp.data_ptr() != out[:n].data_ptr():
        out[:n].copy_(tmp)
    return out


@dataclasses.dataclass
class RankExperts:
    """The experts one EP rank holds: its block's slots and the shared experts."""
    w_gate: torch.Tensor   # [spb, I, H]
    w_up: torch.Tensor     # [spb, I, H]
    w_down: torch.Tensor   # [spb, H, I]
    ws_gate: Optional[torch.Tensor] = None
    ws_up: Optional[torch.Tensor] = None
    ws_down: Optional[torch.Tensor] = None


def local_shape(shape, world: int) -> Shape:
    """The shape the local expert GEMMs see: this rank's slots, no shared experts."""
    s = Shape.of(shape)
    spb = s.n_slots // world
    return Shape(s.hidden, s.inter, spb, min(s.top_k, spb), 0, 0, spb, 1)


@dataclasses.dataclass
class LocalDispatch:
    """This rank's routing and dispatch (its own tokens, all slots)."""
    idx: torch.Tensor
    topk_w: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    inv_perm: torch.Tensor
    x_disp: torch.Tensor


def local_dispatch(shape, T: int, x: torch.Tensor, w_router: torch.Tensor, bias, replica_of=None,
                   stream=None, logits: Optional[torch.Tensor] = None) -> LocalDispatch:
    """Steps 1-2 on this rank's tokens: router + top-k, then the dispatch
    permutation into a buffer grouped by slot (so by EP block).  logits [T, E]
    fp32: route from these instead of the router GEMM."""
    s = Shape.of(shape)
    dev = x.device
    k, S, H = s.top_k, s.n_slots, s.hidden
    n = T * k
    i32 = dict(dtype=torch.int32, device=dev)
    idx, tw = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device=dev)
    rws = torch.empty(max(16, moe_route_workspace_size(s, T)), dtype=torch.uint8, device=dev)
    if logits is None:
        moe_route(s, T, x, w_router, bias, None, None, idx, tw, rws, stream=stream)
    else:
        moe_route(s, T, None, None, None, logits, None, idx, tw, None, stream=stream)
    slot_of, counts, blocks = torch.empty(n, **i32), torch.empty(S + 1, **i32), torch.empty(s.n_blocks, **i32)
    offsets, perm, inv = torch.empty(S + 2, **i32), torch.empty(n, **i32), torch.empty(n, **i32)
    x_disp = torch.empty((n, H), dtype=torch.bfloat16, device=dev)
    moe_dispatch(s, T, x, idx, replica_of, slot_of, counts, blocks, offsets, perm, inv, x_disp, stream=stream)
    return LocalDispatch(idx, tw, counts, offsets, inv, x_disp)


def expert_rows(shape, world: int, plan: dict, recv: torch.Tensor, experts: RankExperts, mode: int = MOE_FFN_AUTO,
                stream=None) -> torch.Tensor:
    """Step 3 on the rows this rank received (source-major): regroup them
    slot-major, run this rank's experts, put the outputs back source-major."""
    R = plan["rows"]
    H = Shape.of(shape).hidden
    dev = recv.device
    y_src = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    if R == 0:
        return y_src
    sfs = torch.from_numpy(plan["slot_from_src"]).to(dev)
    ssf = torch.from_numpy(plan["src_from_slot"]).to(dev)
    x_loc = torch.empty_like(recv)
    moe_gather_rows(recv, sfs, x_loc, stream=stream)
    ls = local_shape(shape, world)
    loc_off = torch.from_numpy(plan["local_offsets"]).to(dev)
    t_eff = (R + ls.top_k - 1) // ls.top_k  # the GEMMs' row buffers hold t_eff * top_k rows
    y_loc = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(16, moe_ffn_workspace_size(ls, t_eff)), dtype=torch.uint8, device=dev)
    moe_expert_ffn(ls, t_eff, x_loc, x_loc, loc_off, experts.w_gate, experts.w_up, experts.w_down, None, None, None,
                   y_loc, None, mode, ws, stream=stream)
    moe_gather_rows(y_loc, ssf, y_src, stream=stream)
    return y_src


def finish(shape, T: int, x: torch.Tensor, experts: RankExperts, y_disp: torch.Tensor, d: LocalDispatch,
           out: torch.Tensor, mode: int = MOE_FFN_AUTO, stream=None) -> torch.Tensor:
    """Steps 4-5 on this rank's tokens, once the expert outputs are back in
    dispatch-buffer order: the shared experts (replicated on every rank) and
    the combine."""
    s = Shape.of(shape)
    dev = x.device
    y_sh = None
    if s.n_shared > 0:
        # this rank's slots with no routed rows (all offsets zero), and the shared experts
        ls = local_shape(shape, s.n_blocks)
        sh = Shape(s.hidden, s.inter, ls.n_experts, ls.top_k, s.n_shared, s.inter_shared, ls.n_slots, 1)
        y_sh = torch.empty((T, s.hidden), dtype=torch.float32, device=dev)
        zero_off = torch.zeros(sh.n_slots + 2, dtype=torch.int32, device=dev)
        y_none = torch.empty((max(1, T * sh.top_k), s.hidden), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(16, moe_ffn_workspace_size(sh, T)), dtype=torch.uint8, device=dev)
        moe_expert_ffn(sh, T, x, x, zero_off, experts.w_gate, experts.w_up, experts.w_down, experts.ws_gate,
                       experts.ws_up, experts.ws_down, y_none, y_sh, mode, ws, stream=stream)
    moe_combine(s, T, y_disp, d.inv_perm, d.topk_w, y_sh, out, stream=stream)
    return out


def ep_forward(shape, T: int, x: torch.Tensor, w_router: torch.Tensor, bias, experts: RankExperts,
               out: torch.Tensor, replica_of=None, group=None, mode: int = MOE_FFN_AUTO, stream=None) -> dict:
    """The MoE layer on this EP rank's T tokens (x [T, H] bf16 on this rank's
    GPU): the routed rows of block g are computed on rank g, everything else
    here.  Returns the plan and the dispatch for inspection."""
    world = dist.get_world_size(group)
    s = Shape.of(shape)
    assert s.n_blocks == world, "one EP block per rank"
    d = local_dispatch(s, T, x, w_router, bias, replica_of, stream)
    recv_counts = exchange_counts(d.counts, world, s.n_slots // world, group)
    plan = moe_ep_plan(s, world, d.counts.cpu().numpy(), recv_counts.cpu().numpy())
    recv = exchange_rows(d.x_disp, plan["send_rows"], plan["recv_rows"], group)
    y_src = expert_rows(s, world, plan, recv, experts, mode, stream)
    y_disp = torch.empty_like(d.x_disp)
    return_rows(y_src, plan["send_rows"], plan["recv_rows"], y_disp, group)
    finish(s, T, x, experts, y_disp, d, out, mode, stream)
    return dict(plan=plan, dispatch=d, recv_counts=recv_counts)


__all__ = ["exchange_counts", "exchange_rows", "return_rows", "RankExperts", "LocalDispatch", "local_shape",
           "local_dispatch", "expert_rows", "finish", "ep_forward"]
