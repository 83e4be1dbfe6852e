"""Expert parallelism across ranks, on the CPU: the exchange of "专家并行(EP)"
section 2.2 steps 2 and 4 between gloo ranks.

Every rank holds one EP block of slots and a shard of the tokens.  The
product's exchange code runs unchanged: the counts all-to-all and the two row
all-to-alls of ``moe_expert_layer_06_gb300.ep`` and libmoe's host planner
``moe_ep_plan``.  The arithmetic of every rank (routing, dispatch, the local
experts, the shared experts, the combine) is the oracle's, in fp64, and the
plan's permutations are applied with torch indexing (on a GPU they are
``moe_gather_rows``).  The layer output assembled over the ranks must equal
the single-process oracle layer bit for bit: every row's arithmetic is the
same, only where it runs changes.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle
from moe_expert_layer_06_gb300 import ep

BASE = mi.WORKLOADS["tiny"].with_(tokens=96, hidden=64, inter=32, n_experts=16, top_k=4, n_shared=1,
                                  inter_shared=32, n_slots=16, skew_alpha=1.5)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case(world: int, replicas: bool):
    w = BASE.with_(n_blocks=world)
    rep = None
    if replicas:  # one replica slot per block, hot experts from the batch's own histogram
        w = w.with_(n_slots=BASE.n_experts + world)
        x = mi.hidden_states(w)
        lo = oracle.router_logits(w, x, mi.router_weight(w), mi.router_bias(w))
        idx, _ = oracle.topk_softmax(lo, w.top_k)
        rep = oracle.plan_replicas(w, np.bincount(idx.ravel(), minlength=w.n_experts), world)
    return w, rep


def _rank(rank: int, world: int, port: int, replicas: bool):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, rep = _case(world, replicas)
        T, k, S, H = w.tokens, w.top_k, w.n_slots, w.hidden
        spb = S // world
        t0, t1 = rank * T // world, (rank + 1) * T // world  # this rank's token shard (even starts)
        Tr = t1 - t0
        x = mi.hidden_states(w, rows=slice(t0, t1))
        wr, b = mi.router_weight(w), mi.router_bias(w)
        wg, wu, wd = mi.stacked_expert_weights(w, rep)
        sg, su, sd = mi.stacked_shared_weights(w)
        # steps 1-2 on this rank's tokens (oracle)
        lo = oracle.router_logits(w, x, wr, b)
        idx, wt = oracle.topk_softmax(lo, k)
        so, invalid = oracle.slot_map(w, idx, rep)
        assert invalid == 0
        counts, _ = oracle.histogram(w, so)
        offsets, perm, inv, xd = oracle.dispatch(w, Tr, so, counts, x)
        x_disp = torch.from_numpy(xd.view(np.int16)).view(torch.bfloat16)
        # the exchange (product code): counts, plan, dispatch all-to-all
        recv_counts = ep.exchange_counts(torch.from_numpy(counts), world, spb)
        plan = m.moe_ep_plan(w, world, counts, recv_counts.numpy())
        assert np.array_equal(plan["send_rows"], counts[:S].reshape(world, spb).sum(1))
        recv = ep.exchange_rows(x_disp, plan["send_rows"], plan["recv_rows"])
        R = plan["rows"]
        assert recv.shape[0] == R == int(recv_counts.sum())
        # step 3 on the rows of this rank's slots (oracle), regrouped slot-major and back
        x_loc = recv[torch.from_numpy(plan["slot_from_src"]).long()]
        ls = ep.local_shape(w, world)
        lw = [t[rank * spb:(rank + 1) * spb] for t in (wg, wu, wd)]
        t_eff = max(1, (R + ls.top_k - 1) // ls.top_k)
        y_loc = oracle.expert_ffn(w.with_(n_slots=spb, n_experts=spb, top_k=ls.top_k, n_blocks=1, n_shared=0),
                                  t_eff, plan["local_offsets"], x_loc, *lw)[:R]
        y_src = torch.from_numpy(y_loc)[torch.from_numpy(plan["src_from_slot"]).long()]
        # combine all-to-all back into this rank's dispatch order, then steps 4-5 (oracle)
        y_disp = torch.zeros((Tr * k, H), dtype=torch.float64)
        ep.return_rows(y_src, plan["send_rows"], plan["recv_rows"], y_disp)
        ysh = oracle.shared_rows(w, x, sg, su, sd)
        out = torch.from_numpy(oracle.combine(w, Tr, y_disp.numpy(), inv, wt, ysh))
        sizes = [(r + 1) * T // world - r * T // world for r in range(world)]
        gathered = [torch.empty((n_, H), dtype=torch.float64) for n_ in sizes]
        dist.all_gather(gathered, out)
        if rank == 0:
            full = torch.cat(gathered).numpy()
            xg = mi.hidden_states(w)
            ref = oracle.moe_forward(w, xg, wr, b, rep, wg, wu, wd, sg, su, sd)
            assert np.array_equal(full, ref["out"]), np.abs(full - ref["out"]).max()
            # every rank received exactly the rows of its slots
            assert sum(int(c) for c in ref["counts"][:S]) == T * k
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,replicas", [(2, False), (8, False), (8, True)])
def test_ep_layer_across_ranks_equals_single_process_layer(world, replicas):
    m.build_library()
    mp.spawn(_rank, args=(world, _free_port(), replicas), nprocs=world, join=True)


def test_ep_plan_hand_case():
    """Four ranks of two slots: row counts both ways, slot-major offsets, and the
    two permutations between the received and the regrouped layouts."""
    w = mi.WORKLOADS["tiny"].with_(n_experts=8, n_slots=8, n_blocks=4)
    counts = np.array([3, 1, 0, 2, 5, 0, 1, 1, 0], np.int32)   # this rank's rows per slot (+ invalid bucket)
    recv = np.array([[3, 1], [2, 0], [0, 4], [1, 1]], np.int32)  # per source, rows for local slots 0 and 1
    p = m.moe_ep_plan(w, 4, counts, recv)
    assert p["send_rows"].tolist() == [4, 2, 5, 2]
    assert p["recv_rows"].tolist() == [4, 2, 4, 2] and p["rows"] == 12
    assert p["local_offsets"].tolist() == [0, 6, 12, 12]
    # received: s0 (slot 0: 0,1,2; slot 1: 3), s1 (slot 0: 4,5), s2 (slot 1: 6..9), s3 (slot 0: 10; slot 1: 11)
    assert p["slot_from_src"].tolist() == [0, 1, 2, 4, 5, 10, 3, 6, 7, 8, 9, 11]
    assert np.array_equal(p["src_from_slot"][p["slot_from_src"]], np.arange(12))
    # errors: world other than the block count, a negative count, maps without room
    with pytest.raises(m.MoeError):
        m.moe_ep_plan(w, 2, counts, np.zeros((2, 4), np.int32))
    bad = counts.copy()
    bad[1] = -1
    with pytest.raises(m.MoeError):
        m.moe_ep_plan(w, 4, bad, recv)


def _plan_by_definition(counts, recv, world, spb):
    """The plan written out from its definition: the rows of source s for local
    slot j arrive in source order, each source's rows in slot order; the
    regrouped layout lists slot 0's rows from source 0, 1, ..., then slot 1's."""
    send = [int(counts[r * spb:(r + 1) * spb].sum()) for r in range(world)]
    recv_rows = [int(recv[s].sum()) for s in range(world)]
    src_pos = {}  # (source, slot, i) -> source-major position
    pos = 0
    for s_ in range(world):
        for j in range(spb):
            for i in range(int(recv[s_, j])):
                src_pos[(s_, j, i)] = pos
                pos += 1
    slot_from_src, offsets = [], [0]
    for j in range(spb):
        for s_ in range(world):
            for i in range(int(recv[s_, j])):
                slot_from_src.append(src_pos[(s_, j, i)])
        offsets.append(len(slot_from_src))
    return send, recv_rows, offsets + [len(slot_from_src)], slot_from_src


@pytest.mark.parametrize("seed", range(12))
def test_ep_plan_matches_its_definition_on_random_counts(seed):
    """Random world sizes, slots per rank and counts (empty slots and sources
    included) against the plan written out row by row."""
    rng = np.random.default_rng([7, seed])
    world = int(rng.choice([1, 2, 4, 8]))
    spb = int(rng.integers(1, 9))
    S = world * spb
    w = mi.WORKLOADS["tiny"].with_(n_experts=S, n_slots=S, n_blocks=world)
    zero = rng.random(2 * S + 1) < 0.3
    counts = np.where(zero[:S + 1], 0, rng.integers(0, 40, S + 1)).astype(np.int32)
    recv = np.where(zero[S + 1:S + 1 + S].reshape(world, spb), 0,
                    rng.integers(0, 40, (world, spb))).astype(np.int32)
    p = m.moe_ep_plan(w, world, counts, recv)
    send, recv_rows, offsets, sfs = _plan_by_definition(counts, recv, world, spb)
    assert p["send_rows"].tolist() == send
    assert p["recv_rows"].tolist() == recv_rows and p["rows"] == len(sfs)
    assert p["local_offsets"].tolist() == offsets
    assert p["slot_from_src"].tolist() == sfs
    assert np.array_equal(p["src_from_slot"][p["slot_from_src"]], np.arange(len(sfs)))
