"""Seeded random layer shapes on the GPU against the fp64 oracle.

The other parity tests use hand-picked shapes; these draw the hidden size,
the intermediate sizes, the expert and block counts, top-k, the shared
experts, the batch size and the routing skew at random (with the ABI's own
constraints: multiples of 16 for one-byte rows), and run the bf16 and the
E4M3 layer in every token-chunk mode; some cases add replica slots (one or two
per block, planned from the plain layer's histogram).  Ragged tails in every
GEMM dimension, output halves that end inside a 128-row block, expert groups
of one and many token chunks, and batches of a single token all come up."""
import numpy as np
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle
from moe_testlib import (DeviceLayer, assert_close, check_counts_of_routing, check_topk, fp8_layer_allowance,
                         to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"
N_CASES = 16


def _case(i):
    rng = np.random.default_rng([20261203, i])
    E = int(rng.choice([1, 2, 4, 8, 16, 32, 48, 64]))
    B = int(rng.choice([b for b in (1, 2, 4, 8) if E % b == 0]))
    k = int(rng.integers(1, min(E, 8) + 1))
    n_sh = int(rng.integers(0, 3))
    w = mi.WORKLOADS["tiny"].with_(
        name=f"fuzz{i}", tokens=int(rng.integers(1, 301)), hidden=16 * int(rng.integers(2, 65)),
        inter=16 * int(rng.integers(1, 33)), n_experts=E, n_slots=E, n_blocks=B, top_k=k, n_shared=n_sh,
        inter_shared=16 * int(rng.integers(1, 17)), skew_alpha=float(rng.choice([0.0, 0.5, 1.5])), seed=i + 1)
    # replica slots in some cases: rb per block, planned from the plain twin's histogram
    rb = int(rng.choice([0, 0, 1, 2]))
    if rb and B * rb <= E:
        w = w.with_(n_slots=E + B * rb)
    return w


def _plan(w):
    if w.n_slots == w.n_experts:
        return None
    base = w.with_(n_slots=w.n_experts)
    lo = oracle.router_logits(base, mi.hidden_states(base), mi.router_weight(base), mi.router_bias(base))
    idx, _ = oracle.topk_softmax(lo, base.top_k)
    return oracle.plan_replicas(w, np.bincount(idx.ravel(), minlength=w.n_experts), w.n_slots - w.n_experts)


CASES = [_case(i) for i in range(N_CASES)]
MODES = [m.MOE_FFN_DECODE, m.MOE_FFN_PREFILL, m.MOE_FFN_AUTO]


def _shared(w):
    if w.n_shared:
        return mi.stacked_shared_weights(w)
    z = torch.zeros((0, w.inter_shared, w.hidden), dtype=torch.bfloat16)
    return z, z, torch.zeros((0, w.hidden, w.inter_shared), dtype=torch.bfloat16)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_bf16_layer_matches_oracle(i, mode):
    w = CASES[i]
    rep = _plan(w)
    x, wr, b = mi.hidden_states(w), mi.router_weight(w), mi.router_bias(w)
    wg, wu, wd = mi.stacked_expert_weights(w, rep)
    sg, su, sd = _shared(w)
    ref = oracle.moe_forward(w, x, wr, b, rep, wg, wu, wd, sg, su, sd)
    layer = DeviceLayer(w, DEV, replica_of=rep, weights=tuple(t.to(DEV) for t in (wg, wu, wd)))
    r = layer.forward(mode)
    idx_g = r["idx"].cpu().numpy()
    sure = check_topk(idx_g, ref["idx"], ref["logits"], w.top_k)
    check_counts_of_routing(w, idx_g, r["counts"].cpu().numpy(), r["blocks"].cpu().numpy(), rep, ref["idx"], sure)
    assert_close(to_np(r["out"])[sure], ref["out"][sure], what=f"{w.name} {w}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_e4m3_layer_matches_fp8_oracle(i, mode):
    w = CASES[i]
    T, H = w.tokens, w.hidden
    rep = _plan(w)
    x, wr, b = mi.hidden_states(w), mi.router_weight(w), mi.router_bias(w)
    wg, wu, wd = mi.stacked_expert_weights(w, rep)
    sg, su, sd = mi.stacked_shared_weights(w) if w.n_shared else (None, None, None)
    q = oracle.quantize_layer_fp8(w, wg, wu, wd, sg, su, sd)
    ref = oracle.moe_forward_fp8(w, x, wr, b, rep, q)
    d = {k_: torch.from_numpy(np.ascontiguousarray(v)).to(DEV) for k_, v in q.items()}
    if not w.n_shared:
        for k_ in ("qsg", "ssg", "qsu", "ssu", "qsd", "ssd"):
            d[k_] = None
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device=DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    counts, blocks = torch.empty(w.n_slots + 1, **i32), torch.empty(w.n_blocks, **i32)
    ws = torch.empty(max(16, m.moe_workspace_size_fp8(w, T)), dtype=torch.uint8, device=DEV)
    bd = torch.from_numpy(b).to(DEV) if b is not None else None
    repd = torch.from_numpy(np.asarray(rep, dtype=np.int32)).to(DEV) if rep is not None else None
    m.moe_forward_fp8(w, T, x.to(DEV), wr.to(DEV), bd, repd, d["qg"], d["sg"], d["qu"], d["su"], d["qd"], d["sd"],
                      d["qsg"], d["ssg"], d["qsu"], d["ssu"], d["qsd"], d["ssd"], out, topk_idx_out=idx,
                      counts_out=counts, block_counts_out=blocks, mode=mode, ws=ws)
    assert m.moe_check_status() == 0, m.last_error()
    lo = oracle.router_logits(w, x, wr, b)
    idx_g = idx.cpu().numpy()
    sure = check_topk(idx_g, ref["idx"], lo, w.top_k)
    check_counts_of_routing(w, idx_g, counts.cpu().numpy(), blocks.cpu().numpy(), rep, ref["idx"], sure)
    assert_close(to_np(out)[sure], ref["out"][sure], what=f"{w.name} E4M3 {w}", e4m3_layer=True,
                 allowance=fp8_layer_allowance(w, ref)[sure])
