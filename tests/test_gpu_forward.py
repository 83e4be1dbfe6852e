"""End-to-end GPU parity of moe_forward against the fp64 oracle.

Small shapes: the oracle computes the whole layer.  The DeepSeek-V3 shapes
(decode T=32, skewed decode T=256, prefill T=4096, redundant experts T=1024):
the oracle computes the routing of every token and the full output of 256
seeded random tokens (every token at T=32), and the launch configuration is
the one bench.py times.  Per-slot counts and block loads are checked on every
call against the oracle's histogram of the GPU's own selection.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle
from moe_testlib import (SAMPLE_TOKENS, DeviceLayer, assert_close, check_counts_of_routing, check_full_size_layer,
                         check_topk, grouped_sure, oracle_sampled_layer, parallel_router_logits, sample_tokens, to_np)
from test_gpu_stages import DEEP, MID, REP

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _small_case(name):
    return {"tiny": mi.WORKLOADS["tiny"], "mid": MID, "deep": DEEP, "rep": REP}[name]


def _small_replica_plan(w):
    base = w.with_(n_slots=w.n_experts)
    x = mi.hidden_states(base)
    lo = oracle.router_logits(base, x, mi.router_weight(base), mi.router_bias(base))
    idx, _ = oracle.topk_softmax(lo, base.top_k)
    return oracle.plan_replicas(w, np.bincount(idx.ravel(), minlength=w.n_experts), w.n_slots - w.n_experts)


@pytest.mark.parametrize("mode", [m.MOE_FFN_AUTO, m.MOE_FFN_DECODE, m.MOE_FFN_PREFILL])
@pytest.mark.parametrize("name", ["tiny", "mid", "deep", "rep"])
def test_forward_small_matches_oracle(name, mode):
    w = _small_case(name)
    rep = _small_replica_plan(w) if name == "rep" else None
    x = mi.hidden_states(w)
    wr = mi.router_weight(w)
    b = mi.router_bias(w)
    wg, wu, wd = mi.stacked_expert_weights(w, rep)
    sg, su, sd = mi.stacked_shared_weights(w)
    ref = oracle.moe_forward(w, x, wr, b, rep, wg, wu, wd, sg, su, sd)
    layer = DeviceLayer(w, DEV, replica_of=rep)
    r = layer.forward(mode)
    idx_g = r["idx"].cpu().numpy()
    sure = check_topk(idx_g, ref["idx"], ref["logits"], w.top_k)
    check_counts_of_routing(w, idx_g, r["counts"].cpu().numpy(), r["blocks"].cpu().numpy(), rep, ref["idx"], sure)
    assert_close(to_np(r["out"])[sure], ref["out"][sure], what=f"{name} out")


def test_generator_is_identical_on_cpu_and_gpu():
    w = mi.WORKLOADS["decode_t32"]
    for e in (0, 77, 255):
        for a, b in zip(mi.expert_weights(w, e), mi.expert_weights(w, e, device=DEV)):
            assert torch.equal(a, b.cpu())
    assert torch.equal(mi.hidden_states(w), mi.hidden_states(w, device=DEV).cpu())
    assert torch.equal(mi.router_weight(w), mi.router_weight(w, device=DEV).cpu())


# ----------------------------------------------------------------------------- full size


@pytest.fixture(scope="module")
def dsv3_weights():
    w = mi.WORKLOADS["decode_t32"]
    return mi.stacked_expert_weights(w, device=DEV)


def test_generator_rows_of_every_expert_match_on_cpu_and_gpu(dsv3_weights):
    """The full-size parity tests give the oracle the generator's expert
    weights as generated on the device (regenerating 22.5 GB on the host would
    take minutes): two seeded rows of every expert matrix regenerated on the
    host match the device copies bit for bit."""
    w = mi.WORKLOADS["decode_t32"]
    H, I = w.hidden, w.inter
    rng = np.random.Generator(np.random.PCG64(5))
    wg, wu, wd = dsv3_weights
    for e in range(w.n_experts):
        for t, tid, rows, cols, fan in ((wg, mi.TID_GATE, I, H, H), (wu, mi.TID_UP, I, H, H),
                                        (wd, mi.TID_DOWN, H, I, I)):
            for r in rng.integers(0, rows, 2):
                host = mi.normal_bf16((cols,), 1.0 / np.sqrt(fan), w.seed, tid, e, offset=int(r) * cols)
                assert torch.equal(t[e, int(r)].cpu(), host), (e, tid, int(r))


def _host_experts(weights):
    """expert_host(e) for the oracle: logical expert e's matrices copied from the
    device stack of the 256 experts (slot e holds expert e there)."""
    return lambda e: tuple(t[e].cpu() for t in weights)


def _check_full(w, r, weights, rep=None, n_sample=SAMPLE_TOKENS):
    sh = mi.stacked_shared_weights(w)
    return check_full_size_layer(w, to_np(r["out"]), r["idx"].cpu().numpy(), r["counts"].cpu().numpy(),
                                 r["blocks"].cpu().numpy(), _host_experts(weights), sh, rep=rep,
                                 n_sample=n_sample)


@pytest.mark.parametrize("name", ["decode_t32", "decode_t256_skew", "decode_t256_skew_a05", "prefill_t4096"])
def test_forward_full_size(name, dsv3_weights):
    """The layer at the bench's launch configuration: every token's routing,
    the counts of the GPU's own routing, and 256 seeded random tokens' outputs
    (all 32 at T=32) element by element against the oracle."""
    w = mi.WORKLOADS[name]
    layer = DeviceLayer(w, DEV, weights=dsv3_weights)
    _check_full(w, layer.forward(), dsv3_weights)


def test_redundant_experts_full_size(dsv3_weights):
    # plan from the skewed decode batch's histogram (oracle routing)
    src = mi.WORKLOADS[mi.REPLICA_PLAN_SOURCE]
    lo = parallel_router_logits(src, mi.hidden_states(src), mi.router_weight(src), mi.router_bias(src))
    idx_src, _ = oracle.topk_softmax(lo, src.top_k)
    w = mi.WORKLOADS["redundant_t1024"]
    rep = oracle.plan_replicas(w, np.bincount(idx_src.ravel(), minlength=w.n_experts), mi.N_REPLICAS)
    # the library's host planner gives the same map from the same counts
    assert np.array_equal(m.moe_eplb_plan_replicas(w, np.bincount(idx_src.ravel(), minlength=w.n_experts),
                                                   mi.N_REPLICAS), rep)
    se = torch.from_numpy(mi.slot_experts(w, rep)).to(DEV)
    assert int((se < 0).sum()) == 0
    weights = tuple(t.index_select(0, se) for t in dsv3_weights)
    layer = DeviceLayer(w, DEV, replica_of=rep, weights=weights)
    r = layer.forward()
    _check_full(w, r, dsv3_weights, rep)
    c = r["counts"].cpu().numpy()
    assert c.sum() == w.tokens * w.top_k and c[-1] == 0
    # the replicated layer gives the non-replicated layer's output
    plain = DeviceLayer(w.with_(n_slots=w.n_experts), DEV, weights=dsv3_weights)
    r0 = plain.forward()
    assert torch.equal(r["idx"], r0["idx"])
    diff = (r["out"].float() - r0["out"].float()).abs().max().item()
    assert diff == 0.0, f"replicated vs plain layer differ by {diff}"
    del weights
    torch.cuda.empty_cache()


@pytest.mark.parametrize("groups", [None, (8, 4)])
def test_forward_full_size_1024_experts(groups):
    """1024 experts of the DeepSeek-V3 shape (90 GB of bf16 weights), plain and
    group-limited routing (8 groups, 4 kept): every token of the batch against
    the oracle."""
    w = mi.WORKLOADS["decode_t32_e1024"]
    weights = mi.stacked_expert_weights(w, device=DEV)
    layer = DeviceLayer(w, DEV, weights=weights)
    if groups is None:
        _check_full(w, layer.forward(), weights)
    else:
        k = w.top_k
        r = layer.forward_grouped(*groups)
        x, wr = mi.hidden_states(w), mi.router_weight(w)
        lo = parallel_router_logits(w, x, wr, None)
        sure, idx_o = grouped_sure(lo, k, *groups)
        idx_g = r["idx"].cpu().numpy()
        assert np.array_equal(idx_g[sure], idx_o[sure])
        check_counts_of_routing(w, idx_g, r["counts"].cpu().numpy(), r["blocks"].cpu().numpy())
        _, wt_o = oracle.topk_grouped(lo, k, *groups)
        toks = sample_tokens(sure)
        ref = oracle_sampled_layer(w, toks, x, idx_o, wt_o, _host_experts(weights), mi.stacked_shared_weights(w))
        assert_close(to_np(r["out"])[toks], ref, what="1024 experts, group-limited")
    del weights, layer
    torch.cuda.empty_cache()
