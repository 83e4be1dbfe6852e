"""End-to-end GPU parity of moe_forward against the fp64 oracle.

Small shapes: the oracle computes the whole layer.  The DeepSeek-V3 shapes
(decode T=32, skewed decode T=256, prefill T=4096, redundant experts T=1024):
the oracle computes the routing of every token and the full output of a
sample of tokens (only their experts are generated on the host), and the
launch configuration is the one bench.py times.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle
from moe_testlib import (grouped_sure, DeviceLayer, assert_close, check_topk, oracle_token_rows, parallel_router_logits,
                         to_np)
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
    sure = check_topk(r["idx"].cpu().numpy(), ref["idx"], ref["logits"], w.top_k)
    if sure.all():
        assert np.array_equal(r["counts"].cpu().numpy(), ref["counts"])
        assert np.array_equal(r["blocks"].cpu().numpy(), ref["block_counts"])
    assert_close(to_np(r["out"])[sure], ref["out"][sure], what=f"{name} out")


def test_generator_is_identical_on_cpu_and_gpu():
    w = mi.WORKLOADS["decode_t32"]
    for e in (0, 77, 255):
        for a, b in zip(mi.expert_weights(w, e), mi.expert_weights(w, e, device=DEV)):
            assert torch.equal(a, b.cpu())
    assert torch.equal(mi.hidden_states(w), mi.hidden_states(w, device=DEV).cpu())
    assert torch.equal(mi.router_weight(w), mi.router_weight(w, device=DEV).cpu())


# ----------------------------------------------------------------------------- full size

_EXPERTS_CPU = {}


@pytest.fixture(scope="module")
def dsv3_weights():
    w = mi.WORKLOADS["decode_t32"]
    return mi.stacked_expert_weights(w, device=DEV)


def _sample_tokens(T, sure, n=3):
    cand = [0, T // 3, (2 * T) // 3 + 1, T - 1]
    out = [t for t in cand if sure[t]]
    return out[:n] if out else [int(np.flatnonzero(sure)[0])]


def _check_full(w, layer, rep=None, n_sample=3):
    r = layer.forward()
    x = mi.hidden_states(w)
    wr = mi.router_weight(w)
    b = mi.router_bias(w)
    lo = parallel_router_logits(w, x, wr, b)
    idx_o, _ = oracle.topk_softmax(lo, w.top_k)
    sure = check_topk(r["idx"].cpu().numpy(), idx_o, lo, w.top_k)
    if sure.all():
        so, _ = oracle.slot_map(w, idx_o, rep)
        c_o, b_o = oracle.histogram(w, so)
        assert np.array_equal(r["counts"].cpu().numpy(), c_o)
        assert np.array_equal(r["blocks"].cpu().numpy(), b_o)
    toks = _sample_tokens(w.tokens, sure, n_sample)
    ref = oracle_token_rows(w, toks, x, wr, b, rep, _EXPERTS_CPU)
    assert_close(to_np(r["out"])[toks], ref["out"], what=f"{w.name} sampled out")
    return r


@pytest.mark.parametrize("name", ["decode_t32", "decode_t256_skew", "prefill_t4096"])
def test_forward_full_size(name, dsv3_weights):
    w = mi.WORKLOADS[name]
    layer = DeviceLayer(w, DEV, weights=dsv3_weights)
    _check_full(w, layer)


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
    r = _check_full(w, layer, rep)
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
    group-limited routing (8 groups, 4 kept): sampled tokens against the oracle."""
    w = mi.WORKLOADS["decode_t32_e1024"]
    weights = mi.stacked_expert_weights(w, device=DEV)
    layer = DeviceLayer(w, DEV, weights=weights)
    if groups is None:
        _check_full(w, layer, n_sample=2)
    else:
        T, k = w.tokens, w.top_k
        r = layer.forward_grouped(*groups)
        x, wr = mi.hidden_states(w), mi.router_weight(w)
        lo = parallel_router_logits(w, x, wr, None)
        sure, idx_o = grouped_sure(lo, k, *groups)
        assert np.array_equal(r["idx"].cpu().numpy()[sure], idx_o[sure])
        toks = _sample_tokens(T, sure, 2)
        ref = oracle_token_rows(w, toks, x, wr, None, None, _EXPERTS_CPU, groups=groups)
        assert_close(to_np(r["out"])[toks], ref["out"], what="1024 experts, group-limited, sampled out")
    del weights, layer
    torch.cuda.empty_cache()
