"""Online EPLB loop on the GPU (section 6.2 of the expert-parallelism post):
the sliding-window monitor against the oracle, and a replica migration that
never changes the layer's output."""
import numpy as np
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle
from moe_testlib import DeviceLayer
from test_gpu_stages import REP

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _random_histograms(w, n, rep, seed):
    rng = np.random.default_rng(seed)
    hist = []
    for b in range(n):
        # skew that moves between batches: expert e drawn with weight depending on b
        p = np.exp(-0.3 * ((np.arange(w.n_experts) - 5 * b) % w.n_experts))
        p /= p.sum()
        idx = np.stack([rng.choice(w.n_experts, w.top_k, replace=False, p=p) for _ in range(w.tokens)])
        so, _ = oracle.slot_map(w, idx.astype(np.int32), rep)
        c, _ = oracle.histogram(w, so)
        hist.append(c)
    return np.array(hist, dtype=np.int32)


@pytest.mark.parametrize("name,window", [("rep", 3), ("redundant_t1024", 4), ("decode_t256_skew", 1)])
def test_window_push_matches_oracle(name, window):
    w = REP if name == "rep" else mi.WORKLOADS[name]
    rep = None
    if w.n_slots > w.n_experts:
        rep = oracle.plan_replicas(w, np.arange(w.n_experts)[::-1].copy(), w.n_slots - w.n_experts)
    hist = _random_histograms(w, 7, rep, seed=hash(name) % 1000)
    state = torch.empty(m.moe_eplb_window_bytes(w, window), dtype=torch.uint8, device=DEV)
    m.moe_eplb_window_reset(w, window, state)
    bl = torch.empty(w.n_blocks, dtype=torch.int64, device=DEV)
    el = torch.empty(w.n_experts, dtype=torch.int64, device=DEV)
    ratio = torch.empty(1, dtype=torch.float64, device=DEV)
    trig = torch.empty(1, dtype=torch.int32, device=DEV)
    repd = torch.from_numpy(rep).to(DEV) if rep is not None else None
    for i in range(len(hist)):
        m.moe_eplb_window_push(w, window, state, torch.from_numpy(hist[i]).to(DEV), repd, 1.2, bl, el, ratio, trig)
        _, bl_o, el_o, ratio_o, trig_o = oracle.eplb_window(w, hist[:i + 1], window, rep, 1.2)
        assert np.array_equal(bl.cpu().numpy(), bl_o)
        assert np.array_equal(el.cpu().numpy(), el_o)
        assert ratio.item() == ratio_o  # same double expression on both sides
        assert bool(trig.item()) == trig_o
    assert m.moe_check_status() == 0


def test_window_fed_by_the_forward_pass():
    w = mi.WORKLOADS["decode_t256_skew"].with_(n_experts=16, n_slots=16, n_blocks=4, hidden=256, inter=128,
                                               inter_shared=128, tokens=64)
    layer = DeviceLayer(w, DEV)
    state = torch.empty(m.moe_eplb_window_bytes(w, 2), dtype=torch.uint8, device=DEV)
    m.moe_eplb_window_reset(w, 2, state)
    bl = torch.empty(w.n_blocks, dtype=torch.int64, device=DEV)
    ratio = torch.empty(1, dtype=torch.float64, device=DEV)
    r = layer.forward()
    m.moe_eplb_window_push(w, 2, state, r["counts"], None, 1.2, bl, None, ratio, None)
    m.moe_eplb_window_push(w, 2, state, r["counts"], None, 1.2, bl, None, ratio, None)
    blocks = r["blocks"].cpu().numpy().astype(np.int64)
    assert np.array_equal(bl.cpu().numpy(), 2 * blocks)
    assert ratio.item() == m.moe_eplb_imbalance(blocks)
    assert ratio.item() > 1.2  # the skew bias concentrates load in a few blocks


def _migrate_and_check(w, weights_plain, plan_a, plan_b):
    """Serve batches with plan A, migrate to plan B while serving, serve with B; outputs never change."""
    se_a = torch.from_numpy(mi.slot_experts(w, plan_a)).to(DEV)
    wg, wu, wd = (t.index_select(0, se_a.clamp(min=0)) for t in weights_plain)
    plain = DeviceLayer(w.with_(n_slots=w.n_experts), DEV, weights=weights_plain)
    ref = plain.forward()["out"].clone()
    layer = DeviceLayer(w, DEV, replica_of=plan_a, weights=(wg, wu, wd))
    tables = {}

    def run(table):
        layer.replica_of = torch.from_numpy(np.ascontiguousarray(table, np.int32)).to(DEV)
        r = layer.forward()
        assert torch.equal(r["out"], ref), "layer output changed"
        return r

    r_a = run(plan_a)
    stable = m.moe_eplb_stable_table(w, plan_a, plan_b)
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    ev_old_done = torch.cuda.Event()
    ev_old_done.record(compute)
    with torch.cuda.stream(copy):
        copy.wait_event(ev_old_done)
        m.moe_eplb_copy_replicas(w, plan_a, plan_b, wg, wu, wd, stream=copy)
        ev_copied = torch.cuda.Event()
        ev_copied.record(copy)
    run(stable)           # served while the copies run
    compute.wait_event(ev_copied)
    r_b = run(plan_b)
    # replica slots of plan B now hold their experts' weights
    for e in np.flatnonzero(plan_b >= 0):
        home = oracle.home_slot(w, int(e))
        assert torch.equal(wd[int(plan_b[e])], wd[home]) and torch.equal(wg[int(plan_b[e])], wg[home])
    # with plan B, odd tokens of a replicated expert land in its new replica slot, even ones at home
    c_b = r_b["counts"].cpu().numpy()
    idx = r_b["idx"].cpu().numpy()
    odd = np.zeros(w.n_experts, np.int64)
    even = np.zeros(w.n_experts, np.int64)
    for t in range(w.tokens):
        for e in idx[t]:
            (odd if t % 2 else even)[e] += 1
    for e in np.flatnonzero(plan_b >= 0):
        assert c_b[plan_b[e]] == odd[e] and c_b[oracle.home_slot(w, int(e))] == even[e]
    assert r_a["counts"].sum() == r_b["counts"].sum()
    assert m.moe_check_status() == 0
    return wg, wu, wd


def test_migration_keeps_the_output_small():
    w = REP.with_(tokens=128)
    base = w.with_(n_slots=w.n_experts)
    weights = mi.stacked_expert_weights(base, device=DEV)
    plan_a = oracle.plan_replicas(w, np.array([9, 1, 7, 0, 3, 3, 8, 2]), 4)
    plan_b = oracle.plan_replicas(w, np.array([0, 9, 1, 8, 7, 3, 2, 6]), 4)
    assert not np.array_equal(plan_a, plan_b)
    _migrate_and_check(w, weights, plan_a, plan_b)


def test_migration_keeps_the_output_dsv3():
    w = mi.WORKLOADS["redundant_t1024"]
    weights = mi.stacked_expert_weights(w.with_(n_slots=w.n_experts), device=DEV)
    counts_a = np.bincount(np.arange(256) % 37, minlength=256)[:256] + np.arange(256)
    plan_a = oracle.plan_replicas(w, counts_a, 8)
    plan_b = oracle.plan_replicas(w, counts_a[::-1].copy(), 8)
    out = _migrate_and_check(w, weights, plan_a, plan_b)
    del out, weights
    torch.cuda.empty_cache()
