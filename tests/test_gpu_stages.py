"""GPU parity of each step of the layer against the fp64 oracle, through the C ABI.

Small and mid-size shapes (oracle in seconds; several tiles and ragged tails in
every dimension) for every step, plus the full DeepSeek-V3 shapes for the
integer steps, which the oracle computes in full.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle
from moe_testlib import grouped_sure as _grouped_sure, assert_close, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"

# ragged everywhere: H = 600 (9.4 K-chunks, 4.7 row blocks), I = 328, I_sh = 200
MID = mi.WORKLOADS["tiny"].with_(name="mid", tokens=100, hidden=600, inter=328, n_experts=16, top_k=4,
                                 n_shared=2, inter_shared=200, n_slots=16, n_blocks=4)
# many rows per slot: 300 rows each (two 256-row chunks, ten 32-row chunks)
DEEP = mi.WORKLOADS["tiny"].with_(name="deep", tokens=600, hidden=136, inter=264, n_experts=4, top_k=2,
                                  n_shared=1, inter_shared=72, n_slots=4, n_blocks=2)
# replicas on a small shape: 8 experts, 4 blocks of 2 + 1 replica slot
REP = mi.WORKLOADS["tiny"].with_(name="rep", tokens=64, hidden=128, inter=64, n_experts=8, top_k=2,
                                 n_shared=1, inter_shared=64, n_slots=12, n_blocks=4)
SMALL = {"tiny": mi.WORKLOADS["tiny"], "mid": MID, "deep": DEEP}
FULL = ["decode_t32", "decode_t256_skew", "decode_t256_skew_a05", "prefill_t4096", "redundant_t1024"]


def _wl(name):
    return SMALL[name] if name in SMALL else mi.WORKLOADS[name]


def _route_from_logits(w, lg):
    T, k = w.tokens, w.top_k
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    lo = torch.empty((T, w.n_experts), dtype=torch.float32, device=DEV)
    m.moe_route(w, T, None, None, None, lg.to(DEV), lo, idx, tw, None)
    assert m.moe_check_status() == 0
    return idx.cpu().numpy(), tw.cpu().numpy(), lo.cpu()


@pytest.mark.parametrize("name", ["tiny", "mid", "deep"] + FULL)
def test_topk_from_fp32_logits_is_bit_exact(name):
    w = _wl(name)
    lg = mi.fp32_logits(w)  # coarse grid: exact ties occur
    idx, tw, lo = _route_from_logits(w, lg)
    idx_o, wt_o = oracle.topk_softmax(lg.double(), w.top_k)
    assert np.array_equal(idx, idx_o)
    assert torch.equal(lo, lg)
    np.testing.assert_allclose(tw, wt_o, rtol=2e-6, atol=1e-9)


def test_topk_tie_cases():
    w = mi.WORKLOADS["tiny"].with_(tokens=3, n_experts=40, n_slots=40, n_blocks=8, top_k=5)
    lg = torch.zeros((3, 40), dtype=torch.float32)
    lg[1, [33, 2, 17, 5]] = 1.0          # equal maxima spread over lanes
    lg[2] = -torch.arange(40, dtype=torch.float32) % 3  # repeating pattern
    lg[2, 39] = -0.0
    idx, _, _ = _route_from_logits(w, lg)
    idx_o, _ = oracle.topk_softmax(lg.double(), 5)
    assert np.array_equal(idx, idx_o)
    assert list(idx[0]) == [0, 1, 2, 3, 4]
    assert list(idx[1]) == [2, 5, 17, 33, 0]


@pytest.mark.parametrize("name", ["tiny", "mid", "decode_t32", "decode_t256_skew", "prefill_t4096"])
def test_router_gemm_logits_and_topk(name):
    w = _wl(name)
    T, k = w.tokens, w.top_k
    x = mi.hidden_states(w)
    wr = mi.router_weight(w)
    b = mi.router_bias(w)
    from moe_testlib import check_topk, parallel_router_logits
    lo_o = parallel_router_logits(w, x, wr, b)
    idx_o, wt_o = oracle.topk_softmax(lo_o, k)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    lo = torch.empty((T, w.n_experts), dtype=torch.float32, device=DEV)
    ws = torch.empty(max(1, m.moe_route_workspace_size(w, T)), dtype=torch.uint8, device=DEV)
    bias = torch.from_numpy(b).to(DEV) if b is not None else None
    m.moe_route(w, T, x.to(DEV), wr.to(DEV), bias, None, lo, idx, tw, ws)
    assert m.moe_check_status() == 0
    lo = lo.cpu().numpy().astype(np.float64)
    err = np.abs(lo - lo_o).max()
    # below half the top-k gap criterion, so no token whose gap exceeds 1e-4 can flip
    assert err <= 5e-5, f"router logits max |err| {err:.3e}"
    idx = idx.cpu().numpy()
    sure = check_topk(idx, idx_o, lo_o, k)
    # combine weights: compare per expert id (order-free)
    tw = tw.cpu().numpy()
    for t in np.flatnonzero(sure):
        a = dict(zip(idx[t], tw[t]))
        for e, v in zip(idx_o[t], wt_o[t]):
            assert abs(a[e] - v) <= 1e-4 * v + 1e-7


def _oracle_idx(w):
    lg = mi.fp32_logits(w)
    return oracle.topk_softmax(lg.double(), w.top_k)


def _replica_plan(w):
    """Plan for workload w from the histogram of its non-replicated twin."""
    if w.n_slots == w.n_experts:
        return None
    base = w.with_(n_slots=w.n_experts)
    idx, _ = _oracle_idx(base)
    counts = np.bincount(idx.ravel(), minlength=w.n_experts)
    return oracle.plan_replicas(w, counts, w.n_slots - w.n_experts)


def _gpu_dispatch(w, x_dev, idx, replica_of):
    r = _gpu_dispatch_raw(w, x_dev, idx, replica_of)
    assert m.moe_check_status() == 0, m.last_error()
    return r


def _gpu_dispatch_raw(w, x_dev, idx, replica_of):
    T, k, S = w.tokens, w.top_k, w.n_slots
    n = T * k
    t32 = dict(dtype=torch.int32, device=DEV)
    r = dict(slot_of=torch.empty(n, **t32), counts=torch.empty(S + 1, **t32),
             blocks=torch.empty(w.n_blocks, **t32), offsets=torch.empty(S + 2, **t32),
             perm=torch.empty(n, **t32), inv=torch.empty(n, **t32),
             x_disp=torch.empty((n, w.hidden), dtype=torch.bfloat16, device=DEV))
    rep = torch.from_numpy(np.asarray(replica_of, np.int32)).to(DEV) if replica_of is not None else None
    m.moe_dispatch(w, T, x_dev, torch.from_numpy(np.ascontiguousarray(idx, np.int32)).to(DEV), rep,
                   r["slot_of"], r["counts"], r["blocks"], r["offsets"], r["perm"], r["inv"], r["x_disp"])
    return r


@pytest.mark.parametrize("name", ["tiny", "mid", "deep", "rep"] + FULL)
def test_dispatch_is_bit_exact(name):
    w = REP if name == "rep" else _wl(name)
    rep = _replica_plan(w) if name in ("rep", "redundant_t1024") else None
    idx, _ = _oracle_idx(w)
    x = mi.hidden_states(w)
    g = _gpu_dispatch(w, x.to(DEV), idx, rep)
    so, inv_cnt = oracle.slot_map(w, idx, rep)
    assert inv_cnt == 0
    counts, blocks = oracle.histogram(w, so)
    small = w.tokens <= 1024
    offsets, perm, inv, xd = oracle.dispatch(w, w.tokens, so, counts, x if small else None)
    assert np.array_equal(g["slot_of"].cpu().numpy(), so)
    assert np.array_equal(g["counts"].cpu().numpy(), counts)
    assert np.array_equal(g["blocks"].cpu().numpy(), blocks)
    assert np.array_equal(g["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(g["perm"].cpu().numpy(), perm)
    assert np.array_equal(g["inv"].cpu().numpy(), inv)
    xg = g["x_disp"].cpu().view(torch.int16).numpy().view(np.uint16)
    assert xg.nbytes == w.tokens * w.top_k * w.hidden * 2
    if small:
        assert np.array_equal(xg, xd)
    else:
        xs = x.view(torch.int16).numpy().view(np.uint16)
        rows = np.random.default_rng(0).choice(w.tokens * w.top_k, 2048, replace=False)
        assert np.array_equal(xg[rows], xs[perm[rows] // w.top_k])


# the chunked index pass (4096 assignments and more): exactly at the threshold,
# a ragged last chunk, and the 128-chunk cap (65600 assignments, 513 per chunk)
# with replicas and out-of-range ids planted across chunk boundaries
CHUNKED = {
    "n4096": mi.WORKLOADS["tiny"].with_(name="n4096", tokens=512, hidden=16, n_experts=64, n_slots=64, top_k=8),
    "n4104": mi.WORKLOADS["tiny"].with_(name="n4104", tokens=513, hidden=16, n_experts=64, n_slots=64, top_k=8),
    "n65600": mi.WORKLOADS["tiny"].with_(name="n65600", tokens=8200, hidden=16, n_experts=256, n_slots=264,
                                         n_blocks=8, top_k=8),
}


@pytest.mark.parametrize("name", sorted(CHUNKED))
def test_chunked_index_pass_is_bit_exact(name):
    w = CHUNKED[name]
    T, k = w.tokens, w.top_k
    rep = None
    if w.n_slots > w.n_experts:
        rep = oracle.plan_replicas(w, np.arange(w.n_experts)[::-1].copy(), w.n_slots - w.n_experts)
    idx, _ = oracle.topk_softmax(mi.fp32_logits(w).double(), k)
    idx = idx.copy()
    bad = [(0, 0), (63, 7), (64, 0), (T // 2, 3), (T - 1, k - 1)]  # chunk edges at multiples of 512 / k tokens
    for t, j in bad:
        idx[t, j] = w.n_experts + t % 3 if t % 2 else -1 - t
    x = mi.hidden_states(w)
    assert m.moe_dispatch_workspace_size(w, T) > 0
    g = _gpu_dispatch_raw(w, x.to(DEV), idx, rep)
    assert m.moe_check_status() == m.MOE_ERR_DEVICE_STATUS  # the planted ids
    so, n_bad = oracle.slot_map(w, idx, rep)
    assert n_bad == len(bad)
    counts, blocks = oracle.histogram(w, so)
    offsets, perm, inv, xd = oracle.dispatch(w, T, so, counts, x)
    assert np.array_equal(g["slot_of"].cpu().numpy(), so)
    assert np.array_equal(g["counts"].cpu().numpy(), counts)
    assert np.array_equal(g["blocks"].cpu().numpy(), blocks)
    assert np.array_equal(g["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(g["perm"].cpu().numpy(), perm)
    assert np.array_equal(g["inv"].cpu().numpy(), inv)
    assert np.array_equal(g["x_disp"].cpu().view(torch.int16).numpy().view(np.uint16), xd)


@pytest.mark.parametrize("name", ["tiny", "rep", "decode_t256_skew", "redundant_t1024"])
def test_expert_histogram_is_bit_exact(name):
    w = REP if name == "rep" else _wl(name)
    rep = _replica_plan(w) if name in ("rep", "redundant_t1024") else None
    idx, _ = _oracle_idx(w)
    counts = torch.empty(w.n_slots + 1, dtype=torch.int32, device=DEV)
    blocks = torch.empty(w.n_blocks, dtype=torch.int32, device=DEV)
    repd = torch.from_numpy(rep).to(DEV) if rep is not None else None
    m.moe_expert_histogram(w, w.tokens, torch.from_numpy(idx).to(DEV), repd, counts, blocks)
    assert m.moe_check_status() == 0
    so, _ = oracle.slot_map(w, idx, rep)
    c_o, b_o = oracle.histogram(w, so)
    assert np.array_equal(counts.cpu().numpy(), c_o)
    assert np.array_equal(blocks.cpu().numpy(), b_o)
    assert int(counts.sum()) == w.tokens * w.top_k


def test_invalid_expert_ids_are_counted_and_flagged():
    w = mi.WORKLOADS["tiny"]
    idx, _ = _oracle_idx(w)
    idx = idx.copy()
    idx[3, 1] = w.n_experts
    idx[7, 0] = -5
    counts = torch.empty(w.n_slots + 1, dtype=torch.int32, device=DEV)
    m.moe_expert_histogram(w, w.tokens, torch.from_numpy(idx).to(DEV), None, counts, None)
    assert m.moe_check_status() == m.MOE_ERR_DEVICE_STATUS
    assert m.moe_check_status() == 0  # cleared by the read
    so, bad = oracle.slot_map(w, idx)
    c_o, _ = oracle.histogram(w, so)
    assert bad == 2 and np.array_equal(counts.cpu().numpy(), c_o)


@pytest.mark.parametrize("mode", [m.MOE_FFN_DECODE, m.MOE_FFN_PREFILL])
@pytest.mark.parametrize("name", ["tiny", "mid", "deep", "rep"])
def test_expert_ffn_matches_oracle(name, mode):
    w = REP if name == "rep" else _wl(name)
    rep = _replica_plan(w) if name == "rep" else None
    T, k = w.tokens, w.top_k
    idx, _ = _oracle_idx(w)
    x = mi.hidden_states(w)
    wg, wu, wd = mi.stacked_expert_weights(w, rep)
    sg, su, sd = mi.stacked_shared_weights(w)
    g = _gpu_dispatch(w, x.to(DEV), idx, rep)
    n = T * k
    y_disp = torch.empty((n, w.hidden), dtype=torch.bfloat16, device=DEV)
    y_sh = torch.empty((T, w.hidden), dtype=torch.float32, device=DEV)
    ws = torch.empty(m.moe_ffn_workspace_size(w, T), dtype=torch.uint8, device=DEV)
    m.moe_expert_ffn(w, T, x.to(DEV), g["x_disp"], g["offsets"], wg.to(DEV), wu.to(DEV), wd.to(DEV),
                     sg.to(DEV), su.to(DEV), sd.to(DEV), y_disp, y_sh, mode, ws)
    assert m.moe_check_status() == 0, m.last_error()
    so, _ = oracle.slot_map(w, idx, rep)
    counts, _ = oracle.histogram(w, so)
    offsets, perm, inv, xd = oracle.dispatch(w, T, so, counts, x)
    y_o = oracle.expert_ffn(w, T, offsets, xd, wg, wu, wd)
    assert_close(to_np(y_disp), y_o, what="y_disp")
    ysh_o = oracle.shared_rows(w, x, sg, su, sd)
    assert_close(to_np(y_sh), ysh_o, what="y_shared", bf16_out=False)


def test_gate_up_and_down_entry_points_compose_to_ffn():
    w = MID
    T, k = w.tokens, w.top_k
    idx, _ = _oracle_idx(w)
    x = mi.hidden_states(w).to(DEV)
    wg, wu, wd = [t.to(DEV) for t in mi.stacked_expert_weights(w)]
    sg, su, sd = [t.to(DEV) for t in mi.stacked_shared_weights(w)]
    g = _gpu_dispatch(w, x, idx, None)
    n = T * k
    h = torch.empty((n, w.inter), dtype=torch.bfloat16, device=DEV)
    hs = torch.empty((T, w.n_shared * w.inter_shared), dtype=torch.bfloat16, device=DEV)
    y1 = torch.empty((n, w.hidden), dtype=torch.bfloat16, device=DEV)
    ys1 = torch.empty((T, w.hidden), dtype=torch.float32, device=DEV)
    m.moe_expert_gate_up(w, T, x, g["x_disp"], g["offsets"], wg, wu, sg, su, h, hs)
    m.moe_expert_down(w, T, h, hs, g["offsets"], wd, sd, y1, ys1)
    y2 = torch.empty_like(y1)
    ys2 = torch.empty_like(ys1)
    ws = torch.empty(m.moe_ffn_workspace_size(w, T), dtype=torch.uint8, device=DEV)
    m.moe_expert_ffn(w, T, x, g["x_disp"], g["offsets"], wg, wu, wd, sg, su, sd, y2, ys2, m.MOE_FFN_AUTO, ws)
    assert m.moe_check_status() == 0
    assert torch.equal(y1, y2) and torch.equal(ys1, ys2)


@pytest.mark.parametrize("name", ["tiny", "mid", "decode_t32", "decode_t256_skew"])
def test_combine_matches_oracle(name):
    w = _wl(name)
    T, k, H = w.tokens, w.top_k, w.hidden
    idx, wt = _oracle_idx(w)
    so, _ = oracle.slot_map(w, idx)
    counts, _ = oracle.histogram(w, so)
    _, _, inv, _ = oracle.dispatch(w, T, so, counts, None)
    y = mi.normal_bf16((T * k, H), 1.0, 7, 100)
    ysh = mi.normal_bf16((T, H), 1.0, 7, 101).float()
    wt32 = wt.astype(np.float32)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    m.moe_combine(w, T, y.to(DEV), torch.from_numpy(inv).to(DEV), torch.from_numpy(wt32).to(DEV), ysh.to(DEV), out)
    assert m.moe_check_status() == 0
    ref = oracle.combine(w, T, y.double().numpy(), inv, wt32.astype(np.float64), ysh.double().numpy())
    assert_close(to_np(out), ref, what="combine")


# ----------------------------------------------------------------------------- group-limited routing

GROUPED = [("tiny", 4, 2), ("mid", 4, 2), ("deep", 2, 1), ("decode_t32", 8, 4), ("decode_t256_skew", 8, 2),
           ("prefill_t4096", 8, 3)]


@pytest.mark.parametrize("name,G,Gk", GROUPED)
def test_grouped_topk_from_fp32_logits_is_bit_exact(name, G, Gk):
    w = _wl(name)
    T, k = w.tokens, w.top_k
    lg = mi.fp32_logits(w)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    m.moe_route_grouped(w, T, G, Gk, None, None, None, lg.to(DEV), None, idx, tw, None)
    assert m.moe_check_status() == 0
    idx_o, wt_o = oracle.topk_grouped(lg.double(), k, G, Gk)
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    np.testing.assert_allclose(tw.cpu().numpy(), wt_o, rtol=2e-6, atol=1e-9)
    gs = w.n_experts // G
    assert all(len({int(e) // gs for e in row}) <= Gk for row in idx_o)


@pytest.mark.parametrize("name,G,Gk", [("mid", 4, 2), ("decode_t32", 8, 4), ("prefill_t4096", 8, 3)])
def test_grouped_routing_from_router_gemm(name, G, Gk):
    w = _wl(name)
    T, k = w.tokens, w.top_k
    from moe_testlib import parallel_router_logits
    x, wr = mi.hidden_states(w), mi.router_weight(w)
    lo_o = parallel_router_logits(w, x, wr, None)
    sure, idx_o = _grouped_sure(lo_o, k, G, Gk)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    ws = torch.empty(max(1, m.moe_route_workspace_size(w, T)), dtype=torch.uint8, device=DEV)
    m.moe_route_grouped(w, T, G, Gk, x.to(DEV), wr.to(DEV), None, None, None, idx, tw, ws)
    assert m.moe_check_status() == 0
    got = np.sort(idx.cpu().numpy(), 1)
    assert sure.mean() > 0.9
    assert np.array_equal(got[sure], np.sort(idx_o, 1)[sure])


def test_grouped_routing_layer_matches_oracle():
    """Staged layer (grouped route, dispatch, FFN, combine) against the oracle's pieces."""
    w = MID
    G, Gk = 4, 2
    T, k, H = w.tokens, w.top_k, w.hidden
    x, wr = mi.hidden_states(w), mi.router_weight(w)
    wg, wu, wd = mi.stacked_expert_weights(w)
    sg, su, sd = mi.stacked_shared_weights(w)
    lo = oracle.router_logits(w, x, wr, None)
    sure, _ = _grouped_sure(lo, k, G, Gk)
    idx_o, wt_o = oracle.topk_grouped(lo, k, G, Gk)
    so, _ = oracle.slot_map(w, idx_o)
    cnt, _ = oracle.histogram(w, so)
    off, perm, inv, xd = oracle.dispatch(w, T, so, cnt, x)
    y_o = oracle.expert_ffn(w, T, off, xd, wg, wu, wd)
    ref = oracle.combine(w, T, y_o, inv, wt_o, oracle.shared_rows(w, x, sg, su, sd))
    d = dict(x=x.to(DEV), wr=wr.to(DEV), wg=wg.to(DEV), wu=wu.to(DEV), wd=wd.to(DEV), sg=sg.to(DEV),
             su=su.to(DEV), sd=sd.to(DEV))
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    ws = torch.empty(max(1, m.moe_route_workspace_size(w, T)), dtype=torch.uint8, device=DEV)
    m.moe_route_grouped(w, T, G, Gk, d["x"], d["wr"], None, None, None, idx, tw, ws)
    g = _gpu_dispatch(w, d["x"], idx.cpu().numpy(), None)
    y = torch.empty((T * k, H), dtype=torch.bfloat16, device=DEV)
    ysh = torch.empty((T, H), dtype=torch.float32, device=DEV)
    fws = torch.empty(m.moe_ffn_workspace_size(w, T), dtype=torch.uint8, device=DEV)
    m.moe_expert_ffn(w, T, d["x"], g["x_disp"], g["offsets"], d["wg"], d["wu"], d["wd"], d["sg"], d["su"], d["sd"],
                     y, ysh, m.MOE_FFN_AUTO, fws)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    m.moe_combine(w, T, y, g["inv"], tw, ysh, out)
    assert m.moe_check_status() == 0
    assert np.array_equal(np.sort(idx.cpu().numpy(), 1)[sure], np.sort(idx_o, 1)[sure])
    assert_close(to_np(out)[sure], ref[sure], what="grouped layer")
