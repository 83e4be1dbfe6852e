"""Degenerate and limit cases of the layer on the GPU against the fp64 oracle:
one token, every expert selected, a single expert, no shared expert, the
largest expert/slot counts and top-k the library accepts, an empty batch, and
out-of-range expert ids reaching dispatch."""
import numpy as np
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle
from moe_testlib import DeviceLayer, assert_close, check_counts_of_routing, check_topk, fp8_layer_allowance, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"

BASE = mi.WORKLOADS["tiny"]
CASES = {
    "one_token": BASE.with_(tokens=1),
    "one_token_wide": BASE.with_(tokens=1, hidden=1024, inter=256, n_experts=64, n_slots=64, top_k=6,
                                 inter_shared=256),
    "k_equals_E": BASE.with_(tokens=24, top_k=8),
    "single_expert": BASE.with_(tokens=33, n_experts=1, n_slots=1, n_blocks=1, top_k=1),
    "no_shared": BASE.with_(tokens=40, n_shared=0),
    "max_experts_topk": BASE.with_(tokens=48, hidden=128, inter=64, n_experts=1024, n_slots=1024, n_blocks=8,
                                   top_k=32, inter_shared=64),
    "odd_rows": BASE.with_(tokens=77, hidden=72, inter=40, inter_shared=24),
}


@pytest.mark.parametrize("mode", [m.MOE_FFN_DECODE, m.MOE_FFN_PREFILL])
@pytest.mark.parametrize("name", sorted(CASES))
def test_edge_case_forward_matches_oracle(name, mode):
    w = CASES[name]
    x, wr = mi.hidden_states(w), mi.router_weight(w)
    wg, wu, wd = mi.stacked_expert_weights(w)
    if w.n_shared:
        sg, su, sd = mi.stacked_shared_weights(w)
    else:
        sg = su = torch.zeros((0, w.inter_shared, w.hidden), dtype=torch.bfloat16)
        sd = torch.zeros((0, w.hidden, w.inter_shared), dtype=torch.bfloat16)
    ref = oracle.moe_forward(w, x, wr, None, None, wg, wu, wd, sg, su, sd)
    layer = DeviceLayer(w, DEV, weights=tuple(t.to(DEV) for t in (wg, wu, wd)))
    r = layer.forward(mode)
    idx_g = r["idx"].cpu().numpy()
    sure = check_topk(idx_g, ref["idx"], ref["logits"], w.top_k)
    check_counts_of_routing(w, idx_g, r["counts"].cpu().numpy(), r["blocks"].cpu().numpy(), None, ref["idx"], sure)
    assert_close(to_np(r["out"])[sure], ref["out"][sure], what=name)


def test_largest_shape_routing_from_logits_is_bit_exact():
    w = CASES["max_experts_topk"].with_(tokens=300)
    lg = mi.fp32_logits(w)
    T, k = w.tokens, w.top_k
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    m.moe_route(w, T, None, None, None, lg.to(DEV), None, idx, tw, None)
    idx_o, wt_o = oracle.topk_softmax(lg.double(), k)
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    np.testing.assert_allclose(tw.cpu().numpy(), wt_o, rtol=2e-6, atol=1e-9)


def test_empty_batch_on_the_device():
    w = mi.WORKLOADS["tiny"]
    layer = DeviceLayer(w, DEV)
    counts = torch.full((w.n_slots + 1,), 7, dtype=torch.int32, device=DEV)
    offsets = torch.full((w.n_slots + 2,), 7, dtype=torch.int32, device=DEV)
    blocks = torch.full((w.n_blocks,), 7, dtype=torch.int32, device=DEV)
    m.moe_dispatch(w, 0, None, None, None, None, counts, blocks, offsets, None, None, None)
    m.moe_expert_histogram(w, 0, None, None, counts, blocks)
    out = torch.full((1, w.hidden), 3.0, dtype=torch.bfloat16, device=DEV)
    m.moe_forward(w, 0, layer.x, layer.wr, None, None, layer.wg, layer.wu, layer.wd, layer.sg, layer.su, layer.sd,
                  out, ws=torch.empty(16, dtype=torch.uint8, device=DEV))
    assert m.moe_check_status() == 0
    assert int(counts.abs().sum()) == 0 and int(offsets.abs().sum()) == 0 and int(blocks.abs().sum()) == 0
    assert torch.all(out == 3.0)  # nothing written


def test_out_of_range_ids_through_dispatch_are_flagged_and_isolated():
    w = mi.WORKLOADS["tiny"]
    T, k, S, H = w.tokens, w.top_k, w.n_slots, w.hidden
    idx, _ = oracle.topk_softmax(mi.fp32_logits(w).double(), k)
    idx = idx.copy()
    idx[2, 0] = 99
    idx[9, 1] = -1
    n = T * k
    i32 = dict(dtype=torch.int32, device=DEV)
    so, c, off = torch.empty(n, **i32), torch.empty(S + 1, **i32), torch.empty(S + 2, **i32)
    perm, inv = torch.empty(n, **i32), torch.empty(n, **i32)
    xd = torch.empty((n, H), dtype=torch.bfloat16, device=DEV)
    m.moe_dispatch(w, T, mi.hidden_states(w).to(DEV), torch.from_numpy(idx).to(DEV), None, so, c, None, off, perm,
                   inv, xd)
    assert m.moe_check_status() == m.MOE_ERR_DEVICE_STATUS
    so_o, bad = oracle.slot_map(w, idx)
    c_o, _ = oracle.histogram(w, so_o)
    off_o, perm_o, inv_o, _ = oracle.dispatch(w, T, so_o, c_o, None)
    assert bad == 2
    assert np.array_equal(c.cpu().numpy(), c_o) and np.array_equal(off.cpu().numpy(), off_o)
    assert np.array_equal(perm.cpu().numpy(), perm_o)
    # the bad assignments sit after every valid slot, in the invalid bucket
    assert off_o[S] == n - 2 and set(perm_o[n - 2:]) == {2 * k + 0, 9 * k + 1}


FP8_CASES = {k_: v for k_, v in CASES.items() if v.hidden % 16 == 0 and v.inter % 16 == 0
             and (v.n_shared * v.inter_shared) % 16 == 0}


@pytest.mark.parametrize("mode", [m.MOE_FFN_DECODE, m.MOE_FFN_PREFILL, m.MOE_FFN_AUTO])
@pytest.mark.parametrize("name", sorted(FP8_CASES))
def test_fp8_edge_case_forward_matches_fp8_oracle(name, mode):
    w = FP8_CASES[name]
    T, H = w.tokens, w.hidden
    x, wr = mi.hidden_states(w), mi.router_weight(w)
    wg, wu, wd = mi.stacked_expert_weights(w)
    if w.n_shared:
        sg, su, sd = mi.stacked_shared_weights(w)
    else:
        sg = su = sd = None
    q = oracle.quantize_layer_fp8(w, wg, wu, wd, sg, su, sd)
    ref = oracle.moe_forward_fp8(w, x, wr, None, None, q)
    d = {k_: torch.from_numpy(np.ascontiguousarray(v)).to(DEV) for k_, v in q.items()}
    if not w.n_shared:
        for k_ in ("qsg", "ssg", "qsu", "ssu", "qsd", "ssd"):
            d[k_] = None
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device=DEV)
    ws = torch.empty(max(16, m.moe_workspace_size_fp8(w, T)), dtype=torch.uint8, device=DEV)
    m.moe_forward_fp8(w, T, x.to(DEV), wr.to(DEV), None, None, d["qg"], d["sg"], d["qu"], d["su"], d["qd"], d["sd"],
                      d["qsg"], d["ssg"], d["qsu"], d["ssu"], d["qsd"], d["ssd"], out, topk_idx_out=idx, mode=mode,
                      ws=ws)
    assert m.moe_check_status() == 0, m.last_error()
    lo = oracle.router_logits(w, x, wr, None)
    sure = check_topk(idx.cpu().numpy(), ref["idx"], lo, w.top_k)
    assert_close(to_np(out)[sure], ref["out"][sure], what=f"{name} fp8", e4m3_layer=True,
                 allowance=fp8_layer_allowance(w, ref)[sure])
