"""Experts with more rows than one prefill token chunk (160 rows), at scale:
12288 tokens over 512 experts (18 to 457 rows each, most of them in two or
three chunks that each stream the expert's weights), bf16 and FP8 against
the oracle on every output whose routing is decided (top-k gap above 1e-4)."""
import numpy as np
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle
from moe_testlib import DeviceLayer, assert_close, check_counts_of_routing, check_topk, fp8_layer_allowance, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"

# ~192 rows per expert: most experts exceed 160 rows
WIDE = mi.WORKLOADS["tiny"].with_(name="many_rows", tokens=12288, hidden=64, inter=32, n_experts=512, n_slots=512,
                                 n_blocks=8, top_k=8, n_shared=1, inter_shared=32)


def _multi_chunk_experts(counts, bn=160):
    return int((counts > bn).sum())


def test_multi_chunk_layer_bf16_matches_oracle():
    w = WIDE
    x, wr = mi.hidden_states(w), mi.router_weight(w)
    wg, wu, wd = mi.stacked_expert_weights(w)
    sg, su, sd = mi.stacked_shared_weights(w)
    ref = oracle.moe_forward(w, x, wr, None, None, wg, wu, wd, sg, su, sd)
    assert _multi_chunk_experts(ref["counts"][:w.n_slots]) > w.n_experts // 2
    layer = DeviceLayer(w, DEV, weights=tuple(t.to(DEV) for t in (wg, wu, wd)))
    r = layer.forward(m.MOE_FFN_PREFILL)
    assert m.moe_check_status() == 0
    idx_g = r["idx"].cpu().numpy()
    sure = check_topk(idx_g, ref["idx"], ref["logits"], w.top_k)
    assert sure.mean() > 0.95  # near-ties (gap under 1e-4) are left out of the index check
    check_counts_of_routing(w, idx_g, r["counts"].cpu().numpy(), r["blocks"].cpu().numpy(), None, ref["idx"], sure)
    assert_close(to_np(r["out"])[sure], ref["out"][sure], what="multi-chunk bf16 layer")


def test_multi_chunk_layer_fp8_matches_oracle():
    w = WIDE
    x, wr = mi.hidden_states(w), mi.router_weight(w)
    wg, wu, wd = mi.stacked_expert_weights(w)
    sg, su, sd = mi.stacked_shared_weights(w)
    q = oracle.quantize_layer_fp8(w, wg, wu, wd, sg, su, sd)
    ref = oracle.moe_forward_fp8(w, x, wr, None, None, q)
    lo = oracle.router_logits(w, x, wr, None)
    counts = np.bincount(ref["idx"].ravel(), minlength=w.n_experts)
    assert _multi_chunk_experts(counts) > w.n_experts // 2
    d = {k_: torch.from_numpy(np.ascontiguousarray(v)).to(DEV) for k_, v in q.items()}
    T, H = w.tokens, w.hidden
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device=DEV)
    ws = torch.empty(m.moe_workspace_size_fp8(w, T), dtype=torch.uint8, device=DEV)
    m.moe_forward_fp8(w, T, x.to(DEV), wr.to(DEV), None, None, d["qg"], d["sg"], d["qu"], d["su"], d["qd"], d["sd"],
                      d["qsg"], d["ssg"], d["qsu"], d["ssu"], d["qsd"], d["ssd"], out, topk_idx_out=idx,
                      mode=m.MOE_FFN_PREFILL, ws=ws)
    assert m.moe_check_status() == 0, m.last_error()
    sure = check_topk(idx.cpu().numpy(), ref["idx"], lo, w.top_k)
    assert sure.mean() > 0.95  # near-ties (gap under 1e-4) are left out of the index check
    assert_close(to_np(out)[sure], ref["out"][sure], what="multi-chunk FP8 layer", e4m3_layer=True,
                 allowance=fp8_layer_allowance(w, ref)[sure])
