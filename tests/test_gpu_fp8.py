"""FP8 path on the GPU against the fp64 oracle of the same quantised layer.

Quantisation decides integers (codes), so codes and scales must match the
oracle bit-exactly; the FP8 GEMM then sees exactly the oracle's operands and
its output is held to the same tolerance as the bf16 path.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle
from moe_testlib import assert_close, check_topk, parallel_router_logits, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"

# ragged in every GEMM dimension; hidden a multiple of 16 for 1-byte rows
MID8 = mi.WORKLOADS["tiny"].with_(name="mid8", tokens=100, hidden=608, inter=328, n_experts=16, top_k=4,
                                  n_shared=2, inter_shared=200, n_slots=16, n_blocks=4)
REP8 = mi.WORKLOADS["tiny"].with_(name="rep8", tokens=64, hidden=128, inter=64, n_experts=8, top_k=2,
                                  n_shared=1, inter_shared=64, n_slots=12, n_blocks=4)


def _u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(DEV)


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV)


def test_row_quantizer_is_bit_exact():
    x = mi.normal_bf16((64, 7168), 1.0, 3, 40)
    x[3] = 0
    x[5, :] = mi.normal_bf16((7168,), 1e-3, 3, 41)
    x[7, 11] = 1e4   # one outlier sets the scale
    x[9] = mi.normal_bf16((7168,), 50.0, 3, 42)
    codes = torch.empty((64, 7168), dtype=torch.uint8, device=DEV)
    scale = torch.empty(64, dtype=torch.float32, device=DEV)
    m.moe_quantize_rows_fp8(x.to(DEV), codes, scale)
    c_o, s_o = oracle.quantize_rows_e4m3(x)
    assert np.array_equal(scale.cpu().numpy(), s_o)
    assert np.array_equal(codes.cpu().numpy(), c_o)


def _quantised_weights(w, rep=None):
    wg, wu, wd = mi.stacked_expert_weights(w, rep)
    sg, su, sd = mi.stacked_shared_weights(w)
    H = w.hidden
    q = {}
    q["qg"], q["sg"] = oracle.quantize_rows_e4m3(wg.reshape(-1, H))
    q["qu"], q["su"] = oracle.quantize_rows_e4m3(wu.reshape(-1, H))
    q["qsg"], q["ssg"] = oracle.quantize_rows_e4m3(sg.reshape(-1, H))
    q["qsu"], q["ssu"] = oracle.quantize_rows_e4m3(su.reshape(-1, H))
    q["wd"] = wd
    return q, sd


@pytest.mark.parametrize("name", ["tiny", "mid8", "rep8"])
def test_fp8_dispatch_is_bit_exact(name):
    w = {"tiny": mi.WORKLOADS["tiny"], "mid8": MID8, "rep8": REP8}[name]
    T, k, S, H = w.tokens, w.top_k, w.n_slots, w.hidden
    rep = None
    if w.n_slots > w.n_experts:
        rep = oracle.plan_replicas(w, np.arange(w.n_experts)[::-1].copy(), w.n_slots - w.n_experts)
    idx, _ = oracle.topk_softmax(mi.fp32_logits(w).double(), k)
    x = mi.hidden_states(w)
    n = T * k
    i32 = dict(dtype=torch.int32, device=DEV)
    g = dict(so=torch.empty(n, **i32), c=torch.empty(S + 1, **i32), b=torch.empty(w.n_blocks, **i32),
             off=torch.empty(S + 2, **i32), perm=torch.empty(n, **i32), inv=torch.empty(n, **i32),
             x8=torch.empty((T, H), dtype=torch.uint8, device=DEV), xs=torch.empty(T, dtype=torch.float32, device=DEV),
             xd8=torch.empty((n, H), dtype=torch.uint8, device=DEV), xds=torch.empty(n, dtype=torch.float32, device=DEV))
    repd = torch.from_numpy(rep).to(DEV) if rep is not None else None
    m.moe_dispatch_fp8(w, T, x.to(DEV), torch.from_numpy(idx).to(DEV), repd, g["so"], g["c"], g["b"], g["off"],
                       g["perm"], g["inv"], g["x8"], g["xs"], g["xd8"], g["xds"])
    assert m.moe_check_status() == 0
    so, _ = oracle.slot_map(w, idx, rep)
    counts, blocks = oracle.histogram(w, so)
    offsets, perm, inv, _ = oracle.dispatch(w, T, so, counts, None)
    qx, sx = oracle.quantize_rows_e4m3(x)
    assert np.array_equal(g["off"].cpu().numpy(), offsets) and np.array_equal(g["perm"].cpu().numpy(), perm)
    assert np.array_equal(g["x8"].cpu().numpy(), qx) and np.array_equal(g["xs"].cpu().numpy(), sx)
    assert np.array_equal(g["xd8"].cpu().numpy(), qx[perm // k])
    assert np.array_equal(g["xds"].cpu().numpy(), sx[perm // k])
    assert g["xd8"].numel() == T * k * H  # one byte per element: half the bf16 dispatch buffer


@pytest.mark.parametrize("mode", [m.MOE_FFN_DECODE, m.MOE_FFN_PREFILL])
@pytest.mark.parametrize("name", ["tiny", "mid8", "rep8"])
def test_fp8_layer_matches_fp8_oracle(name, mode):
    w = {"tiny": mi.WORKLOADS["tiny"], "mid8": MID8, "rep8": REP8}[name]
    rep = None
    if w.n_slots > w.n_experts:
        rep = oracle.plan_replicas(w, np.arange(w.n_experts)[::-1].copy(), w.n_slots - w.n_experts)
    T, H = w.tokens, w.hidden
    x, wr = mi.hidden_states(w), mi.router_weight(w)
    q, sd = _quantised_weights(w, rep)
    ref = oracle.moe_forward_fp8(w, x, wr, None, rep, q, sd)
    lo = oracle.router_logits(w, x, wr, None)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device=DEV)
    ws = torch.empty(m.moe_workspace_size_fp8(w, T), dtype=torch.uint8, device=DEV)
    repd = torch.from_numpy(rep).to(DEV) if rep is not None else None
    m.moe_forward_fp8(w, T, x.to(DEV), wr.to(DEV), None, repd, _u8(q["qg"]), _f32(q["sg"]), _u8(q["qu"]),
                      _f32(q["su"]), q["wd"].to(DEV), _u8(q["qsg"]), _f32(q["ssg"]), _u8(q["qsu"]), _f32(q["ssu"]),
                      sd.to(DEV), out, topk_idx_out=idx, mode=mode, ws=ws)
    assert m.moe_check_status() == 0, m.last_error()
    sure = check_topk(idx.cpu().numpy(), ref["idx"], lo, w.top_k)
    assert_close(to_np(out)[sure], ref["out"][sure], what=f"{name} fp8 layer")


_EXPERTS = {}


def test_fp8_layer_full_decode_shape_sampled_tokens():
    w = mi.WORKLOADS["decode_t32"]
    T, H, k = w.tokens, w.hidden, w.top_k
    wg, wu, wd = mi.stacked_expert_weights(w, device=DEV)
    sg, su, sd = mi.stacked_shared_weights(w, device=DEV)
    qg = torch.empty(wg.shape, dtype=torch.uint8, device=DEV)
    qu = torch.empty(wu.shape, dtype=torch.uint8, device=DEV)
    s_g = torch.empty(wg.shape[0] * wg.shape[1], dtype=torch.float32, device=DEV)
    s_u = torch.empty_like(s_g)
    m.moe_quantize_rows_fp8(wg.view(-1, H), qg, s_g)
    m.moe_quantize_rows_fp8(wu.view(-1, H), qu, s_u)
    del wg, wu
    qsg = torch.empty(sg.shape, dtype=torch.uint8, device=DEV)
    qsu = torch.empty(su.shape, dtype=torch.uint8, device=DEV)
    s_sg = torch.empty(sg.shape[0] * sg.shape[1], dtype=torch.float32, device=DEV)
    s_su = torch.empty_like(s_sg)
    m.moe_quantize_rows_fp8(sg.view(-1, H), qsg, s_sg)
    m.moe_quantize_rows_fp8(su.view(-1, H), qsu, s_su)
    x = mi.hidden_states(w)
    wr = mi.router_weight(w)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    ws = torch.empty(m.moe_workspace_size_fp8(w, T), dtype=torch.uint8, device=DEV)
    m.moe_forward_fp8(w, T, x.to(DEV), wr.to(DEV), None, None, qg, s_g, qu, s_u, wd, qsg, s_sg, qsu, s_su, sd, out,
                      topk_idx_out=idx, topk_w_out=tw, ws=ws)
    assert m.moe_check_status() == 0, m.last_error()
    lo = parallel_router_logits(w, x, wr, None)
    idx_o, wt_o = oracle.topk_softmax(lo, k)
    sure = check_topk(idx.cpu().numpy(), idx_o, lo, k)
    toks = [t for t in (0, 13, 31) if sure[t]]
    qx, sx = oracle.quantize_rows_e4m3(x)
    sgc, suc, sdc = mi.stacked_shared_weights(w)
    shq = [oracle.quantize_rows_e4m3(sgc[j]) + oracle.quantize_rows_e4m3(suc[j]) for j in range(w.n_shared)]
    for t in toks:
        ys = []
        for e in idx_o[t]:
            if int(e) not in _EXPERTS:
                g, u, d = mi.expert_weights(w, int(e))
                _EXPERTS[int(e)] = (oracle.quantize_rows_e4m3(g), oracle.quantize_rows_e4m3(u), d)
            (cg, scg), (cu, scu), d = _EXPERTS[int(e)]
            ys.append(oracle.swiglu_row_fp8(qx[t], sx[t], cg, scg, cu, scu, d))
        ysh = sum(oracle.swiglu_row_fp8(qx[t], sx[t], a, b_, c, d_, sdc[j])
                  for j, (a, b_, c, d_) in enumerate(shq))
        ref = oracle.combine(w.with_(tokens=1), 1, np.stack(ys), np.arange(k, dtype=np.int32), wt_o[t:t + 1],
                             ysh[None, :])
        assert_close(to_np(out)[t:t + 1], ref, what=f"fp8 decode token {t}")
