"""Every element of every output is written.  Each output buffer of the
staged calls and of the whole-layer calls is filled with a sentinel first
(NaN for floating point, 0x7F for E4M3 codes, which the saturating quantiser
never produces, an unlikely value for integers), so an element a kernel skips
cannot pass by holding an earlier run's value.  Ragged shapes, the chunked
index pass, all three kernel variants (32-, 128- and 160-row token chunks),
both precisions, group-limited routing, the histogram-only call and the
combined expert FFN."""
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENT_I32 = -0x7ABC0DEF

TINY = mi.WORKLOADS["tiny"]
# ragged in every GEMM dimension (H, I, I_sh not multiples of 64)
MID = TINY.with_(name="mid", tokens=100, hidden=600, inter=328, n_experts=16, top_k=4, n_shared=2,
                 inter_shared=200, n_slots=16, n_blocks=4)
# E4M3 rows need H and I multiples of 16
MID8 = MID.with_(name="mid8", hidden=608, inter=336)
# 4400 assignments: the chunked index pass; skewed, so some experts span several chunks
WIDE = TINY.with_(name="wide", tokens=2200, hidden=128, inter=64, n_experts=16, top_k=2, n_shared=1,
                  inter_shared=64, n_slots=16, n_blocks=4, skew_alpha=1.5)
MODES = [m.MOE_FFN_DECODE, m.MOE_FFN_PREFILL, m.MOE_FFN_AUTO]


def _f(shape, dtype=torch.float32):
    return torch.full(shape, float("nan"), dtype=dtype, device=DEV)


def _i(shape):
    return torch.full(shape, SENT_I32, dtype=torch.int32, device=DEV)


def _u8(shape):
    return torch.full(shape, 0x7F, dtype=torch.uint8, device=DEV)


def _assert_written(named):
    for name, t in named.items():
        if t.dtype in (torch.float32, torch.bfloat16):
            bad = int(torch.isnan(t).sum())
        elif t.dtype == torch.uint8:
            bad = int((t == 0x7F).sum())
        else:
            bad = int((t == SENT_I32).sum())
        assert bad == 0, f"{name}: {bad} of {t.numel()} elements never written"


def _layer(w):
    x, wr = mi.hidden_states(w, device=DEV), mi.router_weight(w, device=DEV)
    b = mi.router_bias(w)
    b = torch.from_numpy(b).to(DEV) if b is not None else None
    wg, wu, wd = mi.stacked_expert_weights(w, device=DEV)
    sg, su, sd = mi.stacked_shared_weights(w, device=DEV)
    return x, wr, b, wg, wu, wd, sg, su, sd


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("w", [TINY, MID, WIDE], ids=lambda w: w.name)
def test_staged_bf16_calls_write_every_output_element(w, mode):
    T, k, S, H, I, E = w.tokens, w.top_k, w.n_slots, w.hidden, w.inter, w.n_experts
    n, Ks = T * k, w.n_shared * w.inter_shared
    x, wr, b, wg, wu, wd, sg, su, sd = _layer(w)
    o = dict(logits=_f((T, E)), idx=_i((T, k)), tw=_f((T, k)), slot_of=_i((n,)), counts=_i((S + 1,)),
             blocks=_i((w.n_blocks,)), offsets=_i((S + 2,)), perm=_i((n,)), inv=_i((n,)),
             x_disp=_f((n, H), torch.bfloat16), h=_f((n, I), torch.bfloat16), hs=_f((T, Ks), torch.bfloat16),
             y=_f((n, H), torch.bfloat16), ysh=_f((T, H)), out=_f((T, H), torch.bfloat16))
    rws = torch.empty(max(16, m.moe_route_workspace_size(w, T)), dtype=torch.uint8, device=DEV)
    m.moe_route(w, T, x, wr, b, None, o["logits"], o["idx"], o["tw"], rws)
    m.moe_dispatch(w, T, x, o["idx"], None, o["slot_of"], o["counts"], o["blocks"], o["offsets"], o["perm"],
                   o["inv"], o["x_disp"])
    m.moe_expert_gate_up(w, T, x, o["x_disp"], o["offsets"], wg, wu, sg, su, o["h"], o["hs"], mode=mode)
    m.moe_expert_down(w, T, o["h"], o["hs"], o["offsets"], wd, sd, o["y"], o["ysh"], mode=mode)
    m.moe_combine(w, T, o["y"], o["inv"], o["tw"], o["ysh"], o["out"])
    assert m.moe_check_status() == 0, m.last_error()
    _assert_written(o)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("w", [TINY, MID, WIDE], ids=lambda w: w.name)
def test_forward_writes_every_output_element(w, mode):
    T, k = w.tokens, w.top_k
    x, wr, b, wg, wu, wd, sg, su, sd = _layer(w)
    o = dict(out=_f((T, w.hidden), torch.bfloat16), idx=_i((T, k)), tw=_f((T, k)), counts=_i((w.n_slots + 1,)),
             blocks=_i((w.n_blocks,)))
    ws = torch.empty(m.moe_workspace_size(w, T), dtype=torch.uint8, device=DEV)
    m.moe_forward(w, T, x, wr, b, None, wg, wu, wd, sg, su, sd, o["out"], o["idx"], o["tw"], o["counts"],
                  o["blocks"], mode=mode, ws=ws)
    assert m.moe_check_status() == 0, m.last_error()
    _assert_written(o)


def _quant(t):
    q = _u8(t.shape)
    s = _f((t.numel() // t.shape[-1],))
    m.moe_quantize_rows_fp8(t.reshape(-1, t.shape[-1]), q.view(-1, t.shape[-1]), s)
    return q, s


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("w", [TINY.with_(name="tiny16", hidden=64, inter=32), MID8, WIDE],
                         ids=lambda w: w.name)
def test_staged_fp8_calls_write_every_output_element(w, mode):
    T, k, S, H, I = w.tokens, w.top_k, w.n_slots, w.hidden, w.inter
    n, Ks = T * k, w.n_shared * w.inter_shared
    x, wr, b, wg, wu, wd, sg, su, sd = _layer(w)
    (qg, s_g), (qu, s_u), (qd, s_d) = _quant(wg), _quant(wu), _quant(wd)
    (qsg, s_sg), (qsu, s_su) = _quant(sg), _quant(su)
    qsd, s_sd = _quant(sd.permute(1, 0, 2).reshape(H, -1).contiguous())
    _assert_written(dict(qg=qg, s_g=s_g, qu=qu, s_u=s_u, qd=qd, s_d=s_d, qsg=qsg, s_sg=s_sg, qsu=qsu, s_su=s_su,
                         qsd=qsd, s_sd=s_sd))
    idx, tw = torch.empty((T, k), dtype=torch.int32, device=DEV), torch.empty((T, k), device=DEV)
    rws = torch.empty(max(16, m.moe_route_workspace_size(w, T)), dtype=torch.uint8, device=DEV)
    m.moe_route(w, T, x, wr, b, None, None, idx, tw, rws)
    o = dict(slot_of=_i((n,)), counts=_i((S + 1,)), blocks=_i((w.n_blocks,)), offsets=_i((S + 2,)),
             perm=_i((n,)), inv=_i((n,)), x8=_u8((T, H)), xs=_f((T,)), xd8=_u8((n, H)), xds=_f((n,)),
             h=_f((n, I), torch.bfloat16), hs=_f((T, Ks), torch.bfloat16), h8=_u8((n, I)), h8s=_f((n,)),
             hs8=_u8((T, Ks)), hs8s=_f((T,)), y=_f((n, H), torch.bfloat16), ysh=_f((T, H)),
             out=_f((T, H), torch.bfloat16))
    m.moe_dispatch_fp8(w, T, x, idx, None, o["slot_of"], o["counts"], o["blocks"], o["offsets"], o["perm"],
                       o["inv"], o["x8"], o["xs"], o["xd8"], o["xds"])
    m.moe_expert_gate_up_fp8(w, T, o["x8"], o["xs"], o["xd8"], o["xds"], o["offsets"], qg, s_g, qu, s_u, qsg, s_sg,
                             qsu, s_su, o["h"], o["hs"], mode=mode)
    m.moe_quantize_rows_fp8(o["h"], o["h8"], o["h8s"])
    m.moe_quantize_rows_fp8(o["hs"], o["hs8"], o["hs8s"])
    m.moe_expert_down_fp8(w, T, o["h8"], o["h8s"], o["hs8"], o["hs8s"], o["offsets"], qd, s_d, qsd, s_sd, o["y"],
                          o["ysh"], mode=mode)
    m.moe_combine(w, T, o["y"], o["inv"], tw, o["ysh"], o["out"])
    assert m.moe_check_status() == 0, m.last_error()
    _assert_written(o)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("w", [TINY, MID8, WIDE], ids=lambda w: w.name)
def test_forward_fp8_writes_every_output_element(w, mode):
    T, k, H = w.tokens, w.top_k, w.hidden
    x, wr, b, wg, wu, wd, sg, su, sd = _layer(w)
    (qg, s_g), (qu, s_u), (qd, s_d) = _quant(wg), _quant(wu), _quant(wd)
    (qsg, s_sg), (qsu, s_su) = _quant(sg), _quant(su)
    qsd, s_sd = _quant(sd.permute(1, 0, 2).reshape(H, -1).contiguous())
    o = dict(out=_f((T, H), torch.bfloat16), idx=_i((T, k)), tw=_f((T, k)), counts=_i((w.n_slots + 1,)),
             blocks=_i((w.n_blocks,)))
    ws = torch.empty(m.moe_workspace_size_fp8(w, T), dtype=torch.uint8, device=DEV)
    m.moe_forward_fp8(w, T, x, wr, b, None, qg, s_g, qu, s_u, qd, s_d, qsg, s_sg, qsu, s_su, qsd, s_sd, o["out"],
                      o["idx"], o["tw"], o["counts"], o["blocks"], mode=mode, ws=ws)
    assert m.moe_check_status() == 0, m.last_error()
    _assert_written(o)


@pytest.mark.parametrize("w", [TINY, MID, WIDE], ids=lambda w: w.name)
def test_grouped_route_histogram_and_ffn_write_every_output_element(w):
    T, k, S, H, E = w.tokens, w.top_k, w.n_slots, w.hidden, w.n_experts
    n = T * k
    x, wr, b, wg, wu, wd, sg, su, sd = _layer(w)
    groups = (w.n_blocks, max(1, w.n_blocks // 2))
    o = dict(logits=_f((T, E)), idx=_i((T, k)), tw=_f((T, k)), counts=_i((S + 1,)), blocks=_i((w.n_blocks,)))
    rws = torch.empty(max(16, m.moe_route_workspace_size(w, T)), dtype=torch.uint8, device=DEV)
    m.moe_route_grouped(w, T, groups[0], groups[1], x, wr, b, None, o["logits"], o["idx"], o["tw"], rws)
    m.moe_expert_histogram(w, T, o["idx"], None, o["counts"], o["blocks"])
    i32 = dict(dtype=torch.int32, device=DEV)
    so, c, off = torch.empty(n, **i32), torch.empty(S + 1, **i32), torch.empty(S + 2, **i32)
    perm, inv = torch.empty(n, **i32), torch.empty(n, **i32)
    xd = torch.empty((n, H), dtype=torch.bfloat16, device=DEV)
    m.moe_dispatch(w, T, x, o["idx"], None, so, c, None, off, perm, inv, xd)
    o.update(y=_f((n, H), torch.bfloat16), ysh=_f((T, H)))
    fws = torch.empty(max(16, m.moe_ffn_workspace_size(w, T)), dtype=torch.uint8, device=DEV)
    m.moe_expert_ffn(w, T, x, xd, off, wg, wu, wd, sg, su, sd, o["y"], o["ysh"], m.MOE_FFN_AUTO, fws)
    assert m.moe_check_status() == 0, m.last_error()
    _assert_written(o)
