"""FP8 path on the GPU against the fp64 oracle of the same quantised layer.

Quantisation decides integers (codes), so codes and scales of the same bf16
input must match the oracle bit-exactly; each FP8 GEMM then sees exactly the
oracle's operands and its output is held to the same tolerance as the bf16
path.  The layer test compares with the oracle's whole FP8 layer, whose
intermediate h is its own (fp64, then bf16) rather than the kernel's.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle
from moe_testlib import (PAYLOAD_FLIP_SHARE, _report, assert_close, check_full_size_layer, check_topk, e4m3_step,
                         fp8_layer_allowance, parallel_router_logits, to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"

# ragged in every GEMM dimension; hidden a multiple of 16 for 1-byte rows
MID8 = mi.WORKLOADS["tiny"].with_(name="mid8", tokens=100, hidden=608, inter=336, n_experts=16, top_k=4,
                                  n_shared=2, inter_shared=200, n_slots=16, n_blocks=4)
REP8 = mi.WORKLOADS["tiny"].with_(name="rep8", tokens=64, hidden=128, inter=64, n_experts=8, top_k=2,
                                  n_shared=1, inter_shared=64, n_slots=12, n_blocks=4)
# 800 assignments over 32 experts (25 rows a slot on average, so the automatic
# mode gives the E4M3 down 128-row chunks), skewed so that two experts hold
# ~400 rows each: several full chunks and a ragged one, and many empty slots
SKEW8 = mi.WORKLOADS["tiny"].with_(name="skew8", tokens=400, hidden=256, inter=128, n_experts=32, top_k=2,
                                   n_shared=1, inter_shared=128, n_slots=32, n_blocks=4, skew_alpha=1.5)
MODES = [m.MOE_FFN_DECODE, m.MOE_FFN_PREFILL, m.MOE_FFN_AUTO]


def _u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(DEV)


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV)


@pytest.mark.parametrize("rows,cols", [(64, 7168), (300, 2048), (33, 4096), (5, 48), (7, 16384), (6, 16400)])
def test_row_quantizer_is_bit_exact(rows, cols):
    """Every row width the kernel distinguishes: one warp per row (2048, 48),
    several warps per row through shared memory (4096, 7168, 16384), and rows
    too wide for the registers of one CTA (16400)."""
    x = mi.normal_bf16((rows, cols), 1.0, 3, 40)
    x[min(3, rows - 1)] = 0
    if rows > 5:
        x[5, :] = mi.normal_bf16((cols,), 1e-3, 3, 41)
        x[4, 11] = 1e4   # one outlier sets the scale
        x[rows - 1] = mi.normal_bf16((cols,), 50.0, 3, 42)
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=DEV)
    scale = torch.empty(rows, dtype=torch.float32, device=DEV)
    m.moe_quantize_rows_fp8(x.to(DEV), codes, scale)
    c_o, s_o = oracle.quantize_rows_e4m3(x)
    assert np.array_equal(scale.cpu().numpy(), s_o)
    assert np.array_equal(codes.cpu().numpy(), c_o)


def _bf16_sweep_rows(n_rows=256, binades=20, seed=7):
    """Rows holding every bf16 mantissa, both signs, in the `binades` binades at
    and below the row maximum, zero-padded to a multiple of 16 columns.  Row
    maxima: 448 * 2^k (power-of-two scales, so exact E4M3 ties occur), random
    bf16 values, the extremes of the bf16 range, and scales on both sides of
    2^-96."""
    rng = np.random.default_rng(seed)
    maxima = []
    for r in range(n_rows):
        if r % 2 == 0:
            maxima.append(448.0 * 2.0 ** int(rng.integers(-120, 110)))
        else:
            maxima.append(float(torch.tensor(2.0 ** rng.uniform(-125, 126), dtype=torch.float32)
                                .to(torch.bfloat16).float()))
    maxima[:6] = [448.0 * 2.0 ** -96, 446.0 * 2.0 ** -96, 450.0 * 2.0 ** -96, 2.0 ** -130, 3.0e38, 448.0]
    cols = ((2 * binades * 128 + 1 + 15) // 16) * 16
    out = np.zeros((n_rows, cols), dtype=np.uint16)
    for r, mx in enumerate(maxima):
        mb = int(torch.tensor(mx, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()) & 0x7FFF
        top = (mb >> 7) & 0xFF  # biased exponent of the maximum
        vals = []
        for eb in range(max(0, top - binades + 1), top + 1):
            for mant in range(128):
                b = (eb << 7) | mant
                if b <= mb:
                    vals += [b, b | 0x8000]
        row = np.array(vals + [mb], dtype=np.uint16)
        out[r, :len(row)] = row
    return torch.from_numpy(out.view(np.int16)).view(torch.bfloat16)


def test_row_quantizer_over_every_bf16_mantissa_is_bit_exact():
    x = _bf16_sweep_rows()
    rows, cols = x.shape
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=DEV)
    scale = torch.empty(rows, dtype=torch.float32, device=DEV)
    m.moe_quantize_rows_fp8(x.to(DEV), codes, scale)
    c_o, s_o = oracle.quantize_rows_e4m3(x)
    assert np.array_equal(scale.cpu().numpy(), s_o)
    got = codes.cpu().numpy()
    assert np.array_equal(got, c_o), f"{int((got != c_o).sum())} codes differ"
    # the sweep reaches exact ties: values halfway between two E4M3 codes at a power-of-two scale
    assert any(float(s_) == 2.0 ** round(np.log2(float(s_))) for s_ in s_o)


def _quantised_weights(w, rep=None):
    wg, wu, wd = mi.stacked_expert_weights(w, rep)
    sg, su, sd = mi.stacked_shared_weights(w)
    return oracle.quantize_layer_fp8(w, wg, wu, wd, sg, su, sd)


def _dev(q):
    return {k_: (_u8(v) if k_.startswith("q") else _f32(v)) for k_, v in q.items()}


def test_shared_down_matrix_quantised_on_the_device_is_bit_exact():
    w = MID8
    _, _, sd = mi.stacked_shared_weights(w)
    mat = oracle.shared_down_matrix(sd)
    c_o, s_o = oracle.quantize_rows_e4m3(mat)
    codes = torch.empty(mat.shape, dtype=torch.uint8, device=DEV)
    scale = torch.empty(mat.shape[0], dtype=torch.float32, device=DEV)
    m.moe_quantize_rows_fp8(sd.to(DEV).permute(1, 0, 2).reshape(w.hidden, -1).contiguous(), codes, scale)
    assert np.array_equal(codes.cpu().numpy(), c_o) and np.array_equal(scale.cpu().numpy(), s_o)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", ["tiny", "mid8", "skew8"])
def test_fp8_intermediate_and_down_stage(name, mode):
    """Gate/up on the GPU, then the stage under test on the GPU's own h: the
    row quantiser (bit-exact against the oracle on the same bf16 h) and the
    FP8 down GEMM (against the oracle's down row on the same codes)."""
    w = {"tiny": mi.WORKLOADS["tiny"], "mid8": MID8, "skew8": SKEW8}[name]
    T, k, S, H, I = w.tokens, w.top_k, w.n_slots, w.hidden, w.inter
    Ks = w.n_shared * w.inter_shared
    q = _quantised_weights(w)
    d = _dev(q)
    idx, _ = oracle.topk_softmax(mi.fp32_logits(w).double(), k)
    x = mi.hidden_states(w)
    n = T * k
    i32 = dict(dtype=torch.int32, device=DEV)
    so, c, b = torch.empty(n, **i32), torch.empty(S + 1, **i32), torch.empty(w.n_blocks, **i32)
    off, perm, inv = torch.empty(S + 2, **i32), torch.empty(n, **i32), torch.empty(n, **i32)
    x8 = torch.empty((T, H), dtype=torch.uint8, device=DEV)
    xs = torch.empty(T, dtype=torch.float32, device=DEV)
    xd8 = torch.empty((n, H), dtype=torch.uint8, device=DEV)
    xds = torch.empty(n, dtype=torch.float32, device=DEV)
    m.moe_dispatch_fp8(w, T, x.to(DEV), torch.from_numpy(idx).to(DEV), None, so, c, b, off, perm, inv, x8, xs, xd8,
                       xds)
    h = torch.empty((n, I), dtype=torch.bfloat16, device=DEV)
    hs = torch.empty((T, Ks), dtype=torch.bfloat16, device=DEV)
    m.moe_expert_gate_up_fp8(w, T, x8, xs, xd8, xds, off, d["qg"], d["sg"], d["qu"], d["su"], d["qsg"], d["ssg"],
                             d["qsu"], d["ssu"], h, hs, mode=mode)
    h8, h8s = torch.empty((n, I), dtype=torch.uint8, device=DEV), torch.empty(n, dtype=torch.float32, device=DEV)
    hs8, hs8s = torch.empty((T, Ks), dtype=torch.uint8, device=DEV), torch.empty(T, dtype=torch.float32, device=DEV)
    m.moe_quantize_rows_fp8(h, h8, h8s)
    m.moe_quantize_rows_fp8(hs, hs8, hs8s)
    y = torch.empty((n, H), dtype=torch.bfloat16, device=DEV)
    ysh = torch.empty((T, H), dtype=torch.float32, device=DEV)
    m.moe_expert_down_fp8(w, T, h8, h8s, hs8, hs8s, off, d["qd"], d["sd"], d["qsd"], d["ssd"], y, ysh, mode=mode)
    assert m.moe_check_status() == 0, m.last_error()
    qh_o, sh_o = oracle.quantize_rows_e4m3(h.cpu())
    assert np.array_equal(h8.cpu().numpy(), qh_o) and np.array_equal(h8s.cpu().numpy(), sh_o)
    qhs_o, shs_o = oracle.quantize_rows_e4m3(hs.cpu())
    assert np.array_equal(hs8.cpu().numpy(), qhs_o) and np.array_equal(hs8s.cpu().numpy(), shs_o)
    offs = off.cpu().numpy()
    slot_of_row = np.searchsorted(offs[:S + 1], np.arange(n), side="right") - 1
    qd = q["qd"].reshape(S, H, I)
    sd = q["sd"].reshape(S, H)
    y_o = np.stack([oracle.down_row_fp8(qh_o[r], sh_o[r], qd[s_], sd[s_]) for r, s_ in enumerate(slot_of_row)])
    assert_close(to_np(y), y_o, what=f"{name} FP8 down (routed)")
    ysh_o = np.stack([oracle.down_row_fp8(qhs_o[t], shs_o[t], q["qsd"], q["ssd"]) for t in range(T)])
    assert_close(ysh.cpu().numpy().astype(np.float64), ysh_o, what=f"{name} FP8 down (shared)", bf16_out=False)

    # the same down projection with the E4M3 combine payload out
    nbk = (H + oracle.PAYLOAD_BLOCK - 1) // oracle.PAYLOAD_BLOCK
    y8 = torch.full((n, H), 0x7F, dtype=torch.uint8, device=DEV)  # 0x7F (NaN) is never written by a saturating encode
    y8s = torch.full((n, nbk), float("nan"), dtype=torch.float32, device=DEV)
    ysh2 = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    m.moe_expert_down_fp8_payload(w, T, h8, h8s, hs8, hs8s, off, d["qd"], d["sd"], d["qsd"], d["ssd"], y8, y8s, ysh2,
                                  mode=mode)
    assert m.moe_check_status() == 0, m.last_error()
    assert torch.equal(ysh2, ysh)
    c_g, s_g = y8.cpu().numpy(), y8s.cpu().numpy()
    # the payload is the block quantisation (oracle rule) of the bf16 y the plain kernel writes on the same inputs
    c_k, s_k = oracle.quantize_blocks_e4m3(y.cpu(), oracle.PAYLOAD_BLOCK)
    assert np.array_equal(s_g, s_k) and np.array_equal(c_g, c_k)
    # and the oracle's payload of its own fp64 y: equal codes and scales but for rare one-step flips where the
    # kernel's fp32 y and the oracle's fp64 y round to different bf16 values
    deq_o, c_o, s_o = oracle.payload_e4m3(y_o)
    assert np.all(np.abs(s_g / s_o - 1.0) <= 2.0 ** -7)
    assert (s_g != s_o).mean() <= 0.02
    deq_g = oracle.e4m3_decode(c_g).reshape(c_g.shape) * np.repeat(s_g.astype(np.float64), oracle.PAYLOAD_BLOCK,
                                                                    axis=1)[:, :H]
    flips = c_g != c_o
    assert flips.mean() <= PAYLOAD_FLIP_SHARE, f"{flips.sum()} payload codes differ from the oracle's"
    step = e4m3_step(c_o) * np.repeat(s_o.astype(np.float64), oracle.PAYLOAD_BLOCK, axis=1)[:, :H]
    assert np.all(np.abs(deq_g - deq_o) <= step * 1.01 + np.abs(deq_o) * 2.0 ** -6)

    # the E4M3 combine on the oracle's payload (every input from the oracle)
    idx_t = torch.from_numpy(idx).to(DEV)
    tw_o = np.ascontiguousarray(oracle.topk_softmax(mi.fp32_logits(w).double(), k)[1])
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    so_o, _ = oracle.slot_map(w, idx)
    cnt_o, _ = oracle.histogram(w, so_o)
    _, _, inv_o, _ = oracle.dispatch(w, T, so_o, cnt_o, None)
    m.moe_combine_fp8(w, T, torch.from_numpy(c_o).to(DEV), torch.from_numpy(s_o).to(DEV),
                      torch.from_numpy(inv_o).to(DEV), torch.from_numpy(tw_o.astype(np.float32)).to(DEV),
                      torch.from_numpy(ysh_o.astype(np.float32)).to(DEV), out)
    assert m.moe_check_status() == 0, m.last_error()
    ref = oracle.combine(w, T, deq_o, inv_o, tw_o.astype(np.float32).astype(np.float64),
                         ysh_o.astype(np.float32).astype(np.float64))
    assert_close(to_np(out), ref, what=f"{name} E4M3 combine")
    del idx_t


# 4096 dispatched rows of 7168 bytes: the chunked index pass and the bulk-copy scatter
BIG8 = mi.WORKLOADS["decode_t32"].with_(name="big8", tokens=512)


@pytest.mark.parametrize("name", ["tiny", "mid8", "rep8", "big8"])
def test_fp8_dispatch_is_bit_exact(name):
    w = {"tiny": mi.WORKLOADS["tiny"], "mid8": MID8, "rep8": REP8, "big8": BIG8}[name]
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


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", ["tiny", "mid8", "rep8", "skew8"])
def test_fp8_layer_matches_fp8_oracle(name, mode):
    _fp8_layer_case(name, mode)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", ["mid8", "skew8"])
def test_fp8_layer_with_outlier_tokens(name, mode):
    """Hidden states with two planted outliers of 8 to 20 sigma per row: the row
    scale follows the outlier, the other entries quantise coarsely, and the
    kernel must still match the oracle's E4M3 layer on the same codes."""
    _fp8_layer_case(name, mode, outliers=True)


def _fp8_layer_case(name, mode, outliers=False):
    w = {"tiny": mi.WORKLOADS["tiny"], "mid8": MID8, "rep8": REP8, "skew8": SKEW8}[name]
    rep = None
    if w.n_slots > w.n_experts:
        rep = oracle.plan_replicas(w, np.arange(w.n_experts)[::-1].copy(), w.n_slots - w.n_experts)
    T, H = w.tokens, w.hidden
    x, wr = mi.hidden_states(w), mi.router_weight(w)
    if outliers:
        x = mi.with_outliers(x, seed=11)
        qx, _ = oracle.quantize_rows_e4m3(x)
        assert (qx & 0x7F).max() == 0x7E  # the outliers set the row scales
    q = _quantised_weights(w, rep)
    b = mi.router_bias(w)
    ref = oracle.moe_forward_fp8(w, x, wr, b, rep, q)
    lo = oracle.router_logits(w, x, wr, b)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device=DEV)
    ws = torch.empty(m.moe_workspace_size_fp8(w, T), dtype=torch.uint8, device=DEV)
    repd = torch.from_numpy(rep).to(DEV) if rep is not None else None
    d = _dev(q)
    bd = torch.from_numpy(b).to(DEV) if b is not None else None
    m.moe_forward_fp8(w, T, x.to(DEV), wr.to(DEV), bd, repd, d["qg"], d["sg"], d["qu"], d["su"], d["qd"], d["sd"],
                      d["qsg"], d["ssg"], d["qsu"], d["ssu"], d["qsd"], d["ssd"], out, topk_idx_out=idx, mode=mode,
                      ws=ws)
    assert m.moe_check_status() == 0, m.last_error()
    sure = check_topk(idx.cpu().numpy(), ref["idx"], lo, w.top_k)
    stats = assert_close(to_np(out)[sure], ref["out"][sure], what=f"{name} fp8 layer{' outliers' if outliers else ''}",
                         e4m3_layer=True, allowance=fp8_layer_allowance(w, ref)[sure])
    if outliers:  # how far the E4M3 layer is from the bf16 layer on these tokens (reported, not a parity bound)
        wg, wu, wd = mi.stacked_expert_weights(w, rep)
        sg, su, sd = mi.stacked_shared_weights(w)
        r16 = oracle.moe_forward(w, x, wr, b, rep, wg, wu, wd, sg, su, sd)["out"]
        dev16 = float(np.linalg.norm(ref["out"] - r16) / np.linalg.norm(r16))
        _report(dict(kind="e4m3_vs_bf16_layer", what=stats["what"], rel_frob=dev16))
        assert dev16 < 0.2


@pytest.fixture(scope="module")
def dsv3_bf16():
    """The 256 DeepSeek-V3-shaped experts in bf16 on the device: the source of
    the device E4M3 copies and of the host copies the oracle quantises itself."""
    return mi.stacked_expert_weights(mi.WORKLOADS["decode_t32"], device=DEV)


@pytest.fixture(scope="module")
def fp8_dsv3(dsv3_bf16):
    """Every DeepSeek-V3-shaped expert and shared matrix quantised on the device
    (the quantiser itself is pinned bit-exact above)."""
    w = mi.WORKLOADS["decode_t32"]
    H = w.hidden

    def quant(t):
        q = torch.empty(t.shape, dtype=torch.uint8, device=DEV)
        sc = torch.empty(t.numel() // t.shape[-1], dtype=torch.float32, device=DEV)
        m.moe_quantize_rows_fp8(t.view(-1, t.shape[-1]), q, sc)
        return q, sc.view(t.shape[:-1])

    d = {}
    wg, wu, wd = dsv3_bf16
    (d["qg"], d["sg"]), (d["qu"], d["su"]), (d["qd"], d["sd"]) = quant(wg), quant(wu), quant(wd)
    sg, su, sd = mi.stacked_shared_weights(w, device=DEV)
    (d["qsg"], d["ssg"]), (d["qsu"], d["ssu"]) = quant(sg), quant(su)
    d["qsd"], d["ssd"] = quant(sd.permute(1, 0, 2).reshape(H, -1).contiguous())
    del sg, su, sd
    torch.cuda.empty_cache()
    return d


def _replica_plan_of_skewed_batch(w):
    src = mi.WORKLOADS[mi.REPLICA_PLAN_SOURCE]
    lo = parallel_router_logits(src, mi.hidden_states(src), mi.router_weight(src), mi.router_bias(src))
    idx_src, _ = oracle.topk_softmax(lo, src.top_k)
    return oracle.plan_replicas(w, np.bincount(idx_src.ravel(), minlength=w.n_experts), mi.N_REPLICAS)


# decode T=32 runs the 32-row chunk, the skewed T=256 batch the 160-row gate/up
# and the 128-row down chunk of the automatic mode (hot experts hold more than
# one), prefill T=4096 the 160-row chunks with the chunked index pass, the
# redundant T=1024 batch the replica slots; the calibrated skew touches every expert
# with at most 65 rows
@pytest.mark.parametrize("name", ["decode_t32", "decode_t256_skew", "decode_t256_skew_a05", "prefill_t4096",
                                  "redundant_t1024"])
def test_fp8_layer_full_shape(name, dsv3_bf16, fp8_dsv3):
    """The E4M3 layer at the bench's launch configuration against the oracle's
    E4M3 layer: every token's routing, the counts of the GPU's own routing, and
    256 seeded random tokens' outputs (all 32 at T=32) element by element."""
    _fp8_full_shape(name, dsv3_bf16, fp8_dsv3, mi.hidden_states(mi.WORKLOADS[name]))


@pytest.mark.parametrize("name", ["decode_t32", "decode_t256_skew_a05"])
def test_fp8_layer_full_shape_with_outlier_tokens(name, dsv3_bf16, fp8_dsv3):
    """As above with two planted 8-20 sigma entries in every token row, so that
    each row's E4M3 scale is set by an outlier and the rest of the row
    quantises coarsely (the case per-row scaling is weakest at)."""
    x = mi.with_outliers(mi.hidden_states(mi.WORKLOADS[name]), seed=77)
    _fp8_full_shape(name, dsv3_bf16, fp8_dsv3, x, what=f"{name} E4M3 with outliers")


def _fp8_full_shape(name, dsv3_bf16, fp8_dsv3, x, what=None):
    w = mi.WORKLOADS[name]
    T, H, k, S = w.tokens, w.hidden, w.top_k, w.n_slots
    d = dict(fp8_dsv3)
    rep = None
    if S > w.n_experts:
        rep = _replica_plan_of_skewed_batch(w)
        se = torch.from_numpy(mi.slot_experts(w, rep)).to(DEV)
        for key in ("qg", "sg", "qu", "su", "qd", "sd"):
            d[key] = d[key].index_select(0, se)
    b = mi.router_bias(w)
    i32 = dict(dtype=torch.int32, device=DEV)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    idx, counts, blocks = torch.empty((T, k), **i32), torch.empty(S + 1, **i32), torch.empty(w.n_blocks, **i32)
    ws = torch.empty(m.moe_workspace_size_fp8(w, T), dtype=torch.uint8, device=DEV)
    bd = torch.from_numpy(b).to(DEV) if b is not None else None
    repd = torch.from_numpy(rep).to(DEV) if rep is not None else None
    m.moe_forward_fp8(w, T, x.to(DEV), mi.router_weight(w, device=DEV), bd, repd, d["qg"], d["sg"], d["qu"],
                      d["su"], d["qd"], d["sd"], d["qsg"], d["ssg"], d["qsu"], d["ssu"], d["qsd"], d["ssd"], out,
                      topk_idx_out=idx, counts_out=counts, block_counts_out=blocks, ws=ws)
    assert m.moe_check_status() == 0, m.last_error()
    if name == "decode_t256_skew":
        assert int(counts.max()) > 128  # a two-chunk expert is present
    del d
    sgc, suc, sdc = mi.stacked_shared_weights(w)
    qsh = {}
    qsh["qsg"], qsh["ssg"] = oracle.quantize_rows_e4m3(sgc.reshape(-1, H))
    qsh["qsu"], qsh["ssu"] = oracle.quantize_rows_e4m3(suc.reshape(-1, H))
    qsh["qsd"], qsh["ssd"] = oracle.quantize_rows_e4m3(oracle.shared_down_matrix(sdc))
    check_full_size_layer(w, to_np(out), idx.cpu().numpy(), counts.cpu().numpy(), blocks.cpu().numpy(),
                          lambda e: tuple(t[e].cpu() for t in dsv3_bf16), qsh, rep=rep, fp8=True,
                          what=what or f"{name} E4M3 sampled out", x=x)
