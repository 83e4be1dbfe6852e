"""ctypes binding of the fp64 CPU oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library (``moe_expert_layer_06_gb300``) and is never on the
product path.  Arguments are marshalled here; every arithmetic step runs in
the C file, whose functions cite the passages of the blog post
"专家并行(EP)" they follow.

Arrays: bf16 tensors are passed as their uint16 bit patterns; results come
back as float64 / int32 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile liboracle.so (no fast-math, no FP contraction: same result on x86-64 and aarch64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "moe_oracle.h"))):
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-o", _LIB, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "inter", "n_experts", "top_k", "n_shared", "inter_shared", "n_slots", "n_blocks")]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _lib.oracle_home_slot.restype = ctypes.c_int32
        _lib.oracle_slot_map.restype = ctypes.c_int
        _lib.oracle_moe_forward.restype = ctypes.c_int
        _lib.oracle_plan_replicas.restype = ctypes.c_int
    return _lib


def shape_of(w) -> Shape:
    return Shape(*w.shape_tuple)


def _u16(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        assert t.dtype == torch.bfloat16
        return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    a = np.ascontiguousarray(t)
    assert a.dtype == np.uint16
    return a


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


def _i32(a) -> Optional[np.ndarray]:
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _f32(a) -> Optional[np.ndarray]:
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def _f64(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def bf16_to_double(v: int) -> float:
    f = lib().oracle_bf16_to_double
    f.restype = ctypes.c_double
    return f(ctypes.c_uint16(v))


def router_logits(w, x, w_router, bias=None) -> np.ndarray:
    T = x.shape[0]
    xs, wr, b = _u16(x), _u16(w_router), _f32(bias)
    out = np.empty((T, w.n_experts), dtype=np.float64)
    lib().oracle_router_logits(ctypes.byref(shape_of(w)), T, _ptr(xs), _ptr(wr), _ptr(b), _ptr(out))
    return out


def topk_softmax(logits, k: int):
    lg = _f64(logits)
    T, E = lg.shape
    idx = np.empty((T, k), dtype=np.int32)
    wt = np.empty((T, k), dtype=np.float64)
    lib().oracle_topk_softmax(T, E, k, _ptr(lg), _ptr(idx), _ptr(wt))
    return idx, wt


def topk_grouped(logits, k: int, n_groups: int, topk_groups: int):
    lg = _f64(logits)
    T, E = lg.shape
    assert E % n_groups == 0 and topk_groups * (E // n_groups) >= k
    idx = np.empty((T, k), dtype=np.int32)
    wt = np.empty((T, k), dtype=np.float64)
    lib().oracle_topk_grouped(T, E, k, n_groups, topk_groups, _ptr(lg), _ptr(idx), _ptr(wt))
    return idx, wt


def home_slot(w, e: int) -> int:
    return lib().oracle_home_slot(ctypes.byref(shape_of(w)), e)


def slot_map(w, idx, replica_of=None):
    ix = _i32(idx)
    T = ix.shape[0]
    rep = _i32(replica_of)
    out = np.empty(T * w.top_k, dtype=np.int32)
    invalid = lib().oracle_slot_map(ctypes.byref(shape_of(w)), T, _ptr(ix), _ptr(rep), _ptr(out))
    return out, invalid


def histogram(w, slot_of):
    so = _i32(slot_of)
    counts = np.empty(w.n_slots + 1, dtype=np.int32)
    blocks = np.empty(w.n_blocks, dtype=np.int32)
    lib().oracle_histogram(ctypes.byref(shape_of(w)), so.size, _ptr(so), _ptr(counts), _ptr(blocks))
    return counts, blocks


def dispatch(w, T: int, slot_of, counts, x=None):
    so, c = _i32(slot_of), _i32(counts)
    n = T * w.top_k
    offsets = np.empty(w.n_slots + 2, dtype=np.int32)
    perm = np.empty(n, dtype=np.int32)
    inv = np.empty(n, dtype=np.int32)
    xs = _u16(x) if x is not None else None
    xd = np.empty((n, w.hidden), dtype=np.uint16) if x is not None else None
    lib().oracle_dispatch(ctypes.byref(shape_of(w)), T, _ptr(so), _ptr(c), _ptr(xs), _ptr(offsets),
                          _ptr(perm), _ptr(inv), _ptr(xd))
    return offsets, perm, inv, xd


def swiglu_row(x_row, w_gate, w_up, w_down) -> np.ndarray:
    xr, g, u, d = _u16(x_row), _u16(w_gate), _u16(w_up), _u16(w_down)
    I, H = g.shape
    y = np.empty(H, dtype=np.float64)
    lib().oracle_swiglu_row(H, I, _ptr(xr), _ptr(g), _ptr(u), _ptr(d), _ptr(y))
    return y


def shared_rows(w, x, ws_gate, ws_up, ws_down) -> np.ndarray:
    xs, g, u, d = _u16(x), _u16(ws_gate), _u16(ws_up), _u16(ws_down)
    T = xs.shape[0]
    y = np.empty((T, w.hidden), dtype=np.float64)
    sh = shape_of(w)
    for t in range(T):
        lib().oracle_shared_row(ctypes.byref(sh), _ptr(xs[t]), _ptr(g), _ptr(u), _ptr(d),
                                y[t].ctypes.data_as(ctypes.c_void_p))
    return y


def expert_ffn(w, T: int, offsets, x_disp, w_gate, w_up, w_down) -> np.ndarray:
    off, xd = _i32(offsets), _u16(x_disp)
    g, u, d = _u16(w_gate), _u16(w_up), _u16(w_down)
    y = np.zeros((T * w.top_k, w.hidden), dtype=np.float64)
    lib().oracle_expert_ffn(ctypes.byref(shape_of(w)), T, _ptr(off), _ptr(xd), _ptr(g), _ptr(u),
                            _ptr(d), _ptr(y))
    return y


def combine(w, T: int, y_disp, inv_perm, weight, y_shared) -> np.ndarray:
    yd, ip, wt, ys = _f64(y_disp), _i32(inv_perm), _f64(weight), _f64(y_shared)
    out = np.empty((T, w.hidden), dtype=np.float64)
    lib().oracle_combine(ctypes.byref(shape_of(w)), T, _ptr(yd), _ptr(ip), _ptr(wt), _ptr(ys), _ptr(out))
    return out


def moe_forward(w, x, w_router, bias, replica_of, w_gate, w_up, w_down, ws_gate, ws_up, ws_down):
    """Whole layer; returns a dict of every intermediate and ``out`` [T,H] float64."""
    T = x.shape[0]
    E, k, S, H = w.n_experts, w.top_k, w.n_slots, w.hidden
    n = T * k
    r = dict(
        logits=np.empty((T, E), np.float64), idx=np.empty((T, k), np.int32),
        weight=np.empty((T, k), np.float64), slot_of=np.empty(n, np.int32),
        counts=np.empty(S + 1, np.int32), block_counts=np.empty(w.n_blocks, np.int32),
        offsets=np.empty(S + 2, np.int32), perm=np.empty(n, np.int32),
        inv_perm=np.empty(n, np.int32), out=np.empty((T, H), np.float64))
    args = [_u16(x), _u16(w_router), _f32(bias), _i32(replica_of), _u16(w_gate), _u16(w_up),
            _u16(w_down), _u16(ws_gate), _u16(ws_up), _u16(ws_down)]
    invalid = lib().oracle_moe_forward(
        ctypes.byref(shape_of(w)), T, *[_ptr(a) for a in args],
        *[_ptr(r[key]) for key in ("logits", "idx", "weight", "slot_of", "counts", "block_counts",
                                   "offsets", "perm", "inv_perm", "out")])
    r["invalid"] = invalid
    return r


def token_output(w, x_row, weight: Sequence[float], experts_gud: Sequence, ws_gate, ws_up, ws_down):
    """One token's output from its k combine weights and its experts' (gate, up, down)."""
    k = len(experts_gud)
    xr = _u16(x_row)
    keep = [tuple(_u16(m) for m in gud) for gud in experts_gud]
    PtrArr = ctypes.c_void_p * k
    g = PtrArr(*[a[0].ctypes.data for a in keep])
    u = PtrArr(*[a[1].ctypes.data for a in keep])
    d = PtrArr(*[a[2].ctypes.data for a in keep])
    wt = _f64(np.asarray(weight, dtype=np.float64))
    sg, su, sd = _u16(ws_gate), _u16(ws_up), _u16(ws_down)
    out = np.empty(w.hidden, dtype=np.float64)
    lib().oracle_token_output(ctypes.byref(shape_of(w)), _ptr(xr), k, _ptr(wt), g, u, d,
                              _ptr(sg), _ptr(su), _ptr(sd), _ptr(out))
    return out


def plan_replicas(w, expert_counts, n_rep: int) -> np.ndarray:
    c = _i32(expert_counts)
    assert c.size == w.n_experts
    rep = np.empty(w.n_experts, dtype=np.int32)
    rc = lib().oracle_plan_replicas(ctypes.byref(shape_of(w)), _ptr(c), n_rep, _ptr(rep))
    if rc != 0:
        raise ValueError("replica plan does not fit the shape")
    return rep


def eplb_window(w, history, window: int, replica_of=None, threshold: float = 1.2):
    """Sliding-window monitor: returns slot_window, block_load, expert_load, ratio, trigger."""
    h = np.ascontiguousarray(history, dtype=np.int32)
    n = h.shape[0]
    assert h.shape[1] == w.n_slots + 1
    sw = np.empty(w.n_slots + 1, np.int64)
    bl = np.empty(w.n_blocks, np.int64)
    el = np.empty(w.n_experts, np.int64)
    ratio = ctypes.c_double()
    trig = ctypes.c_int()
    lib().oracle_eplb_window(ctypes.byref(shape_of(w)), n, _ptr(h), window, _ptr(_i32(replica_of)),
                             ctypes.c_double(threshold), _ptr(sw), _ptr(bl), _ptr(el), ctypes.byref(ratio),
                             ctypes.byref(trig))
    return sw, bl, el, ratio.value, bool(trig.value)


# ------------------------------------------------------------------ FP8

def e4m3_encode(values) -> np.ndarray:
    f = lib().oracle_e4m3_encode
    f.restype = ctypes.c_uint8
    f.argtypes = [ctypes.c_float]
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([f(float(a)) for a in v], dtype=np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    f = lib().oracle_e4m3_decode
    f.restype = ctypes.c_double
    f.argtypes = [ctypes.c_uint8]
    return np.array([f(int(c)) for c in np.asarray(codes).ravel()], dtype=np.float64)


def quantize_rows_e4m3(x):
    """Per-row E4M3 codes [R, C] (uint8) and fp32 scales [R] of a bf16 tensor."""
    xs = _u16(x)
    R, C = xs.shape[0], int(np.prod(xs.shape[1:]))
    codes = np.empty((R, C), dtype=np.uint8)
    scale = np.empty(R, dtype=np.float32)
    lib().oracle_quantize_rows_e4m3(R, C, _ptr(xs), _ptr(codes), _ptr(scale))
    return codes.reshape(xs.shape), scale


PAYLOAD_BLOCK = 128  # columns per scale of the E4M3 combine payload (ORACLE_PAYLOAD_BLOCK)


def quantize_blocks_e4m3(x, block: int):
    """Per-(row, block of `block` columns) E4M3 codes [R, C] and fp32 scales [R, ceil(C/block)]."""
    xs = _u16(x)
    R, C = xs.shape[0], int(np.prod(xs.shape[1:]))
    nb = (C + block - 1) // block
    codes = np.empty((R, C), dtype=np.uint8)
    scale = np.empty((R, nb), dtype=np.float32)
    lib().oracle_quantize_blocks_e4m3(R, C, block, _ptr(xs), _ptr(codes), _ptr(scale))
    return codes, scale


def payload_e4m3(y):
    """The E4M3 combine payload of expert output rows y [R, H] (float64):
    returns (dequantised y [R, H] float64, codes [R, H] uint8, scales [R, nb] float32)."""
    yy = _f64(y)
    R, C = yy.shape
    nb = (C + PAYLOAD_BLOCK - 1) // PAYLOAD_BLOCK
    deq = np.empty((R, C), dtype=np.float64)
    codes = np.empty((R, C), dtype=np.uint8)
    scale = np.empty((R, nb), dtype=np.float32)
    lib().oracle_payload_e4m3(R, C, _ptr(yy), _ptr(deq), _ptr(codes), _ptr(scale))
    return deq, codes, scale


def bf16_round(values) -> np.ndarray:
    """Nearest bf16 (ties to even) of each value, as uint16 bit patterns."""
    f = lib().oracle_double_to_bf16
    f.restype = ctypes.c_uint16
    f.argtypes = [ctypes.c_double]
    v = np.asarray(values, dtype=np.float64)
    return np.array([f(float(a)) for a in v.ravel()], dtype=np.uint16).reshape(v.shape)


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(a, np.uint8)


def gate_up_row_fp8(qx, sx, qg, sg, qu, su) -> np.ndarray:
    """h = silu(g) * u of one row from E4M3 codes (qg/qu [I, H]) and scales."""
    qg, qu = _u8(qg), _u8(qu)
    I, H = qg.shape
    h = np.empty(I, dtype=np.float64)
    lib().oracle_gate_up_row_fp8(H, I, _ptr(_u8(qx)), ctypes.c_float(float(sx)), _ptr(qg), _ptr(_f32(sg)), _ptr(qu),
                                 _ptr(_f32(su)), _ptr(h))
    return h


def down_row_fp8(qh, sh, qd, sd) -> np.ndarray:
    """y[o] = sh * sd[o] * sum_i qh_i * qd[o, i] over decoded E4M3 codes (qd [H, K])."""
    qd = _u8(qd)
    H, K = qd.shape
    y = np.empty(H, dtype=np.float64)
    lib().oracle_down_row_fp8(K, H, _ptr(_u8(qh)), ctypes.c_float(float(sh)), _ptr(qd), _ptr(_f32(sd)), _ptr(y))
    return y


def swiglu_row_fp8(qx, sx, qg, sg, qu, su, qd, sd) -> np.ndarray:
    """One routed expert on one token in FP8 (gate/up, h -> bf16 -> E4M3 row, down)."""
    qg, qu, qd = _u8(qg), _u8(qu), _u8(qd)
    I, H = qg.shape
    y = np.empty(H, dtype=np.float64)
    lib().oracle_swiglu_row_fp8(H, I, _ptr(_u8(qx)), ctypes.c_float(float(sx)), _ptr(qg), _ptr(_f32(sg)), _ptr(qu),
                                _ptr(_f32(su)), _ptr(qd), _ptr(_f32(sd)), _ptr(y))
    return y


def shared_row_fp8(w, qx, sx, q) -> np.ndarray:
    """Sum of the shared experts on one token in FP8; q holds qsg, ssg, qsu, ssu, qsd, ssd."""
    y = np.empty(w.hidden, dtype=np.float64)
    lib().oracle_shared_row_fp8(ctypes.byref(shape_of(w)), _ptr(_u8(qx)), ctypes.c_float(float(sx)),
                                _ptr(_u8(q["qsg"])), _ptr(_f32(q["ssg"])), _ptr(_u8(q["qsu"])), _ptr(_f32(q["ssu"])),
                                _ptr(_u8(q["qsd"])), _ptr(_f32(q["ssd"])), _ptr(y))
    return y


def shared_down_matrix(ws_down):
    """The shared experts' down weights [n_sh, H, I_sh] as one matrix [H, n_sh*I_sh]
    (expert j's columns at j*I_sh): the shared outputs are summed, so this
    matrix times the concatenated intermediate is their sum."""
    n_sh, H, Is = ws_down.shape
    return ws_down.permute(1, 0, 2).reshape(H, n_sh * Is).contiguous()


def quantize_layer_fp8(w, w_gate, w_up, w_down, ws_gate, ws_up, ws_down) -> dict:
    """E4M3 codes and per-output-row scales of every expert matrix of the FP8
    layer: routed gate/up [S*I, H] rows, routed down [S*H, I] rows, shared
    gate/up [n_sh*I_sh, H] rows, shared down as one [H, n_sh*I_sh] matrix."""
    H, I = w.hidden, w.inter
    q = {}
    q["qg"], q["sg"] = quantize_rows_e4m3(w_gate.reshape(-1, H))
    q["qu"], q["su"] = quantize_rows_e4m3(w_up.reshape(-1, H))
    q["qd"], q["sd"] = quantize_rows_e4m3(w_down.reshape(-1, I))
    if w.n_shared > 0:
        q["qsg"], q["ssg"] = quantize_rows_e4m3(ws_gate.reshape(-1, H))
        q["qsu"], q["ssu"] = quantize_rows_e4m3(ws_up.reshape(-1, H))
        q["qsd"], q["ssd"] = quantize_rows_e4m3(shared_down_matrix(ws_down))
    else:
        for k_, dt in (("qsg", np.uint8), ("qsu", np.uint8), ("qsd", np.uint8)):
            q[k_] = np.zeros(16, dt)
        for k_ in ("ssg", "ssu", "ssd"):
            q[k_] = np.ones(16, np.float32)
    return q


def moe_forward_fp8(w, x, w_router, bias, replica_of, q):
    """Layer in FP8 (payloads and every expert matrix); q as quantize_layer_fp8 returns.

    Also returns the combine weights [T,k], inv_perm [T*k] and the E4M3 combine
    payload (y_codes [T*k, H], y_scale [T*k, nb], rows in dispatch order)."""
    T = x.shape[0]
    n = T * w.top_k
    nb = (w.hidden + PAYLOAD_BLOCK - 1) // PAYLOAD_BLOCK
    idx = np.empty((T, w.top_k), np.int32)
    out = np.empty((T, w.hidden), np.float64)
    weight = np.empty((T, w.top_k), np.float64)
    inv = np.empty(n, np.int32)
    y_codes = np.empty((n, w.hidden), np.uint8)
    y_scale = np.empty((n, nb), np.float32)
    a = {k_: (_u8(q[k_]) if k_.startswith("q") else _f32(q[k_]))
         for k_ in ("qg", "sg", "qu", "su", "qd", "sd", "qsg", "ssg", "qsu", "ssu", "qsd", "ssd")}
    invalid = lib().oracle_moe_forward_fp8_payload(
        ctypes.byref(shape_of(w)), T, _ptr(_u16(x)), _ptr(_u16(w_router)), _ptr(_f32(bias)),
        _ptr(_i32(replica_of)), *(_ptr(a[k_]) for k_ in ("qg", "sg", "qu", "su", "qd", "sd", "qsg", "ssg", "qsu",
                                                        "ssu", "qsd", "ssd")),
        _ptr(idx), _ptr(out), _ptr(weight), _ptr(inv), _ptr(y_codes), _ptr(y_scale))
    return dict(idx=idx, out=out, invalid=invalid, weight=weight, inv_perm=inv, y_codes=y_codes, y_scale=y_scale)
