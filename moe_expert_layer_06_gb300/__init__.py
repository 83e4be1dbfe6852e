"""Python binding of libmoe (include/moe.h): argument marshalling only.

Every function here has the name of a C entry point and forwards torch
tensors (device memory owned by the caller) as raw pointers, plus the current
torch CUDA stream.  Every step of the MoE layer runs in libmoe's CUDA
kernels; there is no fallback path: if libmoe.so is missing or a call fails,
an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_DEVICE_TIMEOUT = 4
MOE_ERR_DEVICE_STATUS = 5
MOE_ERR_WORKSPACE = 6

MOE_FFN_AUTO = 0
MOE_FFN_DECODE = 1
MOE_FFN_PREFILL = 2

# every symbol include/moe.h declares
EXPORTS = (
    "moe_last_error_string", "moe_abi_version", "moe_check_status", "moe_set_wait_limit_ns",
    "moe_debug_expire_wait", "moe_route_workspace_size", "moe_route", "moe_expert_histogram",
    "moe_eplb_imbalance", "moe_eplb_plan_replicas", "moe_dispatch", "moe_expert_gate_up",
    "moe_expert_down", "moe_ffn_workspace_size", "moe_expert_ffn", "moe_combine",
    "moe_workspace_size", "moe_forward", "moe_expert_ffn_noalloc", "moe_route_grouped",
    "moe_eplb_window_bytes", "moe_eplb_window_reset", "moe_eplb_window_push", "moe_eplb_stable_table",
    "moe_eplb_copy_replicas", "moe_quantize_rows_fp8", "moe_dispatch_fp8", "moe_expert_gate_up_fp8",
    "moe_workspace_size_fp8", "moe_forward_fp8", "moe_expert_down_fp8", "moe_dispatch_workspace_size",
    "moe_expert_down_fp8_payload", "moe_combine_fp8", "moe_ep_plan", "moe_gather_rows",
)

# columns per scale of the E4M3 combine payload (MOE_PAYLOAD_BLOCK in include/moe.h)
MOE_PAYLOAD_BLOCK = 128

# capacity of the fixed scratch of moe_expert_ffn_noalloc (include/moe.h)
MOE_FFN_NOALLOC_SCRATCH_BYTES = 8 << 20


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libmoe error {code}: {msg}")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "inter", "n_experts", "top_k", "n_shared", "inter_shared", "n_slots", "n_blocks")]

    @classmethod
    def of(cls, w) -> "Shape":
        """From any object with those attributes (e.g. a moe_inputs.Workload)."""
        return cls(w.hidden, w.inter, w.n_experts, w.top_k, w.n_shared, w.inter_shared, w.n_slots, w.n_blocks)


_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t
_SIG = {
    "moe_last_error_string": (ctypes.c_char_p, []),
    "moe_abi_version": (_I, []),
    "moe_check_status": (_I, [_P]),
    "moe_set_wait_limit_ns": (_I, [ctypes.c_uint64]),
    "moe_debug_expire_wait": (_I, [_P]),
    "moe_route_workspace_size": (_Z, [_P, _I]),
    "moe_route": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_route_grouped": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_expert_histogram": (_I, [_P, _I, _P, _P, _P, _P, _P]),
    "moe_eplb_imbalance": (ctypes.c_double, [_P, _I]),
    "moe_eplb_window_bytes": (_Z, [_P, _I]),
    "moe_eplb_window_reset": (_I, [_P, _I, _P, _Z, _P]),
    "moe_eplb_window_push": (_I, [_P, _I, _P, _Z, _P, _P, ctypes.c_double, _P, _P, _P, _P, _P]),
    "moe_eplb_stable_table": (_I, [_P, _P, _P, _P]),
    "moe_eplb_copy_replicas": (_I, [_P, _P, _P, _P, _P, _P, _P]),
    "moe_eplb_plan_replicas": (_I, [_P, _P, _I, _P]),
    "moe_dispatch_workspace_size": (_Z, [_P, _I]),
    "moe_dispatch": (_I, [_P, _I] + [_P] * 10 + [_P, _Z, _P]),
    "moe_expert_gate_up": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P]),
    "moe_expert_down": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _P]),
    "moe_ffn_workspace_size": (_Z, [_P, _I]),
    "moe_expert_ffn": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _Z, _P]),
    "moe_expert_ffn_noalloc": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P]),
    "moe_combine": (_I, [_P, _I, _P, _P, _P, _P, _P, _P]),
    "moe_quantize_rows_fp8": (_I, [_I, _I, _P, _P, _P, _P]),
    "moe_dispatch_fp8": (_I, [_P, _I] + [_P] * 13 + [_P, _Z, _P]),
    "moe_expert_gate_up_fp8": (_I, [_P, _I] + [_P] * 15 + [_I, _P]),
    "moe_workspace_size_fp8": (_Z, [_P, _I]),
    "moe_expert_down_fp8": (_I, [_P, _I] + [_P] * 11 + [_I, _P]),
    "moe_expert_down_fp8_payload": (_I, [_P, _I] + [_P] * 12 + [_I, _P]),
    "moe_combine_fp8": (_I, [_P, _I] + [_P] * 7),
    "moe_ep_plan": (_I, [_P, _I] + [_P] * 7 + [ctypes.c_int32, _P]),
    "moe_gather_rows": (_I, [_I, _I, _P, _P, _P, _P]),
    "moe_forward_fp8": (_I, [_P, _I] + [_P] * 21 + [_I, _P, _Z, _P]),
    "moe_workspace_size": (_Z, [_P, _I]),
    "moe_forward": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _Z, _P]),
}


def build_library(force: bool = False) -> str:
    """Compile libmoe.so in-tree (nvcc, sm_103a)."""
    import importlib
    return importlib.import_module(__name__ + ".build").build(force=force)


def lib() -> ctypes.CDLL:
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoe.so not built ({LIB_PATH}); run moe_expert_layer_06_gb300.build_library()")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIG.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def last_error() -> str:
    return lib().moe_last_error_string().decode()


def _check(code: int):
    if code != MOE_OK:
        raise MoeError(code, last_error())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, torch.Tensor):
        if t.numel() and not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
        if t.numel() and not t.is_cuda:  # the C ABI takes device pointers
            raise ValueError("tensor must be on a CUDA device")
        return t.data_ptr() if t.numel() else None
    raise TypeError(type(t))


def _stream(stream) -> Optional[int]:
    if stream is None:
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _shape(shape):
    return ctypes.byref(shape if isinstance(shape, Shape) else Shape.of(shape))


# ------------------------------------------------------------------ entry points

def moe_check_status(stream=None) -> int:
    return lib().moe_check_status(_stream(stream))


def moe_set_wait_limit_ns(ns: int):
    _check(lib().moe_set_wait_limit_ns(int(ns)))


def moe_debug_expire_wait(stream=None):
    _check(lib().moe_debug_expire_wait(_stream(stream)))


def moe_route_workspace_size(shape, T: int) -> int:
    return lib().moe_route_workspace_size(_shape(shape), T)


def moe_route(shape, T, x, w_router, bias, logits_in, logits_out, topk_idx, topk_w, ws, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(lib().moe_route(_shape(shape), T, _ptr(x), _ptr(w_router), _ptr(bias), _ptr(logits_in),
                           _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), _ptr(ws), ws_bytes, _stream(stream)))


def moe_route_grouped(shape, T, n_groups, topk_groups, x, w_router, bias, logits_in, logits_out, topk_idx,
                      topk_w, ws, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(lib().moe_route_grouped(_shape(shape), T, n_groups, topk_groups, _ptr(x), _ptr(w_router), _ptr(bias),
                                   _ptr(logits_in), _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), _ptr(ws),
                                   ws_bytes, _stream(stream)))


def moe_expert_histogram(shape, T, topk_idx, replica_of, counts, block_counts, stream=None):
    _check(lib().moe_expert_histogram(_shape(shape), T, _ptr(topk_idx), _ptr(replica_of), _ptr(counts),
                                      _ptr(block_counts), _stream(stream)))


def moe_eplb_imbalance(block_counts) -> float:
    import numpy as np
    a = np.ascontiguousarray(block_counts, dtype=np.int32)
    return lib().moe_eplb_imbalance(a.ctypes.data, a.size)


def moe_eplb_plan_replicas(shape, expert_counts, n_rep: int):
    import numpy as np
    c = np.ascontiguousarray(expert_counts, dtype=np.int32)
    out = np.empty(shape.n_experts, dtype=np.int32)
    _check(lib().moe_eplb_plan_replicas(_shape(shape), c.ctypes.data, n_rep, out.ctypes.data))
    return out


def moe_eplb_window_bytes(shape, window: int) -> int:
    return lib().moe_eplb_window_bytes(_shape(shape), window)


def moe_eplb_window_reset(shape, window, state, stream=None):
    _check(lib().moe_eplb_window_reset(_shape(shape), window, _ptr(state), state.numel() * state.element_size(),
                                       _stream(stream)))


def moe_eplb_window_push(shape, window, state, counts, replica_of=None, threshold=1.2, block_load=None,
                         expert_load=None, ratio=None, trigger=None, stream=None):
    _check(lib().moe_eplb_window_push(_shape(shape), window, _ptr(state), state.numel() * state.element_size(),
                                      _ptr(counts), _ptr(replica_of), float(threshold), _ptr(block_load),
                                      _ptr(expert_load), _ptr(ratio), _ptr(trigger), _stream(stream)))


def moe_eplb_stable_table(shape, old, new):
    import numpy as np
    o = np.ascontiguousarray(old, dtype=np.int32) if old is not None else None
    n = np.ascontiguousarray(new, dtype=np.int32)
    out = np.empty(shape.n_experts, dtype=np.int32)
    _check(lib().moe_eplb_stable_table(_shape(shape), o.ctypes.data if o is not None else None, n.ctypes.data,
                                       out.ctypes.data))
    return out


def moe_eplb_copy_replicas(shape, old, new, w_gate, w_up, w_down, stream=None):
    import numpy as np
    o = np.ascontiguousarray(old, dtype=np.int32) if old is not None else None
    n = np.ascontiguousarray(new, dtype=np.int32)
    _check(lib().moe_eplb_copy_replicas(_shape(shape), o.ctypes.data if o is not None else None, n.ctypes.data,
                                        _ptr(w_gate), _ptr(w_up), _ptr(w_down), _stream(stream)))


def moe_dispatch_workspace_size(shape, T: int) -> int:
    return lib().moe_dispatch_workspace_size(_shape(shape), T)


def _dispatch_ws(shape, T, ws, like):
    """The caller's dispatch workspace, or a fresh one on the device of `like`."""
    if ws is not None:
        return ws
    n = moe_dispatch_workspace_size(shape, T)
    return torch.empty(n, dtype=torch.uint8, device=like.device) if n else None


def moe_dispatch(shape, T, x, topk_idx, replica_of, slot_of, counts, block_counts, offsets, perm, inv_perm,
                 x_disp, ws=None, stream=None):
    ws = _dispatch_ws(shape, T, ws, counts)
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(lib().moe_dispatch(_shape(shape), T, _ptr(x), _ptr(topk_idx), _ptr(replica_of), _ptr(slot_of),
                              _ptr(counts), _ptr(block_counts), _ptr(offsets), _ptr(perm), _ptr(inv_perm),
                              _ptr(x_disp), _ptr(ws), ws_bytes, _stream(stream)))


def moe_expert_gate_up(shape, T, x, x_disp, offsets, w_gate, w_up, ws_gate, ws_up, h_disp, h_shared,
                       mode=MOE_FFN_AUTO, stream=None):
    _check(lib().moe_expert_gate_up(_shape(shape), T, _ptr(x), _ptr(x_disp), _ptr(offsets), _ptr(w_gate),
                                    _ptr(w_up), _ptr(ws_gate), _ptr(ws_up), _ptr(h_disp), _ptr(h_shared), mode,
                                    _stream(stream)))


def moe_expert_down(shape, T, h_disp, h_shared, offsets, w_down, ws_down, y_disp, y_shared,
                    mode=MOE_FFN_AUTO, stream=None):
    _check(lib().moe_expert_down(_shape(shape), T, _ptr(h_disp), _ptr(h_shared), _ptr(offsets), _ptr(w_down),
                                 _ptr(ws_down), _ptr(y_disp), _ptr(y_shared), mode, _stream(stream)))


def moe_ffn_workspace_size(shape, T: int) -> int:
    return lib().moe_ffn_workspace_size(_shape(shape), T)


def moe_expert_ffn(shape, T, x, x_disp, offsets, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, y_disp,
                   y_shared, mode, ws, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(lib().moe_expert_ffn(_shape(shape), T, _ptr(x), _ptr(x_disp), _ptr(offsets), _ptr(w_gate),
                                _ptr(w_up), _ptr(w_down), _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down),
                                _ptr(y_disp), _ptr(y_shared), mode, _ptr(ws), ws_bytes, _stream(stream)))


def moe_expert_ffn_noalloc(shape, T, x, x_disp, offsets, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, y_disp,
                           y_shared, mode=MOE_FFN_AUTO, stream=None):
    """moe_expert_ffn for callers that cannot allocate: the intermediate lives in libmoe's fixed scratch."""
    _check(lib().moe_expert_ffn_noalloc(_shape(shape), T, _ptr(x), _ptr(x_disp), _ptr(offsets), _ptr(w_gate),
                                        _ptr(w_up), _ptr(w_down), _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down),
                                        _ptr(y_disp), _ptr(y_shared), mode, _stream(stream)))


def moe_combine(shape, T, y_disp, inv_perm, topk_w, y_shared, out, stream=None):
    _check(lib().moe_combine(_shape(shape), T, _ptr(y_disp), _ptr(inv_perm), _ptr(topk_w), _ptr(y_shared),
                             _ptr(out), _stream(stream)))


def moe_workspace_size(shape, T: int) -> int:
    return lib().moe_workspace_size(_shape(shape), T)


def moe_forward(shape, T, x, w_router, bias, replica_of, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, out,
                topk_idx_out=None, topk_w_out=None, counts_out=None, block_counts_out=None,
                mode=MOE_FFN_AUTO, ws=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(lib().moe_forward(_shape(shape), T, _ptr(x), _ptr(w_router), _ptr(bias), _ptr(replica_of),
                             _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down),
                             _ptr(out), _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(counts_out),
                             _ptr(block_counts_out), mode, _ptr(ws), ws_bytes, _stream(stream)))


# ------------------------------------------------------------------ FP8 path

def moe_quantize_rows_fp8(x, codes, scale, stream=None):
    rows = x.shape[0]
    cols = x.numel() // max(1, rows)
    _check(lib().moe_quantize_rows_fp8(rows, cols, _ptr(x), _ptr(codes), _ptr(scale), _stream(stream)))


def moe_dispatch_fp8(shape, T, x, topk_idx, replica_of, slot_of, counts, block_counts, offsets, perm, inv_perm,
                     x8, x_scale, x_disp8, x_disp_scale, ws=None, stream=None):
    ws = _dispatch_ws(shape, T, ws, counts)
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(lib().moe_dispatch_fp8(_shape(shape), T, _ptr(x), _ptr(topk_idx), _ptr(replica_of), _ptr(slot_of),
                                  _ptr(counts), _ptr(block_counts), _ptr(offsets), _ptr(perm), _ptr(inv_perm),
                                  _ptr(x8), _ptr(x_scale), _ptr(x_disp8), _ptr(x_disp_scale), _ptr(ws), ws_bytes,
                                  _stream(stream)))


def moe_expert_gate_up_fp8(shape, T, x8, x_scale, x_disp8, x_disp_scale, offsets, qg, sg, qu, su, qsg, ssg, qsu,
                           ssu, h_disp, h_shared, mode=MOE_FFN_AUTO, stream=None):
    _check(lib().moe_expert_gate_up_fp8(_shape(shape), T, _ptr(x8), _ptr(x_scale), _ptr(x_disp8),
                                        _ptr(x_disp_scale), _ptr(offsets), _ptr(qg), _ptr(sg), _ptr(qu), _ptr(su),
                                        _ptr(qsg), _ptr(ssg), _ptr(qsu), _ptr(ssu), _ptr(h_disp), _ptr(h_shared),
                                        mode, _stream(stream)))


def moe_expert_down_fp8(shape, T, h8, h_scale, hs8, hs_scale, offsets, qd, sd, qsd, ssd, y_disp, y_shared,
                        mode=MOE_FFN_AUTO, stream=None):
    _check(lib().moe_expert_down_fp8(_shape(shape), T, _ptr(h8), _ptr(h_scale), _ptr(hs8), _ptr(hs_scale),
                                     _ptr(offsets), _ptr(qd), _ptr(sd), _ptr(qsd), _ptr(ssd), _ptr(y_disp),
                                     _ptr(y_shared), mode, _stream(stream)))


def moe_expert_down_fp8_payload(shape, T, h8, h_scale, hs8, hs_scale, offsets, qd, sd, qsd, ssd, y_disp8,
                                y_disp_scale, y_shared, mode=MOE_FFN_AUTO, stream=None):
    _check(lib().moe_expert_down_fp8_payload(_shape(shape), T, _ptr(h8), _ptr(h_scale), _ptr(hs8), _ptr(hs_scale),
                                             _ptr(offsets), _ptr(qd), _ptr(sd), _ptr(qsd), _ptr(ssd), _ptr(y_disp8),
                                             _ptr(y_disp_scale), _ptr(y_shared), mode, _stream(stream)))


def moe_combine_fp8(shape, T, y_disp8, y_disp_scale, inv_perm, topk_w, y_shared, out, stream=None):
    _check(lib().moe_combine_fp8(_shape(shape), T, _ptr(y_disp8), _ptr(y_disp_scale), _ptr(inv_perm), _ptr(topk_w),
                                 _ptr(y_shared), _ptr(out), _stream(stream)))


def moe_workspace_size_fp8(shape, T: int) -> int:
    return lib().moe_workspace_size_fp8(_shape(shape), T)


def moe_forward_fp8(shape, T, x, w_router, bias, replica_of, qg, sg, qu, su, qd, sd, qsg, ssg, qsu, ssu, qsd, ssd,
                    out, topk_idx_out=None, topk_w_out=None, counts_out=None, block_counts_out=None,
                    mode=MOE_FFN_AUTO, ws=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(lib().moe_forward_fp8(_shape(shape), T, _ptr(x), _ptr(w_router), _ptr(bias), _ptr(replica_of),
                                 _ptr(qg), _ptr(sg), _ptr(qu), _ptr(su), _ptr(qd), _ptr(sd), _ptr(qsg), _ptr(ssg),
                                 _ptr(qsu), _ptr(ssu), _ptr(qsd), _ptr(ssd), _ptr(out), _ptr(topk_idx_out),
                                 _ptr(topk_w_out), _ptr(counts_out), _ptr(block_counts_out), mode, _ptr(ws),
                                 ws_bytes, _stream(stream)))


# ------------------------------------------------------------------ EP across GPUs (bookkeeping)

def moe_ep_plan(shape, world: int, counts, recv_counts, maps: bool = True):
    """Host plan of the two all-to-alls of one EP rank (include/moe.h).

    counts: this rank's dispatch counts [n_slots+1]; recv_counts: [world, spb]
    rows each source sends for each local slot.  Returns a dict of numpy int32
    arrays: send_rows, recv_rows, local_offsets and (maps) slot_from_src,
    src_from_slot, plus rows (R)."""
    import numpy as np
    spb = shape.n_slots // world
    c = np.ascontiguousarray(np.asarray(counts).reshape(-1), dtype=np.int32)
    rc_ = np.ascontiguousarray(np.asarray(recv_counts).reshape(-1), dtype=np.int32)
    assert c.size == shape.n_slots + 1 and rc_.size == world * spb
    send, recv = np.empty(world, np.int32), np.empty(world, np.int32)
    loc = np.empty(spb + 2, np.int32)
    R = int(rc_.sum())
    sfs = np.empty(max(1, R), np.int32) if maps else None
    ssf = np.empty(max(1, R), np.int32) if maps else None
    rows = ctypes.c_int32()
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p) if a is not None else None
    _check(lib().moe_ep_plan(_shape(shape), world, p(c), p(rc_), p(send), p(recv), p(loc), p(sfs), p(ssf),
                             max(1, R), ctypes.byref(rows)))
    out = dict(send_rows=send, recv_rows=recv, local_offsets=loc, rows=rows.value)
    if maps:
        out["slot_from_src"], out["src_from_slot"] = sfs[:R], ssf[:R]
    return out


def moe_gather_rows(src, index, dst, stream=None):
    """dst[i] = src[index[i]] for rows of src (device tensors, rows of a multiple of 16 bytes)."""
    n = index.numel()
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] else dst[0].numel() * dst.element_size()
    _check(lib().moe_gather_rows(n, row_bytes, _ptr(src), _ptr(index), _ptr(dst), _stream(stream)))
