"""The C-ABI library without a GPU: it loads, exports every declared symbol,
validates arguments before touching the device, and its host-only EPLB helpers
agree with the oracle."""
import ctypes
import os
import re

import numpy as np
import torch
import pytest

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")
FAKE = 0x10000  # 16-byte aligned address that is never dereferenced on the host


@pytest.fixture(scope="module", autouse=True)
def built():
    m.build_library()


def _declared():
    src = open(HEADER).read()
    return re.findall(r"^MOE_API [^(]*?\b(moe_\w+)\(", src, flags=re.M)


def test_library_exports_every_declared_symbol():
    names = _declared()
    assert len(names) >= 18
    lib = ctypes.CDLL(m.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(m.EXPORTS)
    assert m.lib().moe_abi_version() == 1


def test_binding_signatures_match_the_header():
    """Every ctypes signature has as many arguments as the declaration, and
    integer parameters sit where the header has int / size_t / double."""
    src = open(HEADER).read()
    decls = re.findall(r"^MOE_API [^(]*?\b(moe_\w+)\(([^;]*?)\);", src, flags=re.M | re.S)
    assert len(decls) == len(m.EXPORTS)
    kinds = {"int": ctypes.c_int, "size_t": ctypes.c_size_t, "double": ctypes.c_double, "uint64_t": ctypes.c_uint64,
             "int32_t": ctypes.c_int32}
    for name, params in decls:
        params = " ".join(params.split())
        plist = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
        sig = m._SIG[name][1]
        assert len(sig) == len(plist), (name, len(sig), len(plist))
        for p, t in zip(plist, sig):
            if "*" in p:
                assert t is ctypes.c_void_p, (name, p)
            else:
                base = p.rsplit(" ", 1)[0].replace("const ", "").strip()
                assert t is kinds[base], (name, p)


def _shape(**kw):
    return m.Shape.of(mi.WORKLOADS["decode_t32"].with_(**kw))


def test_shape_validation_codes():
    L = m.lib()
    buf = ctypes.c_void_p(FAKE)
    assert L.moe_route(None, 4, buf, buf, None, None, None, buf, buf, buf, 1 << 30, None) == m.MOE_ERR_INVALID_ARG
    assert "shape" in m.last_error()
    cases = [
        (dict(top_k=300), m.MOE_ERR_INVALID_ARG),     # k > E
        (dict(top_k=33, n_experts=64, n_slots=64), m.MOE_ERR_INVALID_ARG),  # k > 32
        (dict(hidden=7170), m.MOE_ERR_INVALID_ARG),   # H % 8
        (dict(inter=2050), m.MOE_ERR_INVALID_ARG),
        (dict(n_slots=260), m.MOE_ERR_INVALID_ARG),   # S % blocks
        (dict(n_slots=128, n_experts=256), m.MOE_ERR_INVALID_ARG),
        (dict(n_experts=2048, n_slots=2048), m.MOE_ERR_UNSUPPORTED),
        (dict(n_slots=1032), m.MOE_ERR_UNSUPPORTED),
        (dict(n_blocks=0), m.MOE_ERR_INVALID_ARG),
    ]
    for kw, code in cases:
        s = _shape(**kw)
        rc = L.moe_route(ctypes.byref(s), 4, buf, buf, None, None, None, buf, buf, buf, 1 << 30, None)
        assert rc == code, (kw, rc, m.last_error())
    s = _shape()
    assert L.moe_route(ctypes.byref(s), -1, buf, buf, None, None, None, buf, buf, buf, 0, None) == m.MOE_ERR_INVALID_ARG


def test_pointer_and_workspace_validation_codes():
    L = m.lib()
    s = _shape()
    b = ctypes.c_void_p(FAKE)
    mis = ctypes.c_void_p(FAKE + 2)
    # null / misaligned
    assert L.moe_route(ctypes.byref(s), 4, None, b, None, None, None, b, b, b, 1 << 30, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_route(ctypes.byref(s), 4, mis, b, None, None, None, b, b, b, 1 << 30, None) == m.MOE_ERR_INVALID_ARG
    assert "aligned" in m.last_error()
    # logits_in together with bias
    assert L.moe_route(ctypes.byref(s), 4, None, None, b, b, None, b, b, None, 0, None) == m.MOE_ERR_INVALID_ARG
    # workspace too small
    need = L.moe_route_workspace_size(ctypes.byref(s), 4)
    assert need > 0
    assert L.moe_route(ctypes.byref(s), 4, b, b, None, None, None, b, b, b, need - 1, None) == m.MOE_ERR_WORKSPACE
    fw = L.moe_workspace_size(ctypes.byref(s), 32)
    assert fw > 32 * 8 * 7168 * 2 * 2
    args = [ctypes.byref(s), 32] + [b] * 11 + [None] * 4 + [0, b, fw - 1, None]
    assert L.moe_forward(*args) == m.MOE_ERR_WORKSPACE
    args = [ctypes.byref(s), 32] + [b] * 11 + [None] * 4 + [7, b, fw, None]
    assert L.moe_forward(*args) == m.MOE_ERR_INVALID_ARG  # bad mode
    assert L.moe_ffn_workspace_size(ctypes.byref(s), 32) == 32 * 8 * 2048 * 2 + 32 * 2 * 2048 * 2
    # combine: null output
    assert L.moe_combine(ctypes.byref(s), 4, b, b, b, None, None, None) == m.MOE_ERR_INVALID_ARG
    # dispatch workspace: none below 4096 assignments, one histogram row of S+1 ints per 512-assignment chunk above
    assert L.moe_dispatch_workspace_size(ctypes.byref(s), 511) == 0
    assert L.moe_dispatch_workspace_size(ctypes.byref(s), 512) == ((8 * 257 * 4 + 255) // 256) * 256
    assert L.moe_dispatch_workspace_size(ctypes.byref(s), 4096) == ((64 * 257 * 4 + 255) // 256) * 256
    assert L.moe_dispatch_workspace_size(ctypes.byref(s), 65536) == ((128 * 257 * 4 + 255) // 256) * 256
    need = L.moe_dispatch_workspace_size(ctypes.byref(s), 4096)
    args = [ctypes.byref(s), 4096] + [b] * 10
    assert L.moe_dispatch(*args, None, 0, None) == m.MOE_ERR_WORKSPACE
    assert L.moe_dispatch(*args, b, need - 1, None) == m.MOE_ERR_WORKSPACE
    assert L.moe_dispatch(*args, mis, need, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch_fp8(ctypes.byref(s), 4096, *([b] * 13), None, 0, None) == m.MOE_ERR_WORKSPACE
    fw8 = L.moe_workspace_size_fp8(ctypes.byref(s), 4096)
    fw = L.moe_workspace_size(ctypes.byref(s), 4096)
    n = 4096 * 8
    # the E4M3 forward holds both E4M3 payloads (dispatch: n*H codes; combine: n*H codes and n*56 block
    # scales) in place of the bf16 combine payload (n*H*2 bytes)
    assert fw8 >= fw - n * 7168 * 2 + 2 * n * 7168 + n * 56 * 4
    assert fw8 < fw + n * 7168


def test_empty_batch_is_a_no_op():
    L = m.lib()
    s = _shape()
    assert L.moe_route(ctypes.byref(s), 0, None, None, None, None, None, None, None, None, 0, None) == m.MOE_OK
    assert L.moe_combine(ctypes.byref(s), 0, None, None, None, None, None, None) == m.MOE_OK
    assert L.moe_expert_gate_up(ctypes.byref(s), 0, *([None] * 9), 0, None) == m.MOE_OK
    assert L.moe_expert_down(ctypes.byref(s), 0, *([None] * 7), 0, None) == m.MOE_OK
    assert L.moe_forward(ctypes.byref(s), 0, *([None] * 15), 0, None, 0, None) == m.MOE_OK
    assert L.moe_workspace_size(ctypes.byref(s), 0) == 0 or L.moe_workspace_size(ctypes.byref(s), 0) < 4096


def test_wait_limit_setter():
    assert m.lib().moe_set_wait_limit_ns(0) == m.MOE_ERR_INVALID_ARG
    assert m.lib().moe_set_wait_limit_ns(2_000_000_000) == m.MOE_OK


def test_imbalance_ratio():
    assert m.moe_eplb_imbalance([10, 10, 10, 10]) == 1.0
    assert m.moe_eplb_imbalance([0, 0]) == 0.0
    assert abs(m.moe_eplb_imbalance([30, 10, 10, 10]) - 2.0) < 1e-12


def test_replica_plan_agrees_with_oracle():
    rng = np.random.default_rng(1)
    w = mi.WORKLOADS["redundant_t1024"]
    for trial in range(200):
        if trial % 3 == 0:
            counts = rng.integers(0, 5, size=w.n_experts)      # many ties
        elif trial % 3 == 1:
            counts = (rng.pareto(1.2, size=w.n_experts) * 20).astype(np.int64)
        else:
            counts = np.zeros(w.n_experts, dtype=np.int64)
            counts[rng.choice(32, 8, replace=False)] = rng.integers(1, 100, size=8)  # all hot in block 0
        n_rep = int(rng.integers(0, 9))
        got = m.moe_eplb_plan_replicas(w, counts, n_rep)
        want = oracle.plan_replicas(w, counts, n_rep)
        assert np.array_equal(got, want), (trial, counts, n_rep)
    tiny = mi.WORKLOADS["tiny"].with_(n_blocks=4, n_slots=12)
    got = m.moe_eplb_plan_replicas(tiny, np.array([10, 1, 7, 0, 3, 3, 9, 2]), 3)
    assert list(got) == [5, -1, 8, -1, -1, -1, 2, -1]
    with pytest.raises(m.MoeError):
        m.moe_eplb_plan_replicas(tiny, np.zeros(8), 5)


def test_grouped_route_argument_checks():
    L = m.lib()
    s = _shape()  # E = 256, k = 8
    b = ctypes.c_void_p(FAKE)
    for G, Gk in ((0, 1), (33, 1), (3, 1), (8, 0), (8, 9), (64, 1)):
        rc = L.moe_route_grouped(ctypes.byref(s), 4, G, Gk, b, b, None, None, None, b, b, b, 1 << 30, None)
        assert rc == m.MOE_ERR_INVALID_ARG, (G, Gk)
    s2 = _shape(n_experts=32, n_slots=32, top_k=8)  # groups of 4: k=8 needs 2 groups
    rc = L.moe_route_grouped(ctypes.byref(s2), 4, 8, 1, b, b, None, None, None, b, b, b, 1 << 30, None)
    assert rc == m.MOE_ERR_INVALID_ARG and "top_k" in m.last_error()
    assert L.moe_route_grouped(ctypes.byref(s), 0, 8, 4, None, None, None, None, None, None, None, None, 0,
                               None) == m.MOE_OK


def test_eplb_window_and_migration_argument_checks():
    L = m.lib()
    w = mi.WORKLOADS["redundant_t1024"]
    s = _shape(n_slots=264)
    b = ctypes.c_void_p(FAKE)
    n1 = L.moe_eplb_window_bytes(ctypes.byref(s), 1)
    n4 = L.moe_eplb_window_bytes(ctypes.byref(s), 4)
    assert n1 > 0 and n4 - n1 >= 3 * 265 * 4 - 16 and L.moe_eplb_window_bytes(ctypes.byref(s), 0) == 0
    assert L.moe_eplb_window_reset(ctypes.byref(s), 0, b, n4, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_eplb_window_reset(ctypes.byref(s), 4, None, n4, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_eplb_window_reset(ctypes.byref(s), 4, b, n4 - 1, None) == m.MOE_ERR_WORKSPACE
    push = lambda win, st, nb, cnt, thr: L.moe_eplb_window_push(ctypes.byref(s), win, st, nb, cnt, None, thr,
                                                                None, None, None, None, None)
    assert push(4, b, n4, None, 1.2) == m.MOE_ERR_INVALID_ARG
    assert push(4, b, n4, b, 0.0) == m.MOE_ERR_INVALID_ARG
    assert push(4, b, n1, b, 1.2) == m.MOE_ERR_WORKSPACE
    assert push(4, ctypes.c_void_p(FAKE + 4), n4, b, 1.2) == m.MOE_ERR_INVALID_ARG
    # stable table: keep replicas both plans agree on
    old = np.full(256, -1, np.int32)
    new = np.full(256, -1, np.int32)
    old[[3, 40, 77]] = [65, 98, 131]
    new[[3, 40, 90]] = [65, 131, 98]
    st = m.moe_eplb_stable_table(w, old, new)
    assert list(np.flatnonzero(st >= 0)) == [3] and st[3] == 65
    assert list(m.moe_eplb_stable_table(w, None, new)) == [-1] * 256
    # copies are validated before anything is enqueued
    bad = new.copy()
    bad[5] = 34   # a home slot (block 1 holds experts 32..63 in slots 33..64)
    with pytest.raises(m.MoeError):
        m.moe_eplb_copy_replicas(w, old, bad, FAKE, FAKE, FAKE)
    dup = new.copy()
    dup[7] = 65
    with pytest.raises(m.MoeError):
        m.moe_eplb_copy_replicas(w, old, dup, FAKE, FAKE, FAKE)


def test_workspace_sizes_never_shrink_as_the_batch_grows():
    """A workspace sized for the largest batch serves every smaller one."""
    for name in ("tiny", "decode_t32", "redundant_t1024", "decode_t32_e1024"):
        w = mi.WORKLOADS[name]
        for fn in (m.moe_workspace_size, m.moe_workspace_size_fp8, m.moe_route_workspace_size,
                   m.moe_ffn_workspace_size, m.moe_dispatch_workspace_size):
            sizes = [fn(w, T) for T in range(0, 5000)]
            drops = [T for T in range(1, len(sizes)) if sizes[T] < sizes[T - 1]]
            assert not drops, (name, fn.__name__, drops[:3])


def test_binding_refuses_host_and_strided_tensors_before_calling_the_library():
    w = mi.WORKLOADS["tiny"]
    T, H = w.tokens, w.hidden
    host = torch.zeros((T * w.top_k, H), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA device"):
        m.moe_combine(w, T, host, None, None, None, torch.zeros((T, H), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="contiguous"):
        m.moe_combine(w, T, host.t(), None, None, None, None)


def test_fp8_argument_checks():
    L = m.lib()
    b = ctypes.c_void_p(FAKE)
    # the row quantiser: rows >= 0, cols a positive multiple of 16; no rows is a no-op
    assert L.moe_quantize_rows_fp8(-1, 64, b, b, b, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_rows_fp8(4, 24, b, b, b, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_rows_fp8(0, 64, None, None, None, None) == m.MOE_OK
    # one-byte rows need H, I and n_sh*I_sh multiples of 16 (the bf16 path needs 8)
    h8 = _shape(hidden=7176)
    i8 = _shape(inter=2056)
    sh8 = _shape(n_shared=1, inter_shared=2056)
    assert L.moe_dispatch_fp8(ctypes.byref(h8), 32, *([b] * 13), None, 0, None) == m.MOE_ERR_INVALID_ARG
    assert "16" in m.last_error()
    assert L.moe_expert_gate_up_fp8(ctypes.byref(h8), 32, *([b] * 15), 0, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_expert_down_fp8(ctypes.byref(i8), 32, *([b] * 11), 0, None) == m.MOE_ERR_INVALID_ARG
    assert L.moe_expert_down_fp8(ctypes.byref(sh8), 32, *([b] * 11), 0, None) == m.MOE_ERR_INVALID_ARG
    for s in (h8, i8, sh8):
        assert L.moe_forward_fp8(ctypes.byref(s), 32, *([b] * 21), 0, b, 1 << 40, None) == m.MOE_ERR_INVALID_ARG
    ok = _shape()
    assert L.moe_forward_fp8(ctypes.byref(ok), 32, *([b] * 21), 9, b, 1 << 40, None) == m.MOE_ERR_INVALID_ARG
    assert "mode" in m.last_error()
