"""moe_expert_ffn_noalloc: the expert FFN for callers that cannot allocate device
memory (a plugin whose host program owns every allocation, or a path that cannot
afford cudaMalloc's implicit synchronisation).  Its SwiGLU intermediate lives in a
fixed array inside libmoe instead of a caller workspace.  Both entry points run
the same kernels on the same inputs, so the results must be bit-identical to
moe_expert_ffn's, call after call, although every call reuses the same array:
a larger batch followed by a smaller one (a stale tail of the array, and the
shared intermediate moved to a new offset, must not leak into the result), and
a batch whose intermediate fills the array to its last byte.  On the mid shape
the result is also checked against the fp64 oracle.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle
from moe_testlib import assert_close, to_np

DEV = "cuda"

MID = mi.WORKLOADS["tiny"].with_(name="mid", tokens=100, hidden=600, inter=328, n_experts=16, top_k=4,
                                 n_shared=2, inter_shared=200, n_slots=16, n_blocks=4)
# T=1024 tokens x (8 x 256 routed + 2 x 1024 shared) intermediate columns x 2 bytes = 8 MiB:
# the intermediate of the largest batch this shape accepts ends on the array's last byte
FULL = mi.WORKLOADS["tiny"].with_(name="fills_scratch", tokens=1024, hidden=256, inter=256, n_experts=16, top_k=8,
                                  n_shared=2, inter_shared=1024, n_slots=16, n_blocks=4)


def _intermediate_bytes(w, T):
    h = T * w.top_k * w.inter * 2
    return ((h + 255) & ~255) + T * w.n_shared * w.inter_shared * 2


def test_noalloc_rejects_batches_beyond_its_scratch():
    m.build_library()
    b = ctypes.c_void_p(0x10000)
    for w, t_max in ((mi.WORKLOADS["decode_t32"], 204), (FULL, 1024)):
        s = m.Shape.of(w)
        assert _intermediate_bytes(w, t_max) <= m.MOE_FFN_NOALLOC_SCRATCH_BYTES
        assert _intermediate_bytes(w, t_max + 1) > m.MOE_FFN_NOALLOC_SCRATCH_BYTES
        rc = m.lib().moe_expert_ffn_noalloc(ctypes.byref(s), t_max + 1, *([b] * 11), 0, None)
        assert rc == m.MOE_ERR_UNSUPPORTED
        assert "scratch" in m.last_error()
    assert _intermediate_bytes(FULL, 1024) == m.MOE_FFN_NOALLOC_SCRATCH_BYTES


def _batch(w, T, seed_offset):
    """T tokens of workload w (inputs vary with seed_offset), routed by the oracle
    and dispatched through libmoe; the oracle's own dispatch is returned too."""
    k, S = w.top_k, w.n_slots
    wx = w.with_(tokens=T, seed=w.seed + seed_offset)
    x = mi.hidden_states(wx)
    lo = oracle.router_logits(wx, x, mi.router_weight(w), None)
    idx, _ = oracle.topk_softmax(lo, k)
    n = T * k
    i32 = dict(dtype=torch.int32, device=DEV)
    offsets = torch.empty(S + 2, **i32)
    x_disp = torch.empty((n, w.hidden), dtype=torch.bfloat16, device=DEV)
    xd = x.to(DEV)
    m.moe_dispatch(wx, T, xd, torch.from_numpy(idx).to(DEV), None, torch.empty(n, **i32), torch.empty(S + 1, **i32),
                   None, offsets, torch.empty(n, **i32), torch.empty(n, **i32), x_disp)
    so, _ = oracle.slot_map(wx, idx)
    counts, _ = oracle.histogram(wx, so)
    off_o, _, _, xd_o = oracle.dispatch(wx, T, so, counts, x)
    return xd, x_disp, offsets, x, off_o, xd_o


@pytest.mark.gpu
@pytest.mark.parametrize("name,batches", [("mid", (100, 37)), ("decode_t32", (32, 7)),
                                          ("fills_scratch", (1024, 300))])
def test_noalloc_matches_workspace_entry_point_twice_in_a_row(name, batches):
    m.build_library()
    w = {"mid": MID, "fills_scratch": FULL}.get(name) or mi.WORKLOADS[name]
    H = w.hidden
    wg, wu, wd = mi.stacked_expert_weights(w, device=DEV)
    sg, su, sd = mi.stacked_shared_weights(w, device=DEV)
    ws = torch.empty(m.moe_ffn_workspace_size(w, max(batches)), dtype=torch.uint8, device=DEV)
    for call, T in enumerate(batches):  # a larger batch, then a smaller one, sharing the fixed scratch
        x, x_disp, offsets, x_cpu, off_o, xd_o = _batch(w, T, call)
        assert np.array_equal(offsets.cpu().numpy(), off_o)
        y_ref = torch.empty((T * w.top_k, H), dtype=torch.bfloat16, device=DEV)
        ys_ref = torch.empty((T, H), dtype=torch.float32, device=DEV)
        m.moe_expert_ffn(w, T, x, x_disp, offsets, wg, wu, wd, sg, su, sd, y_ref, ys_ref, m.MOE_FFN_AUTO, ws)
        y = torch.full_like(y_ref, float("nan"))
        ys = torch.full_like(ys_ref, float("nan"))
        m.moe_expert_ffn_noalloc(w, T, x, x_disp, offsets, wg, wu, wd, sg, su, sd, y, ys, m.MOE_FFN_AUTO)
        assert m.moe_check_status() == m.MOE_OK, m.last_error()
        assert torch.equal(y, y_ref), f"{name} call {call} (T={T}): y_disp differs from moe_expert_ffn's"
        assert torch.equal(ys, ys_ref), f"{name} call {call} (T={T}): y_shared differs from moe_expert_ffn's"
        if name == "mid":  # and the oracle on the same dispatched rows
            y_o = oracle.expert_ffn(w, T, off_o, xd_o, wg.cpu(), wu.cpu(), wd.cpu())
            assert_close(to_np(y), y_o, what=f"mid call {call} y_disp vs oracle")
            ys_o = oracle.shared_rows(w, x_cpu, sg.cpu(), su.cpu(), sd.cpu())
            assert_close(ys.cpu().numpy().astype(np.float64), ys_o, what=f"mid call {call} y_shared vs oracle",
                         bf16_out=False)
    del wg, wu, wd
    torch.cuda.empty_cache()
