"""moe_expert_ffn_noalloc: the expert FFN for callers that cannot allocate device
memory (a plugin whose host program owns every allocation, or a path that cannot
afford cudaMalloc's implicit synchronisation).  Its SwiGLU intermediate lives in a
fixed array inside libmoe instead of a caller workspace; its results must match
moe_expert_ffn's, call after call, although every call reuses the same array.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process."""
import ctypes

import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
from moe_testlib import assert_close

DEV = "cuda"

MID = mi.WORKLOADS["tiny"].with_(name="mid", tokens=100, hidden=600, inter=328, n_experts=16, top_k=4,
                                 n_shared=2, inter_shared=200, n_slots=16, n_blocks=4)


def test_noalloc_rejects_batches_beyond_its_scratch():
    m.build_library()
    w = mi.WORKLOADS["decode_t32"]
    s = m.Shape.of(w)
    b = ctypes.c_void_p(0x10000)
    rc = m.lib().moe_expert_ffn_noalloc(ctypes.byref(s), 205, *([b] * 11), 0, None)
    assert rc == m.MOE_ERR_UNSUPPORTED
    assert "scratch" in m.last_error()
    assert 204 * (8 * 2048 * 2 + 2 * 2048 * 2) <= m.MOE_FFN_NOALLOC_SCRATCH_BYTES


def _routed_inputs(w, seed_offset):
    """Routing and dispatch through libmoe for a batch of workload w (inputs vary with seed_offset)."""
    T, k = w.tokens, w.top_k
    wx = w.with_(seed=w.seed + seed_offset)
    x = mi.hidden_states(wx, device=DEV)
    wr = mi.router_weight(w, device=DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    rws = torch.empty(max(16, m.moe_route_workspace_size(w, T)), dtype=torch.uint8, device=DEV)
    m.moe_route(w, T, x, wr, None, None, None, idx, tw, rws)
    n, S = T * k, w.n_slots
    i32 = dict(dtype=torch.int32, device=DEV)
    offsets = torch.empty(S + 2, **i32)
    x_disp = torch.empty((n, w.hidden), dtype=torch.bfloat16, device=DEV)
    m.moe_dispatch(w, T, x, idx, None, torch.empty(n, **i32), torch.empty(S + 1, **i32), None, offsets,
                   torch.empty(n, **i32), torch.empty(n, **i32), x_disp)
    return x, x_disp, offsets


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["mid", "decode_t32"])
def test_noalloc_matches_workspace_entry_point_twice_in_a_row(name):
    m.build_library()
    w = MID if name == "mid" else mi.WORKLOADS[name]
    T, H = w.tokens, w.hidden
    wg, wu, wd = mi.stacked_expert_weights(w, device=DEV)
    sg, su, sd = mi.stacked_shared_weights(w, device=DEV)
    ws = torch.empty(m.moe_ffn_workspace_size(w, T), dtype=torch.uint8, device=DEV)
    for call in range(2):  # two calls in a row, on different batches, sharing the fixed scratch
        x, x_disp, offsets = _routed_inputs(w, call)
        y_ref = torch.empty((T * w.top_k, H), dtype=torch.bfloat16, device=DEV)
        ys_ref = torch.empty((T, H), dtype=torch.float32, device=DEV)
        m.moe_expert_ffn(w, T, x, x_disp, offsets, wg, wu, wd, sg, su, sd, y_ref, ys_ref, m.MOE_FFN_AUTO, ws)
        y = torch.full_like(y_ref, float("nan"))
        ys = torch.full_like(ys_ref, float("nan"))
        m.moe_expert_ffn_noalloc(w, T, x, x_disp, offsets, wg, wu, wd, sg, su, sd, y, ys, m.MOE_FFN_AUTO)
        assert m.moe_check_status() == m.MOE_OK, m.last_error()
        assert_close(y.float().cpu().numpy(), y_ref.float().cpu().numpy(), what=f"{name} call {call} y_disp")
        assert_close(ys.cpu().numpy(), ys_ref.cpu().numpy(), what=f"{name} call {call} y_shared", bf16_out=False)
    del wg, wu, wd
    torch.cuda.empty_cache()
