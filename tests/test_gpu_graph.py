"""moe_forward enqueues kernels only (no host sync, no allocation), so a
serving loop can capture it once in a CUDA graph and replay it."""
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
from moe_testlib import DeviceLayer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "decode_t32"])
def test_forward_replays_from_a_cuda_graph(name):
    w = mi.WORKLOADS[name]
    layer = DeviceLayer(w, "cuda")
    T = w.tokens
    ref = layer.forward()["out"].clone()
    out = torch.empty_like(ref)
    ws = torch.empty(m.moe_workspace_size(w, T), dtype=torch.uint8, device="cuda")
    x_static = layer.x.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up call outside capture
        m.moe_forward(w, T, x_static, layer.wr, layer.bias, None, layer.wg, layer.wu, layer.wd, layer.sg, layer.su,
                      layer.sd, out, ws=ws)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.moe_forward(w, T, x_static, layer.wr, layer.bias, None, layer.wg, layer.wu, layer.wd, layer.sg, layer.su,
                      layer.sd, out, ws=ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    # new input in the captured buffer: the replay computes the new batch
    x_static.copy_(mi.hidden_states(w.with_(seed=7), device="cuda"))
    g.replay()
    layer.x = x_static.clone()
    torch.cuda.synchronize()
    assert torch.equal(out, layer.forward()["out"])
    assert m.moe_check_status() == 0


def _fp8_layer(w):
    import numpy as np
    import oracle
    wg, wu, wd = mi.stacked_expert_weights(w)
    sg, su, sd = mi.stacked_shared_weights(w)
    q = oracle.quantize_layer_fp8(w, wg, wu, wd, sg, su, sd)
    return {k_: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k_, v in q.items()}


def _fp8_forward(w, T, x, wr, d, out, ws):
    m.moe_forward_fp8(w, T, x, wr, None, None, d["qg"], d["sg"], d["qu"], d["su"], d["qd"], d["sd"], d["qsg"],
                      d["ssg"], d["qsu"], d["ssu"], d["qsd"], d["ssd"], out, ws=ws)


@pytest.mark.parametrize("tokens", [16, 2560])  # programmatic launches / plain launches and the chunked index pass
def test_fp8_forward_replays_from_a_cuda_graph(tokens):
    w = mi.WORKLOADS["tiny"].with_(tokens=tokens)
    T, H = w.tokens, w.hidden
    d = _fp8_layer(w)
    x = mi.hidden_states(w, device="cuda")
    wr = mi.router_weight(w, device="cuda")
    ws = torch.empty(m.moe_workspace_size_fp8(w, T), dtype=torch.uint8, device="cuda")
    ref = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    _fp8_forward(w, T, x, wr, d, ref, ws)
    torch.cuda.synchronize()
    out = torch.empty_like(ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _fp8_forward(w, T, x, wr, d, out, ws)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _fp8_forward(w, T, x, wr, d, out, ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert m.moe_check_status() == 0


def test_two_streams_run_independent_layers_concurrently():
    """No state is shared between calls beyond the caller's buffers: a small
    batch (programmatic launches) and a large one (chunked index pass, plain
    launches) on two streams at once give exactly their sequential results."""
    ws_ = [mi.WORKLOADS["tiny"].with_(tokens=16, seed=3), mi.WORKLOADS["tiny"].with_(tokens=2560, seed=4)]
    layers = [DeviceLayer(w, "cuda") for w in ws_]
    refs = [layer.forward()["out"].clone() for layer in layers]
    outs = [torch.empty_like(r) for r in refs]
    bufs = [torch.empty(m.moe_workspace_size(w, w.tokens), dtype=torch.uint8, device="cuda") for w in ws_]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(3):
        for w, layer, out, ws, st in zip(ws_, layers, outs, bufs, streams):
            with torch.cuda.stream(st):
                m.moe_forward(w, w.tokens, layer.x, layer.wr, layer.bias, None, layer.wg, layer.wu, layer.wd,
                              layer.sg, layer.su, layer.sd, out, ws=ws, stream=st)
        torch.cuda.synchronize()
        for out, ref in zip(outs, refs):
            assert torch.equal(out, ref)
    assert m.moe_check_status() == 0
