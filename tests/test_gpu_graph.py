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
