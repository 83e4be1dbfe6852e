"""The C ABI from several host threads at once.  In a fresh process four
threads make the library's first calls together (the per-device set-up of
each kernel races), each on its own stream with its own buffers, for two
layer shapes that take different kernels (32- and 160-row GEMM chunks, the
single-CTA and the chunked index pass); every thread's outputs equal a
single-threaded pass bit for bit."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

SCRIPT = r"""
import sys, threading
sys.path[:0] = [sys.argv[1], sys.argv[2]]
import torch
import moe_expert_layer_06_gb300 as m
import moe_inputs as mi

dev = torch.device("cuda", 0)
torch.cuda.set_device(dev)
cases = {
    "tiny": mi.WORKLOADS["tiny"],
    # 4400 assignments: chunked index pass, 160-row GEMM chunks
    "wide": mi.WORKLOADS["tiny"].with_(name="wide", tokens=2200, hidden=128, inter=64, n_experts=16, top_k=2,
                                       n_shared=1, inter_shared=64, n_slots=16, n_blocks=4),
}
inputs = {}
for name, w in cases.items():  # torch kernels only: the library has not been called yet
    wg, wu, wd = mi.stacked_expert_weights(w, device=dev)
    sg, su, sd = mi.stacked_shared_weights(w, device=dev)
    inputs[name] = (mi.hidden_states(w, device=dev), mi.router_weight(w, device=dev), wg, wu, wd, sg, su, sd)
torch.cuda.synchronize()


def run(name, stream, passes):
    w = cases[name]
    T = w.tokens
    x, wr, wg, wu, wd, sg, su, sd = inputs[name]
    with torch.cuda.stream(stream):
        ws = torch.empty(m.moe_workspace_size(w, T), dtype=torch.uint8, device=dev)
        res = []
        for _ in range(passes):
            out = torch.empty((T, w.hidden), dtype=torch.bfloat16, device=dev)
            idx = torch.empty((T, w.top_k), dtype=torch.int32, device=dev)
            counts = torch.empty(w.n_slots + 1, dtype=torch.int32, device=dev)
            m.moe_forward(w, T, x, wr, None, None, wg, wu, wd, sg, su, sd, out, topk_idx_out=idx,
                          counts_out=counts, ws=ws, stream=stream)
            res.append((out, idx, counts))
    stream.synchronize()
    return res


start = threading.Barrier(4)
results, errors = {}, []


def worker(i, name):
    try:
        s = torch.cuda.Stream(dev)
        start.wait()
        results[i] = (name, run(name, s, 3))
    except Exception as e:  # reported by the main thread
        errors.append(f"thread {i}: {e!r}")


threads = [threading.Thread(target=worker, args=(i, n)) for i, n in enumerate(["tiny", "wide", "tiny", "wide"])]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errors, errors
assert m.moe_check_status() == 0, m.last_error()
ref = {name: run(name, torch.cuda.Stream(dev), 1)[0] for name in cases}
for i, (name, passes) in sorted(results.items()):
    for out, idx, counts in passes:
        assert torch.equal(out, ref[name][0]), (i, name, "out")
        assert torch.equal(idx, ref[name][1]), (i, name, "idx")
        assert torch.equal(counts, ref[name][2]), (i, name, "counts")
assert m.moe_dispatch_workspace_size(cases["wide"], cases["wide"].tokens) > 0  # the chunked index pass ran
print("ok", len(results))
"""


def test_concurrent_first_calls_from_four_threads_match_a_single_thread():
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT, HERE], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-4000:])
    assert r.stdout.strip().endswith("ok 4")
