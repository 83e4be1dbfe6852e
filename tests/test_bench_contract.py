"""bench.py without a GPU: the reference arm's JSON line (the timed fp64
oracle) and the algorithmic byte / flop accounting behind the roofline."""
import json
import os
import subprocess
import sys

import numpy as np

import moe_inputs as mi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "2", "--warmup", "1", "--cpu-sample", "4"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2
    assert d["warmup"] >= 3  # at least three warm-up steps whatever was asked
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny" and d["vs_baseline"] is None and d["gpu_launches"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_algorithmic_bytes_and_flops():
    w = mi.WORKLOADS["decode_t32"]
    T, H, I, k, E = w.tokens, w.hidden, w.inter, w.top_k, w.n_experts
    counts = np.zeros(w.n_slots + 1, np.int64)
    counts[:163] = 1
    bf = bench.layer_bytes_flops(w, counts)
    # touched slots' weights once, shared experts, router, x, dispatch and expert-output payloads, out
    per_slot = 3 * H * I * 2
    assert per_slot == 88_080_384
    want = 163 * per_slot + 2 * 3 * H * 2048 * 2 + E * H * 2 + T * H * 2 + 2 * T * k * H * 2 * 2 + T * H * 2
    assert bf["bytes"] == want and bf["touched"] == 163
    assert bf["flops"] == 6 * H * I * T * k + 6 * H * 2048 * 2 * T + 2 * T * H * E
    # E4M3: every expert weight and both payloads at one byte, the combine payload with 56 block scales a row
    bf8 = bench.layer_bytes_flops(w, counts, fp8=True)
    want8 = 163 * per_slot // 2 + 2 * 3 * H * 2048 + E * H * 2 + T * H * 2 + 2 * T * k * H + \
        2 * T * k * (H + 56 * 4) + T * H * 2
    assert bf8["bytes"] == want8


def test_routing_stats_on_a_hand_case():
    w = mi.WORKLOADS["tiny"].with_(n_experts=8, n_slots=12, n_blocks=4)  # blocks of 2 experts + 1 replica slot
    counts = np.zeros(13, np.int64)
    counts[[0, 1, 3, 4, 6, 7, 9, 10]] = [10, 0, 1, 1, 1, 1, 1, 1]
    counts[2] = 6  # block 0's replica slot, holding expert 5 (home slot 7)
    rep = np.full(8, -1)
    rep[5] = 2
    blocks = np.array([16, 2, 2, 2])
    st = bench.routing_stats(w, counts, blocks, rep)
    assert st["max_rows_per_slot"] == 10 and st["touched_experts"] == 7
    assert st["block_max_over_mean"] == round(16 * 4 / 22, 4)
    # without replicas expert 5's 7 rows go back to block 2
    assert st["block_max_over_mean_without_replicas"] == round(10 * 4 / 22, 4)
    assert st["top30pct_expert_share"] == round((10 + 7 + 1) / 22, 4)
