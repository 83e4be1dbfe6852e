"""Benchmark of the MoE layer forward pass on GB300 (one JSON line on rank 0).

Default workload: the DeepSeek-V3 MoE layer decode step (T=32 tokens, hidden
7168, 256 routed experts SwiGLU 2048, top-8, 2 shared experts, bf16,
near-uniform routing), every input resident in HBM.  One step = one forward
pass of the layer over the batch: router GEMM + top-k, dispatch, expert
gate/up, expert down, combine (7 kernels of libmoe).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the reference arm of this
project) on the host cores on a bounded sample of the same workload.
With N > 1 (torchrun), every rank runs an independent replica of the layer
on its own batch (weak scaling, no collective on the data path); the step
time is the max over ranks.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import moe_inputs as mi  # noqa: E402

METRIC = "MoE-layer tokens/s and % of roofline (HBM GB/s decode, TFLOPS prefill), 1 GB300"
DEFAULT_CONFIG = "decode_t32"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


# ------------------------------------------------------------------------------ helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def max_over_ranks(value: float, device, world: int) -> float:
    """The largest value over the ranks of the job (a step's time is its slowest
    rank's); the value itself on one rank."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's step time."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("grouped_gemm.cu", "common.cuh", "kernels.h"):
        with open(os.path.join(ROOT, "moe_expert_layer_06_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
        e = d[kernel][workload]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.reader.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            p = [x.strip() for x in l.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def routing_stats(w, counts_np, blocks_np, replica_of=None):
    """Load statistics of one routed batch from the device histogram: rows per
    slot, the share of assignments taken by the 30% most loaded experts, and
    the EP-block imbalance max/mean with the replicas as placed and as if
    every expert stayed in its home block."""
    E, S, B = w.n_experts, w.n_slots, w.n_blocks
    epb, spb = E // B, S // B
    slot = counts_np[:S].astype(np.int64)
    home = np.array([(e // epb) * spb + e % epb for e in range(E)])
    expert = slot[home].copy()
    if replica_of is not None:
        for e, r in enumerate(replica_of):
            if r >= 0:
                expert[e] += slot[r]
    total = max(1, int(expert.sum()))
    top = np.sort(expert)[::-1][:max(1, (3 * E + 9) // 10)]
    blocks = blocks_np.astype(np.int64)
    home_blocks = expert.reshape(B, epb).sum(axis=1)
    ratio = lambda b: float(b.max() * B / b.sum()) if b.sum() else 0.0
    return {"max_rows_per_slot": int(slot.max()), "touched_experts": int((expert > 0).sum()),
            "top30pct_expert_share": round(float(top.sum()) / total, 4),
            "block_max_over_mean": round(ratio(blocks), 4),
            "block_max_over_mean_without_replicas": round(ratio(home_blocks), 4)}


def layer_bytes_flops(w, counts_np, fp8=False):
    """Algorithmic bytes and flops of one layer pass (touched expert weights read once).

    fp8: expert weights and both payloads are one byte per element (plus the
    combine payload's fp32 scale per 128-column block).
    """
    H, I, E, k, T = w.hidden, w.inter, w.n_experts, w.top_k, w.tokens
    gb = 1 if fp8 else 2  # bytes per expert weight and per dispatched element
    touched = int((counts_np[:w.n_slots] > 0).sum())
    expert_bytes = 3 * H * I * gb
    shared_bytes = w.n_shared * 3 * H * w.inter_shared * gb
    y_row = H + 4 * ((H + 127) // 128) if fp8 else 2 * H  # combine payload bytes per assignment
    act = T * H * 2 + 2 * T * k * H * gb + 2 * T * k * y_row + T * H * 2
    B = touched * expert_bytes + shared_bytes + E * H * 2 + act
    F = 6 * H * I * T * k + 6 * H * w.inter_shared * w.n_shared * T + 2 * T * H * E
    # gate/up launch: gate+up weights of touched slots and shared, x_disp + x read, h written
    B_gu = touched * 2 * H * I * gb + w.n_shared * 2 * H * w.inter_shared * gb + T * k * H * gb + T * H * gb + \
        T * k * I * 2 + T * w.n_shared * w.inter_shared * 2
    return dict(touched=touched, bytes=B, flops=F, gate_up_bytes=B_gu)


# ------------------------------------------------------------------------------ our arm

# workloads timed after the headline one, in the same run and with the same step count
# (decode_t256_skew_a05: the skewed batch with the bias calibrated to the pages'
# ~30% of experts taking ~60% of the assignments, beside the literal formula)
EXTRA_CONFIGS = ("decode_t256_skew", "decode_t256_skew_a05", "prefill_t4096", "redundant_t1024")


class DeviceWeights:
    """Expert weights on the device, generated once per expert shape and shared by
    the workloads of that shape (a replica slot is a byte copy of its expert)."""

    def __init__(self, m, dev):
        self.m, self.dev = m, dev
        self.key, self.base, self.q = None, None, None

    def _base(self, w):
        key = (w.hidden, w.inter, w.n_experts, w.n_shared, w.inter_shared, w.seed)
        if key != self.key:  # one expert shape resident at a time
            self.key, self.base, self.q = None, None, None
            torch.cuda.empty_cache()
            base = w.with_(n_slots=w.n_experts)
            wg, wu, wd = mi.stacked_expert_weights(base, device=self.dev)
            sg, su, sd = mi.stacked_shared_weights(base, device=self.dev)
            mi.clear_cache()
            self.key, self.base = key, (wg, wu, wd, sg, su, sd)
        return self.base

    def bf16(self, w, rep):
        wg, wu, wd, sg, su, sd = self._base(w)
        if w.n_slots > w.n_experts:
            se = torch.from_numpy(mi.slot_experts(w, rep)).to(self.dev)
            wg, wu, wd = (t.index_select(0, se) for t in (wg, wu, wd))
        return wg, wu, wd, sg, su, sd

    def fp8(self, w, rep):
        """E4M3 codes and one scale per output row of every expert matrix; the shared
        experts' down matrices as one [H, n_sh*I_sh] matrix (their outputs are summed)."""
        m, dev = self.m, self.dev
        wg, wu, wd, sg, su, sd = self._base(w)
        if self.q is None:
            def quant(t):
                q = torch.empty(t.shape, dtype=torch.uint8, device=dev)
                sc = torch.empty(t.shape[:-1], dtype=torch.float32, device=dev)
                m.moe_quantize_rows_fp8(t.view(-1, t.shape[-1]), q, sc)
                return q, sc
            self.q = quant(wg) + quant(wu) + quant(wd) + quant(sg) + quant(su) + \
                quant(sd.permute(1, 0, 2).reshape(w.hidden, -1).contiguous())
            torch.cuda.synchronize(dev)
        q = list(self.q)
        if w.n_slots > w.n_experts:
            se = torch.from_numpy(mi.slot_experts(w, rep)).to(dev)
            q[:6] = [t.index_select(0, se) for t in q[:6]]
        return tuple(q)


def measure(m, args, w, dev, rank, world, local_rank, weights, with_cpu_baseline):
    """Time one workload: K device-timed steps (stage kernels through the C ABI),
    then K end-to-end steps through moe_forward with host copies.  Returns the
    JSON fields of that workload (rank 0) or None."""
    T = w.tokens
    rep = None
    if w.n_slots > w.n_experts:
        rep = replica_plan_gpu(m, w, dev)
    x = mi.hidden_states(w, device=dev)
    wr = mi.router_weight(w, device=dev)
    b = mi.router_bias(w)
    bias = torch.from_numpy(b).to(dev) if b is not None else None
    fp8 = bool(args.fp8)
    if fp8:
        qg, s_g, qu, s_u, qd, s_d, qsg, s_sg, qsu, s_su, qsd, s_sd = weights.fp8(w, rep)
    else:
        wg, wu, wd, sg, su, sd = weights.bf16(w, rep)
    repd = torch.from_numpy(rep).to(dev) if rep is not None else None
    torch.cuda.empty_cache()

    k, H, I, S, E = w.top_k, w.hidden, w.inter, w.n_slots, w.n_experts
    n = T * k
    i32 = dict(dtype=torch.int32, device=dev)
    idx = torch.empty((T, k), **i32)
    tw = torch.empty((T, k), dtype=torch.float32, device=dev)
    slot_of = torch.empty(n, **i32)
    counts = torch.empty(S + 1, **i32)
    blocks = torch.empty(w.n_blocks, **i32)
    offsets = torch.empty(S + 2, **i32)
    perm = torch.empty(n, **i32)
    inv = torch.empty(n, **i32)
    x_disp = torch.empty((n, H), dtype=torch.bfloat16, device=dev)
    if fp8:
        x8 = torch.empty((T, H), dtype=torch.uint8, device=dev)
        xs8 = torch.empty(T, dtype=torch.float32, device=dev)
        x_disp8 = torch.empty((n, H), dtype=torch.uint8, device=dev)
        xds8 = torch.empty(n, dtype=torch.float32, device=dev)
        h8 = torch.empty((n, I), dtype=torch.uint8, device=dev)
        h8s = torch.empty(n, dtype=torch.float32, device=dev)
        hs8 = torch.empty((T, w.n_shared * w.inter_shared), dtype=torch.uint8, device=dev)
        hs8s = torch.empty(T, dtype=torch.float32, device=dev)
        y8 = torch.empty((n, H), dtype=torch.uint8, device=dev)
        y8s = torch.empty((n, (H + m.MOE_PAYLOAD_BLOCK - 1) // m.MOE_PAYLOAD_BLOCK), dtype=torch.float32, device=dev)
    h = torch.empty((n, I), dtype=torch.bfloat16, device=dev)
    hs = torch.empty((T, w.n_shared * w.inter_shared), dtype=torch.bfloat16, device=dev)
    y = torch.empty((n, H), dtype=torch.bfloat16, device=dev)
    ysh = torch.empty((T, H), dtype=torch.float32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    rws = torch.empty(max(16, m.moe_route_workspace_size(w, T)), dtype=torch.uint8, device=dev)
    dws = torch.empty(max(16, m.moe_dispatch_workspace_size(w, T)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    ffn_mode = {"auto": m.MOE_FFN_AUTO, "decode": m.MOE_FFN_DECODE, "prefill": m.MOE_FFN_PREFILL}[args.ffn_mode]
    groups = None
    if args.route_groups:
        groups = tuple(int(v) for v in args.route_groups.split(":"))

    def step(ev=None, st=None):
        if groups:
            m.moe_route_grouped(w, T, groups[0], groups[1], x, wr, bias, None, None, idx, tw, rws)
        else:
            m.moe_route(w, T, x, wr, bias, None, None, idx, tw, rws)
        if st is not None:
            st[0].record(stream)
        if fp8:
            m.moe_dispatch_fp8(w, T, x, idx, repd, slot_of, counts, blocks, offsets, perm, inv, x8, xs8, x_disp8,
                               xds8, ws=dws)
        else:
            m.moe_dispatch(w, T, x, idx, repd, slot_of, counts, blocks, offsets, perm, inv, x_disp, ws=dws)
        if ev is not None:
            ev[0].record(stream)
        if fp8:
            m.moe_expert_gate_up_fp8(w, T, x8, xs8, x_disp8, xds8, offsets, qg, s_g, qu, s_u, qsg, s_sg, qsu, s_su,
                                     h, hs, mode=ffn_mode)
        else:
            m.moe_expert_gate_up(w, T, x, x_disp, offsets, wg, wu, sg, su, h, hs, mode=ffn_mode)
        if ev is not None:
            ev[1].record(stream)
        if fp8:
            m.moe_quantize_rows_fp8(h, h8, h8s)
            if w.n_shared:
                m.moe_quantize_rows_fp8(hs, hs8, hs8s)
            m.moe_expert_down_fp8_payload(w, T, h8, h8s, hs8, hs8s, offsets, qd, s_d, qsd, s_sd, y8, y8s, ysh,
                                          mode=ffn_mode)
        else:
            m.moe_expert_down(w, T, h, hs, offsets, wd, sd, y, ysh, mode=ffn_mode)
        if st is not None:
            st[1].record(stream)
        if fp8:
            m.moe_combine_fp8(w, T, y8, y8s, inv, tw, ysh, out)
        else:
            m.moe_combine(w, T, y, inv, tw, ysh, out)

    # router GEMM + top-k, index pass (three launches in chunks for large batches), scatter
    # (E4M3: + token quantisation), gate/up, (E4M3: + intermediate quantisation), down, combine
    index_launches = 3 if m.moe_dispatch_workspace_size(w, T) > 0 else 1
    launches_per_step = 2 + index_launches + 1 + 1 + 1 + 1
    if fp8:
        launches_per_step += 1 + 1 + (w.n_shared > 0)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    rc = m.moe_check_status(stream)
    if rc != 0:
        raise RuntimeError("device status after warm-up: " + m.last_error())

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sts = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)] if args.stage_times else [None] * args.steps
    t0.record(stream)
    for i in range(args.steps):
        step(evs[i], sts[i])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if rank == 0 else None
    elapsed_ms = t0.elapsed_time(t1)
    gu_ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    elapsed_ms = max_over_ranks(elapsed_ms, dev, world)
    rc = m.moe_check_status(stream)
    if rc != 0:
        raise RuntimeError("device status after timing: " + m.last_error())

    # end-to-end through the public C-ABI call with host buffers (pinned), copies inside the timed
    # region, double-buffered as a serving loop would: step i+1's input goes up and step i-1's output
    # comes down on a copy stream while step i computes
    x_host = x.cpu().pin_memory()
    out_host = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    out_dev = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ws = torch.empty((m.moe_workspace_size_fp8 if fp8 else m.moe_workspace_size)(w, T), dtype=torch.uint8,
                     device=dev)
    copy_stream = torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]

    def layer(xb, ob):  # one pass of the layer through the public API, on `stream`
        if groups:  # the staged calls (moe_forward routes over all experts)
            x.copy_(xb)
            step()
            ob.copy_(out)
        elif fp8:
            m.moe_forward_fp8(w, T, xb, wr, bias, repd, qg, s_g, qu, s_u, qd, s_d, qsg, s_sg, qsu, s_su, qsd, s_sd,
                              ob, mode=ffn_mode, ws=ws)
        else:
            m.moe_forward(w, T, xb, wr, bias, repd, wg, wu, wd, sg, su, sd, ob, mode=ffn_mode, ws=ws)

    def e2e_run(n, e_begin=None, e_end=None):
        with torch.cuda.stream(copy_stream):
            if e_begin is not None:
                e_begin.record(copy_stream)
            x_dev[0].copy_(x_host, non_blocking=True)
            in_ready[0].record(copy_stream)
        for i in range(n):
            b = i & 1
            stream.wait_event(in_ready[b])
            if i >= 2:
                stream.wait_event(out_read[b])  # out_dev[b] has gone down (step i-2)
            layer(x_dev[b], out_dev[b])
            computed[b].record(stream)
            with torch.cuda.stream(copy_stream):
                if i + 1 < n:
                    if i >= 1:
                        copy_stream.wait_event(computed[b ^ 1])  # step i-1 has read x_dev[b^1]
                    x_dev[b ^ 1].copy_(x_host, non_blocking=True)
                    in_ready[b ^ 1].record(copy_stream)
                copy_stream.wait_event(computed[b])
                out_host[b].copy_(out_dev[b], non_blocking=True)
                out_read[b].record(copy_stream)
        if e_end is not None:
            e_end.record(copy_stream)

    e2e_run(args.warmup)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_run(args.steps, e0, e1)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev, world)
    if m.moe_check_status(stream) != 0:
        raise RuntimeError("device status after e2e: " + m.last_error())

    if rank != 0:
        return None
    cnt = counts.cpu().numpy()
    bf = layer_bytes_flops(w, cnt, fp8)
    hbm, tf_burst, tf_sus, src = peaks()
    ms_step = elapsed_ms / args.steps
    t_roof_ms = max(bf["bytes"] / (hbm * 1e9), bf["flops"] / (tf_sus * 1e12)) * 1e3
    achieved = bf["gate_up_bytes"] / (gu_ms * 1e-3) / 1e9
    tflops = bf["flops"] / (ms_step * 1e-3) / 1e12
    res = {
        "value": round(job_tokens_per_s(T, world, ms_step), 1),
        "unit": "tokens/s",
        "ms_per_step": round(ms_step, 4),
        "config": {
            "workload": w.name, "description": w.description, "tokens": T, "hidden": H, "inter": I,
            "n_experts": E, "top_k": k, "n_shared": w.n_shared, "n_slots": S,
            "touched_slots": bf["touched"], "ffn_mode": args.ffn_mode,
            "l2": "inputs larger than L2: each step streams %.1f GB of touched expert weights" % (bf["bytes"] / 1e9),
            "parallelism": "replica x%d (independent layer per GPU)" % world,
            "routing": ("group-limited: %d groups, keep %d" % groups) if groups else "top-%d of all experts" % k,
            "precision": ("E4M3 expert weights (gate, up, down; shared included), dispatch payload, SwiGLU "
                          "intermediate (per-row scales) and combine payload (one scale per 128-column block), "
                          "fp32 accumulate; bf16 router and layer output")
            if fp8 else "bf16 weights and activations, fp32 accumulate",
        },
        "us_per_layer": round(ms_step * 1e3, 2),
        "layer_roofline": {
            "bound": "hbm" if bf["bytes"] / (hbm * 1e9) >= bf["flops"] / (tf_sus * 1e12) else "tensor",
            "algorithmic_bytes": bf["bytes"], "flops": bf["flops"], "t_roof_us": round(t_roof_ms * 1e3, 2),
            "frac": round(t_roof_ms / ms_step, 4), "peaks": src,
            "achieved_gbs": round(bf["bytes"] / (ms_step * 1e-3) / 1e9, 1),
            "achieved_tflops": round(tflops, 2),
            "tensor_frac_of_sustained_bf16": round(tflops / tf_sus, 4),
        },
        "roofline": {
            "kernel": ("grouped_gemm_kernel<gate_up_e4m3> (moe_expert_gate_up_fp8)" if fp8
                       else "grouped_gemm_kernel<gate_up> (moe_expert_gate_up)"),
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": hbm,
            "unit": "GB/s",
            "frac": round(achieved / hbm, 4),
            "traffic": recorded_traffic("gate_up_fp8" if fp8 else "gate_up", w.name),
            "algorithmic_bytes_per_launch": bf["gate_up_bytes"],
            "avg_launch_us": round(gu_ms * 1e3, 2),
            "peak_source": src + " (hbm_gbs, copy bandwidth)",
        },
        "e2e": {
            "value": round(job_tokens_per_s(T, world, e2e_ms / args.steps), 1),
            "unit": "tokens/s",
            "h2d_bytes_per_step": T * H * 2,
            "d2h_bytes_per_step": T * H * 2,
            "api": ("moe_forward_fp8" if fp8 else "moe_forward") +
                   " (C ABI) with pinned host input/output copies in the timed region, double-buffered: "
                   "the next step's input and the previous step's output move on a copy stream while a "
                   "step computes",
        },
        "gpu_launches": launches_per_step * args.steps,
        "routing_stats": routing_stats(w, cnt, blocks.cpu().numpy(), rep),
        "clocks": clk,
    }
    if args.stage_times:  # per-stage means; the extra events sit between launches of the step
        res["stage_us"] = {
            "dispatch": round(sum(s_[0].elapsed_time(e_[0]) for s_, e_ in zip(sts, evs)) / args.steps * 1e3, 2),
            "gate_up": round(gu_ms * 1e3, 2),
            "down": round(sum(e_[1].elapsed_time(s_[1]) for s_, e_ in zip(sts, evs)) / args.steps * 1e3, 2),
        }
    if with_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, dev, args.cpu_sample)
    return res


def run_ours(args, rank, world, local_rank):
    import moe_expert_layer_06_gb300 as m
    if rank == 0:
        m.build_library()
    if world > 1:
        torch.distributed.barrier()
    m.build_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    weights = DeviceWeights(m, dev)
    w = mi.WORKLOADS[args.config]
    main = measure(m, args, w, dev, rank, world, local_rank, weights, world == 1 and not args.no_cpu_baseline)
    extra = {}
    if args.config == DEFAULT_CONFIG and not args.no_extra_configs and not args.route_groups:
        for name in EXTRA_CONFIGS:
            r = measure(m, args, mi.WORKLOADS[name], dev, rank, world, local_rank, weights, False)
            if r is not None:
                extra[name] = r
    if rank != 0:
        return None
    res = {
        "metric": METRIC,
        "value": main["value"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": main["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if args.fp8 else "bf16",
        "data": "synthetic (seeded counter-based generator; random-init DeepSeek-V3 MoE layer weights)",
    }
    res.update({k_: v for k_, v in main.items() if k_ not in ("value", "unit", "ms_per_step")})
    if extra:
        res["configs"] = extra
    return res


def replica_plan_gpu(m, w, dev):
    """Replica map from the histogram of the skewed decode batch, through libmoe."""
    src = mi.WORKLOADS[mi.REPLICA_PLAN_SOURCE]
    x = mi.hidden_states(src, device=dev)
    wr = mi.router_weight(src, device=dev)
    b = torch.from_numpy(mi.router_bias(src)).to(dev)
    idx = torch.empty((src.tokens, src.top_k), dtype=torch.int32, device=dev)
    tw = torch.empty((src.tokens, src.top_k), dtype=torch.float32, device=dev)
    ws = torch.empty(m.moe_route_workspace_size(src, src.tokens), dtype=torch.uint8, device=dev)
    m.moe_route(src, src.tokens, x, wr, b, None, None, idx, tw, ws)
    counts = torch.empty(src.n_slots + 1, dtype=torch.int32, device=dev)
    m.moe_expert_histogram(src, src.tokens, idx, None, counts, None)
    c = counts.cpu().numpy()[:src.n_experts]
    return m.moe_eplb_plan_replicas(w, c, w.n_slots - w.n_experts)


# ------------------------------------------------------------------------------ CPU oracle (baseline)

def _oracle_sample_inputs(w, n_tok, dev):
    """Inputs for the oracle on the first n_tok tokens (weights of the experts they use)."""
    import oracle
    toks = list(range(min(n_tok, w.tokens)))
    x = mi.hidden_states(w, rows=slice(0, len(toks)))
    wr = mi.router_weight(w)
    b = mi.router_bias(w)
    lo = oracle.router_logits(w, x, wr, b)
    idx, _ = oracle.topk_softmax(lo, w.top_k)
    gen_dev = dev if dev is not None else "cpu"
    experts = {}
    for e in sorted(set(int(v) for v in idx.ravel())):
        experts[e] = tuple(t.cpu() for t in mi.expert_weights(w, e, device=gen_dev))
    sh = tuple(t.cpu() for t in mi.stacked_shared_weights(w, device=gen_dev))
    mi.clear_cache()
    return toks, x, wr, b, experts, sh


def _oracle_tokens(w, toks, x, wr, b, experts, sh, threads):
    """The oracle's layer output for the sampled tokens: router, top-k, experts, shared, combine."""
    import oracle

    def one(i):
        lo = oracle.router_logits(w, x[i:i + 1], wr, b)
        idx, wt = oracle.topk_softmax(lo, w.top_k)
        gud = [experts[int(e)] for e in idx[0]]
        return oracle.token_output(w, x[i], wt[0], gud, *sh)

    with cf.ThreadPoolExecutor(threads) as ex:
        return list(ex.map(one, range(len(toks))))


def cpu_baseline(w, dev, n_tok, min_seconds=10.0):
    """The oracle on the host cores: the first n_tok tokens of the batch, in
    passes until at least min_seconds of wall time (bounded to 64 passes)."""
    threads = max(1, min(os.cpu_count() or 1, n_tok))
    toks, x, wr, b, experts, sh = _oracle_sample_inputs(w, n_tok, dev)
    passes = 0
    t = time.perf_counter()
    while True:
        _oracle_tokens(w, toks, x, wr, b, experts, sh, threads)
        passes += 1
        dt = time.perf_counter() - t
        if dt >= min_seconds or passes >= 64:
            break
    return {"value": round(passes * len(toks) / dt, 3), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"full layer output (router, top-{w.top_k}, {w.top_k} expert FFNs, shared, combine) of the "
                      f"first {len(toks)} tokens of the {w.name} batch, {passes} passes, fp64 C oracle, one token "
                      f"per thread",
            "seconds": round(dt, 3)}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    w = mi.WORKLOADS[args.config]
    n_tok = args.cpu_sample
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else None
    threads = max(1, min(os.cpu_count() or 1, n_tok))
    toks, x, wr, b, experts, sh = _oracle_sample_inputs(w, n_tok, dev)
    for _ in range(args.warmup):
        _oracle_tokens(w, toks, x, wr, b, experts, sh, threads)
    t = time.perf_counter()
    for _ in range(args.steps):
        _oracle_tokens(w, toks, x, wr, b, experts, sh, threads)
    dt = (time.perf_counter() - t) / max(1, args.steps)
    v = round(len(toks) / dt, 3)
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": w.name, "description": w.description, "tokens_per_step": len(toks)},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"first {len(toks)} tokens of the {w.name} batch per step, fp64 C oracle, "
                                   f"one token per thread"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_eplb(args):
    """Cost of the online EPLB loop on the redundant-expert workload (one JSON line).

    Times the layer alone, the layer plus the sliding-window push after every
    batch, and a full replica migration (all replica slots re-planned) copied
    on a side stream while the compute stream keeps serving with the stable
    table.
    """
    import moe_expert_layer_06_gb300 as m
    m.build_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = mi.WORKLOADS["redundant_t1024"] if args.config == DEFAULT_CONFIG else mi.WORKLOADS[args.config]
    assert w.n_slots > w.n_experts, "the EPLB mode needs a workload with replica slots"
    T, window = w.tokens, 8
    plan_a = replica_plan_gpu(m, w, dev)
    plan_b = m.moe_eplb_plan_replicas(w, np.arange(w.n_experts, dtype=np.int32)[::-1].copy(), w.n_slots - w.n_experts)
    x = mi.hidden_states(w, device=dev)
    wr = mi.router_weight(w, device=dev)
    bias = torch.from_numpy(mi.router_bias(w)).to(dev) if w.skew_alpha else None
    wg, wu, wd = mi.stacked_expert_weights(w, plan_a, device=dev)
    sg, su, sd = mi.stacked_shared_weights(w, device=dev)
    mi.clear_cache()
    out = torch.empty((T, w.hidden), dtype=torch.bfloat16, device=dev)
    counts = torch.empty(w.n_slots + 1, dtype=torch.int32, device=dev)
    ws = torch.empty(m.moe_workspace_size(w, T), dtype=torch.uint8, device=dev)
    state = torch.empty(m.moe_eplb_window_bytes(w, window), dtype=torch.uint8, device=dev)
    m.moe_eplb_window_reset(w, window, state)
    bl = torch.empty(w.n_blocks, dtype=torch.int64, device=dev)
    el = torch.empty(w.n_experts, dtype=torch.int64, device=dev)
    ratio = torch.empty(1, dtype=torch.float64, device=dev)
    trig = torch.empty(1, dtype=torch.int32, device=dev)
    tables = {n: torch.from_numpy(np.ascontiguousarray(t, np.int32)).to(dev)
              for n, t in (("a", plan_a), ("b", plan_b), ("stable", m.moe_eplb_stable_table(w, plan_a, plan_b)))}
    stream = torch.cuda.current_stream(dev)

    def fwd(table):
        m.moe_forward(w, T, x, wr, bias, tables[table], wg, wu, wd, sg, su, sd, out, counts_out=counts, ws=ws)

    def push():
        m.moe_eplb_window_push(w, window, state, counts, tables["a"], 1.2, bl, el, ratio, trig)

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n

    for _ in range(args.warmup):
        fwd("a")
        push()
    steps = max(args.steps, 10)
    t_plain = timed(lambda: fwd("a"), steps)
    t_window = timed(lambda: (fwd("a"), push()), steps)
    t_push = timed(push, steps)
    # migration: copies on a side stream, serving continues with the stable table
    copy = torch.cuda.Stream(device=dev)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    ready = torch.cuda.Event()
    ready.record(stream)
    with torch.cuda.stream(copy):
        copy.wait_event(ready)
        c0.record(copy)
        m.moe_eplb_copy_replicas(w, plan_a, plan_b, wg, wu, wd, stream=copy)
        c1.record(copy)
    s0.record(stream)
    fwd("stable")  # one step served concurrently with the copies
    s1.record(stream)
    stream.wait_event(c1)
    fwd("b")
    torch.cuda.synchronize(dev)
    if m.moe_check_status() != 0:
        raise RuntimeError(m.last_error())
    copy_ms = c0.elapsed_time(c1)
    changed = int(sum(1 for e in range(w.n_experts) if plan_b[e] >= 0 and plan_b[e] != plan_a[e]))
    copy_bytes = changed * 3 * w.hidden * w.inter * 2
    return {
        "mode": "eplb", "metric": "online EPLB loop cost", "unit": "ms", "higher_is_better": False,
        "config": {"workload": w.name, "tokens": T, "n_slots": w.n_slots, "window_batches": window,
                   "threshold": 1.2, "replicas_moved": changed},
        "ms_per_step_layer": round(t_plain, 4),
        "ms_per_step_layer_plus_window": round(t_window, 4),
        "window_push_us": round(t_push * 1e3, 2),
        "migration_copy_ms": round(copy_ms, 3),
        "migration_copy_gbs": round(2 * copy_bytes / (copy_ms * 1e-3) / 1e9, 1),
        "ms_one_step_concurrent_with_copy": round(s0.elapsed_time(s1), 4),
        "imbalance_ratio": round(float(ratio.item()), 4), "trigger": int(trig.item()),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(mi.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stage-times", action="store_true",
                    help="also record CUDA events around the dispatch and the down projection of every step")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="time the headline workload only (by default the decode line also times "
                         + ", ".join(EXTRA_CONFIGS) + ")")
    ap.add_argument("--route-groups", default="", help="G:Gk group-limited routing (timed region only)")
    ap.add_argument("--eplb", action="store_true", help="time the online EPLB loop instead (own JSON line)")
    ap.add_argument("--fp8", action="store_true", help="E4M3 expert weights and dispatch payload")
    ap.add_argument("--ffn-mode", default="auto", choices=["auto", "decode", "prefill"],
                    help="expert GEMM token chunk: automatic, 32 rows, or 160 rows")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.eplb:
        print(json.dumps(run_eplb(args)), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        if world > 1:
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        res = run_ours(args, rank, world, local_rank)
        if world > 1:
            torch.distributed.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
