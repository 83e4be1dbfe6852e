"""Helpers shared by the test files: device inputs, tolerance checks, oracle runs."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle

# Float tolerance of the bf16 layer output against the fp64 oracle.
REL_FROB = 5e-3
ELEM_RMS = 3e-2
TOPK_GAP = 1e-4

THREADS = max(1, min(32, os.cpu_count() or 1))


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy()


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |v| (8 significant bits): the rounding error a
    bf16 output may carry on top of its arithmetic error."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def assert_close(got, want, rel_frob=REL_FROB, elem_rms=ELEM_RMS, what="", bf16_out=True):
    """Relative Frobenius error <= rel_frob and every |err| <= elem_rms * rms(want),
    plus, for a bf16 output compared with the unrounded oracle, half the bf16
    spacing at that element (a value between two bf16 numbers is at least
    that far from both)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = got - want
    nw = np.linalg.norm(want)
    rel = np.linalg.norm(err) / nw if nw > 0 else np.linalg.norm(err)
    rms = np.sqrt(np.mean(want ** 2)) if want.size else 0.0
    assert rel <= rel_frob, f"{what}: relative Frobenius error {rel:.3e} > {rel_frob}"
    if err.size:
        bound = elem_rms * rms + 1e-30 + (bf16_half_ulp(want) if bf16_out else 0.0)
        worst = np.argmax(np.abs(err) - bound)
        e_w, b_w = np.abs(err).ravel()[worst], np.broadcast_to(bound, err.shape).ravel()[worst]
        assert e_w <= b_w, (f"{what}: |err| {e_w:.3e} > bound {b_w:.3e} ({elem_rms}*rms {elem_rms * rms:.3e}"
                            f"{' + half bf16 ulp' if bf16_out else ''}) at value {want.ravel()[worst]:.4g}")
    mx = np.abs(err).max() if err.size else 0.0
    return rel, mx / rms if rms else 0.0


def topk_gap(logits: np.ndarray, k: int) -> np.ndarray:
    """Gap between the k-th and (k+1)-th largest logit of each row (inf if k = E)."""
    s = -np.sort(-logits, axis=1)
    if s.shape[1] <= k:
        return np.full(s.shape[0], np.inf)
    return s[:, k - 1] - s[:, k]


def check_topk(idx_gpu, idx_ref, logits_ref, k, gap=TOPK_GAP):
    """Top-k parity where rounding cannot decide it.

    The selected set must match on every token whose k-th and (k+1)-th oracle
    logits differ by more than ``gap``; the order must match too where every
    adjacent pair among the top k+1 differs by more than ``gap``.  Returns the
    boolean mask of tokens whose set was checked.
    """
    idx_gpu = np.asarray(idx_gpu)
    idx_ref = np.asarray(idx_ref)
    s = -np.sort(-np.asarray(logits_ref), axis=1)[:, :k + 1]
    adj = s[:, :-1] - s[:, 1:]
    if s.shape[1] > k:
        set_ok = adj[:, k - 1] > gap
        order_ok = adj.min(axis=1) > gap
    else:
        set_ok = np.ones(s.shape[0], bool)
        order_ok = adj.min(axis=1) > gap if adj.shape[1] else set_ok
    bad_set = np.flatnonzero(set_ok & np.any(np.sort(idx_gpu, 1) != np.sort(idx_ref, 1), axis=1))
    assert bad_set.size == 0, f"top-k set differs on {bad_set.size} tokens with gap > {gap}: {bad_set[:8]}"
    bad_ord = np.flatnonzero(order_ok & np.any(idx_gpu != idx_ref, axis=1))
    assert bad_ord.size == 0, f"top-k order differs on {bad_ord.size} tokens with all gaps > {gap}: {bad_ord[:8]}"
    return set_ok


def grouped_sure(lo, k, G, Gk, gap=1e-4):
    """Tokens whose group choice and expert choice (group-limited routing) are
    both decided by more than gap, and the oracle's selection."""
    T, E = lo.shape
    gmax = -np.sort(-lo.reshape(T, G, E // G).max(axis=2), axis=1)
    g_ok = (gmax[:, Gk - 1] - gmax[:, Gk]) > gap if Gk < G else np.ones(T, bool)
    idx, _ = oracle.topk_grouped(lo, k, G, Gk)
    masked = np.full_like(lo, -np.inf)
    for t in range(T):
        keep = sorted({int(e) // (E // G) for e in idx[t]} |
                      set(np.argsort(-lo[t].reshape(G, E // G).max(axis=1), kind="stable")[:Gk].tolist()))
        for g in keep:
            masked[t, g * (E // G):(g + 1) * (E // G)] = lo[t, g * (E // G):(g + 1) * (E // G)]
    s = -np.sort(-masked, axis=1)
    e_ok = (s[:, k - 1] - s[:, k]) > gap if s.shape[1] > k else np.ones(T, bool)
    return g_ok & e_ok, idx


def parallel_router_logits(w, x_cpu, wr_cpu, bias):
    """Oracle logits for all rows, rows split across host threads (the C code is pure)."""
    T = x_cpu.shape[0]
    chunks = np.array_split(np.arange(T), min(THREADS, max(1, T)))
    with cf.ThreadPoolExecutor(len(chunks)) as ex:
        parts = list(ex.map(lambda r: oracle.router_logits(w, x_cpu[r[0]:r[-1] + 1], wr_cpu, bias)
                            if len(r) else np.zeros((0, w.n_experts)), chunks))
    return np.concatenate(parts, axis=0)


class DeviceLayer:
    """Device copies of one workload's inputs (generated on the device)."""

    def __init__(self, w, device="cuda", replica_of=None, weights=None):
        self.w = w
        self.dev = torch.device(device)
        self.x = mi.hidden_states(w, device=self.dev)
        self.wr = mi.router_weight(w, device=self.dev)
        b = mi.router_bias(w)
        self.bias = torch.from_numpy(b).to(self.dev) if b is not None else None
        self.replica_of_np = replica_of
        self.replica_of = (torch.from_numpy(np.asarray(replica_of, dtype=np.int32)).to(self.dev)
                           if replica_of is not None else None)
        if weights is None:
            weights = mi.stacked_expert_weights(w, replica_of, device=self.dev)
        self.wg, self.wu, self.wd = weights
        if w.n_shared > 0:
            self.sg, self.su, self.sd = mi.stacked_shared_weights(w, device=self.dev)
        else:
            self.sg = self.su = self.sd = None

    def forward(self, mode=m.MOE_FFN_AUTO):
        w, T = self.w, self.w.tokens
        out = torch.empty((T, w.hidden), dtype=torch.bfloat16, device=self.dev)
        idx = torch.empty((T, w.top_k), dtype=torch.int32, device=self.dev)
        tw = torch.empty((T, w.top_k), dtype=torch.float32, device=self.dev)
        counts = torch.empty(w.n_slots + 1, dtype=torch.int32, device=self.dev)
        blocks = torch.empty(w.n_blocks, dtype=torch.int32, device=self.dev)
        ws = torch.empty(max(1, m.moe_workspace_size(w, T)), dtype=torch.uint8, device=self.dev)
        m.moe_forward(w, T, self.x, self.wr, self.bias, self.replica_of, self.wg, self.wu, self.wd,
                      self.sg, self.su, self.sd, out, idx, tw, counts, blocks, mode=mode, ws=ws)
        rc = m.moe_check_status()
        assert rc == 0, m.last_error()
        return dict(out=out, idx=idx, w=tw, counts=counts, blocks=blocks)

    def forward_grouped(self, n_groups, topk_groups, mode=m.MOE_FFN_AUTO):
        """The layer through the staged calls with group-limited routing."""
        w, T, dev = self.w, self.w.tokens, self.dev
        k, S, H, n = w.top_k, w.n_slots, w.hidden, w.tokens * w.top_k
        i32 = dict(dtype=torch.int32, device=dev)
        idx, tw = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device=dev)
        rws = torch.empty(max(16, m.moe_route_workspace_size(w, T)), dtype=torch.uint8, device=dev)
        m.moe_route_grouped(w, T, n_groups, topk_groups, self.x, self.wr, self.bias, None, None, idx, tw, rws)
        so, counts, blocks = torch.empty(n, **i32), torch.empty(S + 1, **i32), torch.empty(w.n_blocks, **i32)
        offsets, perm, inv = torch.empty(S + 2, **i32), torch.empty(n, **i32), torch.empty(n, **i32)
        x_disp = torch.empty((n, H), dtype=torch.bfloat16, device=dev)
        m.moe_dispatch(w, T, self.x, idx, self.replica_of, so, counts, blocks, offsets, perm, inv, x_disp)
        y = torch.empty((n, H), dtype=torch.bfloat16, device=dev)
        ysh = torch.empty((T, H), dtype=torch.float32, device=dev)
        fws = torch.empty(max(16, m.moe_ffn_workspace_size(w, T)), dtype=torch.uint8, device=dev)
        m.moe_expert_ffn(w, T, self.x, x_disp, offsets, self.wg, self.wu, self.wd, self.sg, self.su, self.sd, y,
                         ysh if w.n_shared else None, mode, fws)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        m.moe_combine(w, T, y, inv, tw, ysh if w.n_shared else None, out)
        assert m.moe_check_status() == 0, m.last_error()
        return dict(out=out, idx=idx, w=tw, counts=counts, blocks=blocks)


def oracle_token_rows(w, tokens, x_cpu, wr_cpu, bias, replica_of=None, expert_cache=None, groups=None):
    """Oracle routing and output for a sample of tokens of a full-size workload
    (groups = (n_groups, topk_groups) for group-limited routing).

    Only the experts those tokens select are generated (on the CPU).
    """
    expert_cache = {} if expert_cache is None else expert_cache
    xs = x_cpu[tokens]
    logits = oracle.router_logits(w, xs, wr_cpu, bias)
    if groups is None:
        idx, wt = oracle.topk_softmax(logits, w.top_k)
    else:
        idx, wt = oracle.topk_grouped(logits, w.top_k, *groups)
    need = sorted(set(int(e) for e in idx.ravel()) - set(expert_cache))
    for e in need:
        expert_cache[e] = mi.expert_weights(w, e)
    sg, su, sd = mi.stacked_shared_weights(w)

    def one(i):
        gud = [expert_cache[int(e)] for e in idx[i]]
        ys = [oracle.swiglu_row(xs[i], *g) for g in gud]
        out = oracle.token_output(w, xs[i], wt[i], gud, sg, su, sd)
        return ys, out

    with cf.ThreadPoolExecutor(min(THREADS, len(tokens))) as ex:
        res = list(ex.map(one, range(len(tokens))))
    return dict(logits=logits, idx=idx, weight=wt, y=[r[0] for r in res], out=np.stack([r[1] for r in res]))
