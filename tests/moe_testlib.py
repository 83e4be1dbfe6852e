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


# Elements with |ref| <= PLAIN_BOUND_RMS * rms(ref) are held to the scope's bound
# elem_rms * rms(ref) alone, without the half-ulp allowance: there the output's
# own bf16 rounding is at most PLAIN_BOUND_RMS * rms * 2^-8 (0.0156 rms), about
# half of the bound, which leaves the other half for the arithmetic.
PLAIN_BOUND_RMS = 4.0


def _report(record: dict) -> None:
    """Append one JSON line to $MOE_PARITY_REPORT (if set): the numbers the
    parity tests measured (errors, near-tie counts, sample sizes)."""
    path = os.environ.get("MOE_PARITY_REPORT")
    if not path:
        return
    import json
    with open(path, "a") as f:
        f.write(json.dumps(record) + "\n")


# An E4M3 combine payload code is decided by the kernel from its fp32 expert
# output and by the oracle from its fp64 one; where the two round to different
# bf16 values next to an E4M3 rounding boundary, a code differs by one step.
# Elements that need it may exceed the bound by one step of each routed
# contribution (payload_allowance), and at most this share of the elements may.
PAYLOAD_FLIP_SHARE = 2e-3


def e4m3_step(codes) -> np.ndarray:
    """Spacing between an E4M3 code and its larger-magnitude neighbour: 2^(e-10) in
    binade e >= 1, 2^-9 among the subnormals."""
    e = (np.asarray(codes, np.int64) >> 3) & 15
    return np.where(e == 0, 2.0 ** -9, np.ldexp(1.0, (e - 10).astype(np.int64)))


def payload_allowance(y_codes, y_scale, rows, weight, hidden) -> np.ndarray:
    """[T, H]: sum over a token's k payload rows of |w| * one E4M3 step at that
    element's block scale (rows [T, k]: payload row of each contribution)."""
    rows = np.asarray(rows)
    T, k = rows.shape
    blk = np.arange(hidden) // oracle.PAYLOAD_BLOCK
    out = np.zeros((T, hidden))
    for j in range(k):
        r = rows[:, j]
        out += np.abs(np.asarray(weight)[:, j])[:, None] * e4m3_step(y_codes[r]) * \
            y_scale[r][:, blk].astype(np.float64)
    return out


def assert_close(got, want, rel_frob=REL_FROB, elem_rms=ELEM_RMS, what="", bf16_out=True, e4m3_layer=False,
                 allowance=None):
    """Relative Frobenius error <= rel_frob and every |err| <= elem_rms * rms(want),
    plus, for a bf16 output compared with the unrounded oracle, half the bf16
    spacing at that element (a value between two bf16 numbers is at least
    that far from both); elements with |want| <= PLAIN_BOUND_RMS * rms(want)
    must meet elem_rms * rms(want) without that allowance, except in an E4M3
    layer's output (e4m3_layer): there the kernel quantises its own fp32
    intermediate and the oracle its fp64 one, so an intermediate code can
    differ by one step where the two round to different bf16 values, an
    error of its own beside the output's rounding; those outputs report the
    count without asserting it.  allowance ([same shape]): elements beyond the
    bound must lie within bound + allowance, and at most PAYLOAD_FLIP_SHARE of
    them (plus two) may (the E4M3 combine payload's one-step flips).

    Returns a dict: rel_frob, worst |err|/rms, how many elements exceed the
    plain bound (and so rely on the half-ulp allowance), and the largest
    |want|/rms among them."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = got - want
    nw = np.linalg.norm(want)
    rel = np.linalg.norm(err) / nw if nw > 0 else np.linalg.norm(err)
    rms = np.sqrt(np.mean(want ** 2)) if want.size else 0.0
    assert rel <= rel_frob, f"{what}: relative Frobenius error {rel:.3e} > {rel_frob}"
    stats = dict(what=what, elements=int(err.size), rel_frob=float(rel), worst_err_over_rms=0.0,
                 over_plain_bound=0, max_ref_over_rms_over_plain_bound=0.0)
    if err.size:
        plain = elem_rms * rms + 1e-30
        bound = plain + (bf16_half_ulp(want) if bf16_out else 0.0)
        if allowance is not None:
            beyond = np.abs(err) > bound
            stats["payload_flip_elements"] = int(beyond.sum())
            limit = PAYLOAD_FLIP_SHARE * err.size + 2
            assert beyond.sum() <= limit, (f"{what}: {int(beyond.sum())} elements beyond the bound, more than the "
                                           f"{limit:.0f} one-step payload flips allowed")
            bound = bound + np.where(beyond, allowance, 0.0)
        worst = np.argmax(np.abs(err) - bound)
        e_w, b_w = np.abs(err).ravel()[worst], np.broadcast_to(bound, err.shape).ravel()[worst]
        assert e_w <= b_w, (f"{what}: |err| {e_w:.3e} > bound {b_w:.3e} ({elem_rms}*rms {elem_rms * rms:.3e}"
                            f"{' + half bf16 ulp' if bf16_out else ''}) at value {want.ravel()[worst]:.4g}")
        over = np.abs(err) > plain
        inner = np.abs(want) <= PLAIN_BOUND_RMS * rms
        bad = np.flatnonzero((over & inner).ravel())
        assert e4m3_layer or bad.size == 0, (f"{what}: {bad.size} elements with |ref| <= {PLAIN_BOUND_RMS}*rms exceed "
                               f"{elem_rms}*rms without the half-ulp allowance, e.g. |err| "
                               f"{np.abs(err).ravel()[bad[0]]:.3e} at value {want.ravel()[bad[0]]:.4g}")
        stats["worst_err_over_rms"] = float(np.abs(err).max() / rms) if rms else 0.0
        stats["over_plain_bound"] = int(over.sum())
        if over.any():
            stats["max_ref_over_rms_over_plain_bound"] = float(np.abs(want[over]).max() / rms)
            stats["inner_over_plain_bound"] = int(bad.size)
    _report(dict(stats, kind="assert_close"))
    return stats


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


# ----------------------------------------------------------------------------- full-size sampled parity

SAMPLE_TOKENS = 256   # tokens per full-size workload checked element by element (all of them if fewer)
SAMPLE_SEED = 20261203


def sample_tokens(sure, n=SAMPLE_TOKENS, seed=SAMPLE_SEED) -> np.ndarray:
    """A seeded uniform sample of n tokens among those whose top-k selection is
    decided (all of them when there are at most n), ascending."""
    cand = np.flatnonzero(np.asarray(sure))
    if cand.size <= n:
        return cand
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.sort(rng.choice(cand, size=n, replace=False))


def check_counts_of_routing(w, idx_gpu, counts_gpu, blocks_gpu, rep=None, idx_oracle=None, sure=None):
    """The GPU's per-slot counts and block loads equal the oracle's remap and
    histogram of the GPU's own top-k selection (always), and of the oracle's
    selection when every token's selection is decided.  Returns the number of
    near-tie tokens (top-k gap <= TOPK_GAP)."""
    so, invalid = oracle.slot_map(w, np.asarray(idx_gpu), rep)
    assert invalid == 0
    c_o, b_o = oracle.histogram(w, so)
    assert np.array_equal(np.asarray(counts_gpu), c_o), "per-slot counts differ from the oracle's histogram"
    assert np.array_equal(np.asarray(blocks_gpu), b_o), "block loads differ from the oracle's histogram"
    ties = 0 if sure is None else int((~np.asarray(sure)).sum())
    if idx_oracle is not None and ties == 0:
        so2, _ = oracle.slot_map(w, idx_oracle, rep)
        c2, b2 = oracle.histogram(w, so2)
        assert np.array_equal(np.asarray(counts_gpu), c2) and np.array_equal(np.asarray(blocks_gpu), b2)
    return ties


def _pool_map(fn, items):
    with cf.ThreadPoolExecutor(min(THREADS, max(1, len(items)))) as ex:
        return list(ex.map(fn, items))


def oracle_sampled_layer(w, toks, x_cpu, idx, weight, expert_host, shared, fp8=False, window=16):
    """The oracle's layer output [len(toks), H] for the sampled tokens, given
    their selection idx[t] and combine weights weight[t] (oracle routing).

    Expert-major: the experts the sample selects are fetched `window` at a
    time through expert_host(e) -> (gate [I,H], up [I,H], down [H,I]) bf16 on
    the host, every (token, expert) pair of the window is computed by the
    oracle on the host threads, then the shared experts and the combine, in
    the oracle's order (j ascending, shared last).  fp8: the same with the
    layer's E4M3 quantisation, the oracle quantising each fetched expert's
    rows, and the E4M3 combine payload; shared = the oracle's E4M3 shared
    matrices (quantize_layer_fp8 keys qsg, ssg, qsu, ssu, qsd, ssd), else
    (gate, up, down) stacked bf16.  fp8 returns (out, payload_allowance).
    """
    toks = np.asarray(toks)
    n, k, H = len(toks), w.top_k, w.hidden
    xs = x_cpu[torch.as_tensor(toks, dtype=torch.long)]
    if fp8:
        qx, sx = oracle.quantize_rows_e4m3(xs)
    pairs = {}
    for i, t in enumerate(toks):
        for j in range(k):
            pairs.setdefault(int(idx[t, j]), []).append((i, j))
    y = np.zeros((n * k, H), dtype=np.float64)
    experts = sorted(pairs)
    for e0 in range(0, len(experts), window):
        group = experts[e0:e0 + window]
        mats = dict(zip(group, _pool_map(lambda e: tuple(a.contiguous() for a in expert_host(e)), group)))
        if fp8:
            flat = [(e, a) for e in group for a in range(3)]
            q = _pool_map(lambda ea: oracle.quantize_rows_e4m3(mats[ea[0]][ea[1]]), flat)
            mats = {e: tuple(q[3 * gi + a] for a in range(3)) for gi, e in enumerate(group)}

        def one(job):
            e, i, j = job
            if fp8:
                (cg, scg), (cu, scu), (cd, scd) = mats[e]
                y[i * k + j] = oracle.swiglu_row_fp8(qx[i], sx[i], cg, scg, cu, scu, cd, scd)
            else:
                y[i * k + j] = oracle.swiglu_row(xs[i], *mats[e])

        _pool_map(one, [(e, i, j) for e in group for (i, j) in pairs[e]])
        del mats
    allowance = None
    if fp8:  # the E4M3 combine payload (rows token-major: row i*k+j)
        y, y_codes, y_scale = oracle.payload_e4m3(y)
        wt_s = np.asarray(weight)[toks]
        allowance = payload_allowance(y_codes, y_scale, np.arange(n * k).reshape(n, k), wt_s, H)
    if w.n_shared == 0:
        ysh = np.zeros((n, H))
    elif fp8:
        ysh = np.stack(_pool_map(lambda i: oracle.shared_row_fp8(w, qx[i], sx[i], shared), range(n)))
    else:
        sg, su, sd = shared
        ysh = np.concatenate(_pool_map(lambda i: oracle.shared_rows(w, xs[i:i + 1], sg, su, sd), range(n)))
    wt = np.ascontiguousarray(np.asarray(weight)[toks], dtype=np.float64)
    out = oracle.combine(w.with_(tokens=n), n, y, np.arange(n * k, dtype=np.int32), wt, ysh)
    return (out, allowance) if fp8 else out


def check_full_size_layer(w, out_gpu, idx_gpu, counts_gpu, blocks_gpu, expert_host, shared, rep=None, fp8=False,
                          n_sample=SAMPLE_TOKENS, what="", x=None):
    """Parity of a full-size layer pass against the oracle.

    Routing of every token (oracle logits in fp64 on the host threads): top-k
    sets and order where decided; counts and block loads of the GPU's own
    routing, unconditionally.  Output: n_sample seeded random tokens with a
    decided selection, element by element.  x: the layer input the GPU ran
    (default: the workload's generated hidden states).  Returns the report
    record."""
    if x is None:
        x = mi.hidden_states(w)
    wr = mi.router_weight(w)
    b = mi.router_bias(w)
    lo = parallel_router_logits(w, x, wr, b)
    idx_o, wt_o = oracle.topk_softmax(lo, w.top_k)
    idx_g = np.asarray(idx_gpu)
    sure = check_topk(idx_g, idx_o, lo, w.top_k)
    ties = check_counts_of_routing(w, idx_g, counts_gpu, blocks_gpu, rep, idx_o, sure)
    toks = sample_tokens(sure, n_sample)
    ref = oracle_sampled_layer(w, toks, x, idx_o, wt_o, expert_host, shared, fp8=fp8)
    ref, allowance = ref if fp8 else (ref, None)
    stats = assert_close(np.asarray(out_gpu)[toks], ref, what=what or f"{w.name} sampled out", e4m3_layer=fp8,
                         allowance=allowance)
    rec = dict(stats, kind="full_size_layer", workload=w.name, precision="e4m3" if fp8 else "bf16",
               tokens=int(w.tokens), sampled_tokens=int(len(toks)), near_tie_tokens=ties)
    _report(rec)
    return rec


def fp8_layer_allowance(w, ref) -> np.ndarray:
    """payload_allowance of an oracle.moe_forward_fp8 result."""
    inv = ref["inv_perm"].reshape(-1, w.top_k)
    return payload_allowance(ref["y_codes"], ref["y_scale"], inv, ref["weight"], w.hidden)
