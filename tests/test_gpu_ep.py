"""Expert parallelism across ranks emulated on one GPU.

Each rank's steps are the product's (``moe_expert_layer_06_gb300.ep``:
routing and dispatch of its token shard, ``moe_ep_plan``, the slot-major
regroup and the local experts' GEMMs with ``moe_gather_rows`` around them,
the shared experts and the combine), all on libmoe kernels.  The two
all-to-alls are emulated by copying each (source, destination) segment, so no
kernel waits on another rank.  The layer output over all shards must match
the oracle and the single-GPU layer on the whole batch.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_06_gb300 as m
import moe_inputs as mi
import oracle
from moe_expert_layer_06_gb300 import ep
from moe_testlib import DeviceLayer, _report, assert_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"

SMALL = mi.WORKLOADS["tiny"].with_(name="ep_small", tokens=256, hidden=512, inter=256, n_experts=64, top_k=8,
                                   n_shared=1, inter_shared=256, n_slots=64, n_blocks=8, skew_alpha=1.5)


def _segments(counts, world, spb):
    """Row range of each destination rank's block in a dispatch buffer."""
    off = np.concatenate([[0], np.cumsum(counts[:world * spb])])
    return [(int(off[g * spb]), int(off[(g + 1) * spb])) for g in range(world)]


def _emulated_ep_layer(w, x, wr, bias, rep, weights, shared, logits=None):
    world = w.n_blocks
    T, S, H = w.tokens, w.n_slots, w.hidden
    spb = S // world
    shards = [(r * T // world, (r + 1) * T // world) for r in range(world)]
    experts = [ep.RankExperts(*(t[r * spb:(r + 1) * spb] for t in weights), *shared) for r in range(world)]
    repd = torch.from_numpy(rep).to(DEV) if rep is not None else None
    # steps 1-2 on every rank
    ds = [ep.local_dispatch(w, t1 - t0, x[t0:t1], wr, bias, repd,
                            logits=None if logits is None else logits[t0:t1]) for t0, t1 in shards]
    counts = [d.counts.cpu().numpy() for d in ds]
    seg = [_segments(c, world, spb) for c in counts]
    # counts all-to-all and plans
    plans = []
    for r in range(world):
        recv_counts = np.stack([counts[s][r * spb:(r + 1) * spb] for s in range(world)])
        plans.append(m.moe_ep_plan(w, world, counts[r], recv_counts))
    # dispatch all-to-all: rank r receives block r's segment of every source, source-major
    recv = [torch.cat([ds[s].x_disp[seg[s][r][0]:seg[s][r][1]] for s in range(world)]) for r in range(world)]
    # step 3 on every rank
    y_src = [ep.expert_rows(w, world, plans[r], recv[r], experts[r]) for r in range(world)]
    # combine all-to-all: each source's segment returns to its dispatch-buffer positions
    y_disp = [torch.empty_like(d.x_disp) for d in ds]
    for r in range(world):
        p0 = 0
        for s in range(world):
            a, b = seg[s][r]
            y_disp[s][a:b] = y_src[r][p0:p0 + (b - a)]
            p0 += b - a
    outs = []
    for r, (t0, t1) in enumerate(shards):
        out = torch.empty((t1 - t0, H), dtype=torch.bfloat16, device=DEV)
        ep.finish(w, t1 - t0, x[t0:t1], experts[r], y_disp[r], ds[r], out)
        outs.append(out)
    assert m.moe_check_status() == 0, m.last_error()
    return torch.cat(outs), plans, ds


def _replica_plan(w):
    base = w.with_(n_slots=w.n_experts)
    lo = oracle.router_logits(base, mi.hidden_states(base), mi.router_weight(base), mi.router_bias(base))
    idx, _ = oracle.topk_softmax(lo, base.top_k)
    return oracle.plan_replicas(w, np.bincount(idx.ravel(), minlength=w.n_experts), w.n_slots - w.n_experts)


def _single_gpu_from_logits(w, layer, logits, rep):
    """The layer on the whole batch through the staged calls, routed from fp32 logits."""
    T, k, S, H, n = w.tokens, w.top_k, w.n_slots, w.hidden, w.tokens * w.top_k
    i32 = dict(dtype=torch.int32, device=DEV)
    idx, tw = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device=DEV)
    m.moe_route(w, T, None, None, None, logits, None, idx, tw, None)
    off, inv, xd = torch.empty(S + 2, **i32), torch.empty(n, **i32), torch.empty((n, H), dtype=torch.bfloat16,
                                                                                 device=DEV)
    m.moe_dispatch(w, T, layer.x, idx, layer.replica_of, torch.empty(n, **i32), torch.empty(S + 1, **i32), None, off,
                   torch.empty(n, **i32), inv, xd)
    y, ysh = torch.empty_like(xd), torch.empty((T, H), dtype=torch.float32, device=DEV)
    ws = torch.empty(m.moe_ffn_workspace_size(w, T), dtype=torch.uint8, device=DEV)
    m.moe_expert_ffn(w, T, layer.x, xd, off, layer.wg, layer.wu, layer.wd, layer.sg, layer.su, layer.sd, y, ysh,
                     m.MOE_FFN_AUTO, ws)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    m.moe_combine(w, T, y, inv, tw, ysh, out)
    return out


def _within_two_ulps(a, b):
    ulp = np.ldexp(1.0, (np.floor(np.log2(np.maximum(np.abs(b), 2.0 ** -120))) - 7).astype(np.int64))
    assert np.all(np.abs(a - b) <= 2 * ulp), np.abs(a - b).max()
    assert np.linalg.norm(a - b) <= 1e-3 * np.linalg.norm(b)
    return int((a != b).sum())


def _oracle_from_logits(w, x, logits, rep, weights, shared):
    """The oracle's layer routed from the same fp32 logits."""
    T, k = w.tokens, w.top_k
    idx, wt = oracle.topk_softmax(logits.double().cpu().numpy(), k)
    so, _ = oracle.slot_map(w, idx, rep)
    counts, _ = oracle.histogram(w, so)
    off, _, inv, xd = oracle.dispatch(w, T, so, counts, x.cpu())
    y = oracle.expert_ffn(w, T, off, xd, *(t.cpu() for t in weights))
    ysh = oracle.shared_rows(w, x.cpu(), *(t.cpu() for t in shared))
    return oracle.combine(w, T, y, inv, wt, ysh)


@pytest.mark.parametrize("case", ["small_8_ranks", "small_4_ranks_replicas", "dsv3_decode_8_ranks"])
def test_ep_ranks_on_one_gpu_match_the_single_gpu_layer(case):
    """Routed from the same fp32 logits, the EP layer matches the oracle within
    the layer tolerance and the single-GPU layer within two bf16 ulps: the
    tensor cores' fp32 sums depend on how rows are grouped into token chunks
    (a rank's 32-row shard against a 160-row chunk of the whole batch), so an
    output can move by an ulp.  Routed by the router GEMM (whose K split also
    follows the batch size, so a near-tie can resolve either way), at least 99%
    of the tokens select alike and those agree within the layer tolerance."""
    if case == "small_8_ranks":
        w, rep = SMALL, None
    elif case == "small_4_ranks_replicas":
        w = SMALL.with_(n_blocks=4, n_slots=SMALL.n_experts + 4)
        rep = _replica_plan(w)
    else:  # the DeepSeek-V3 layer, 8 ranks of a 32-token decode batch each
        w, rep = mi.WORKLOADS["decode_t32"].with_(tokens=256), None
    layer = DeviceLayer(w, DEV, replica_of=rep)
    shared = (layer.sg, layer.su, layer.sd) if w.n_shared else (None, None, None)
    weights = (layer.wg, layer.wu, layer.wd)
    logits = mi.fp32_logits(w, device=DEV)
    ref = _single_gpu_from_logits(w, layer, logits, rep)
    out, plans, _ = _emulated_ep_layer(w, layer.x, layer.wr, layer.bias, rep, weights, shared, logits)
    # every assignment crossed to the rank of its slot exactly once
    assert sum(p["rows"] for p in plans) == w.tokens * w.top_k
    differ = _within_two_ulps(to_np(out), to_np(ref))
    _report(dict(kind="ep_vs_single_gpu", what=case, elements=int(out.numel()), differing=differ))
    if case != "dsv3_decode_8_ranks":
        assert_close(to_np(out), _oracle_from_logits(w, layer.x, logits, rep, weights, shared),
                     what=f"{case}: EP layer vs oracle")
    # the router GEMM path of both, on the tokens whose top-k both select alike (a near-tie can go
    # either way when the logits differ in their last bits)
    out2, _, ds2 = _emulated_ep_layer(w, layer.x, layer.wr, layer.bias, rep, weights, shared)
    idx2, tw2 = torch.cat([d.idx for d in ds2]), torch.cat([d.topk_w for d in ds2])
    r = layer.forward()
    same = (idx2 == r["idx"]).all(dim=1).cpu().numpy()
    assert same.mean() >= 0.99
    a, b = to_np(out2), to_np(r["out"])
    t_w, c_w = np.unravel_index(np.argmax(np.abs(a - b) * same[:, None]), a.shape)
    _report(dict(kind="ep_vs_single_gpu_router_gemm", what=case, same_selection=float(same.mean()),
                 differing=int((a[same] != b[same]).sum()), worst_token=int(t_w), worst_col=int(c_w),
                 ep=float(a[t_w, c_w]), single=float(b[t_w, c_w]),
                 topk_w_max_rel_diff=float(((tw2[t_w] - r["w"][t_w]).abs() / r["w"][t_w].abs()).max())))
    assert_close(a[same], b[same], what=f"{case}: EP vs single GPU, router GEMM")
    del layer
    torch.cuda.empty_cache()


def test_gather_rows_moves_whole_rows():
    src = torch.arange(7 * 48, dtype=torch.int32, device=DEV).view(7, 48).to(torch.uint8)  # 48-byte rows
    idx = torch.tensor([6, 0, 3, 3, 1], dtype=torch.int32, device=DEV)
    dst = torch.empty((5, 48), dtype=torch.uint8, device=DEV)
    m.moe_gather_rows(src, idx, dst)
    assert m.moe_check_status() == 0
    assert torch.equal(dst, src[idx.long()])
