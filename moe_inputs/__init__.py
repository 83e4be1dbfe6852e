"""Seeded synthetic inputs for the DeepSeek-V3-style MoE layer.

This module is the only code shared by the CUDA library's callers and by the
CPU oracle's callers.  It holds workload definitions (shapes, seeds, routing
skew) and a counter-based value generator; it holds none of the layer's
arithmetic (no routing, no permutation, no FFN, no combine).

Value generator
---------------
Every tensor is a pure function of (seed, tensor id, logical expert id,
element index), so a caller can regenerate one expert's weights without
generating the others, and the CPU and the GPU produce identical bits.

* A 32-bit integer hash ("PCG hash": one LCG step followed by a random
  xorshift and a multiply, Jarzynski and Olano, "Hash Functions for GPU
  Rendering", JCGT 2020) is applied twice per element:
  ``o = pcg(pcg(i) ^ key)``, with ``key`` derived from the stream triple.
* The four bytes of ``o`` are summed (Irwin-Hall sum of four discrete
  uniforms on 0..255: mean 510, variance 4*(256**2-1)/12), centred and
  scaled to unit variance.  This is an approximately normal variate bounded
  at +-3.45 sigma with 1021 levels.
* One float32 multiply by ``std / 147.8006...`` and a round-to-nearest-even
  cast to bf16 finish the value.

Only integer ops, one IEEE float32 multiply and one IEEE rounding are used, so
``torch`` gives the same bits on CPU and CUDA (the constants stay below 2**30,
so no int64 product overflows).

Workloads
---------
The five workloads are the DeepSeek-V3 MoE layer (hidden 7168, 256 routed
experts with SwiGLU intermediate 2048, top-8, two shared experts) at a decode
batch of 32 tokens, a skewed decode batch of 256, a 4096-token prefill, and a
1024-token skewed batch with 8 redundant expert slots; plus a tiny layer
(hidden 64, 8 experts, intermediate 32, top-2, one shared expert) that the
oracle finishes in well under a second.  The expert layout (256 experts in 8
contiguous blocks of 32, shared experts replicated) follows the blog post
"专家并行(EP)", section 2.1; the 264-slot redundant layout follows its
section 6.3.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np
import torch

M32 = 0xFFFFFFFF

# tensor ids of the generator streams
TID_X = 1
TID_ROUTER = 2
TID_GATE = 3
TID_UP = 4
TID_DOWN = 5
TID_SH_GATE = 6
TID_SH_UP = 7
TID_SH_DOWN = 8
TID_LOGITS = 9

_IH_MEAN = 510
_IH_STD = math.sqrt(4.0 * (256.0 ** 2 - 1.0) / 12.0)  # 147.8006...


def _pcg(v: torch.Tensor) -> torch.Tensor:
    """32-bit PCG hash on int64 tensors holding values in [0, 2**32)."""
    state = (v * 747796405 + 2891336453) & M32
    word = (((state >> ((state >> 28) + 4)) ^ state) * 277803737) & M32
    return (word >> 22) ^ word


def _pcg_int(v: int) -> int:
    state = (v * 747796405 + 2891336453) & M32
    word = (((state >> ((state >> 28) + 4)) ^ state) * 277803737) & M32
    return (word >> 22) ^ word


def stream_key(seed: int, tensor_id: int, expert: int) -> int:
    return _pcg_int(_pcg_int(_pcg_int(seed & M32) ^ tensor_id) ^ (expert & M32))


_counter_cache: Dict[str, torch.Tensor] = {}


def _hashed_counter(n: int, device: torch.device) -> torch.Tensor:
    """pcg(i) for i in [0, n), cached per device (grown on demand)."""
    key = str(device)
    cached = _counter_cache.get(key)
    if cached is None or cached.numel() < n:
        size = max(n, 1 << 20)
        cached = _pcg(torch.arange(size, dtype=torch.int64, device=device))
        _counter_cache[key] = cached
    return cached[:n]


def clear_cache() -> None:
    _counter_cache.clear()


def normal_bf16(shape, std: float, seed: int, tensor_id: int, expert: int = 0,
                device="cpu", offset: int = 0) -> torch.Tensor:
    """Approximately N(0, std**2) bf16 tensor from stream (seed, tensor_id, expert).

    ``offset`` skips that many elements of the stream (row slices of a tensor
    regenerate exactly: rows r0..r1 of a [R, C] tensor are elements
    r0*C .. r1*C).
    """
    n = int(np.prod(shape)) if len(shape) else 1
    assert offset + n <= (1 << 32)
    device = torch.device(device)
    key = stream_key(seed, tensor_id, expert)
    base = _hashed_counter(offset + n, device)[offset:offset + n]
    o = _pcg(base ^ key)
    s = (o & 255) + ((o >> 8) & 255) + ((o >> 16) & 255) + (o >> 24)
    z = (s - _IH_MEAN).to(torch.float32)
    scale = torch.tensor(float(np.float32(std / _IH_STD)), dtype=torch.float32, device=device)
    return (z * scale).to(torch.bfloat16).reshape(shape)


def normal_bf16_experts(shape, std: float, seed: int, tensor_id: int, experts, device="cpu") -> torch.Tensor:
    """normal_bf16 for several streams at once: result [len(experts), *shape].

    Row e of the result equals normal_bf16(shape, std, seed, tensor_id, experts[e]).
    """
    n = int(np.prod(shape))
    device = torch.device(device)
    keys = torch.tensor([stream_key(seed, tensor_id, int(e)) for e in experts], dtype=torch.int64, device=device)
    base = _hashed_counter(n, device)
    o = _pcg(base[None, :] ^ keys[:, None])
    s = (o & 255) + ((o >> 8) & 255) + ((o >> 16) & 255) + (o >> 24)
    del o
    z = (s - _IH_MEAN).to(torch.float32)
    del s
    scale = torch.tensor(float(np.float32(std / _IH_STD)), dtype=torch.float32, device=device)
    return (z * scale).to(torch.bfloat16).reshape((len(experts),) + tuple(shape))


def uniform_f32(shape, lo: float, hi: float, seed: int, tensor_id: int, expert: int = 0,
                device="cpu") -> torch.Tensor:
    """Float32 values on a 2**-24 grid of [lo, hi) from the same hash stream."""
    n = int(np.prod(shape))
    device = torch.device(device)
    key = stream_key(seed, tensor_id, expert)
    o = _pcg(_hashed_counter(n, device) ^ key)
    u = (o >> 8).to(torch.float32) * float(2.0 ** -24)
    return (u * float(hi - lo) + float(lo)).reshape(shape)


# --------------------------------------------------------------------------------------
# Workload definitions
# --------------------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tokens: int
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    n_shared: int
    inter_shared: int
    n_slots: int
    n_blocks: int
    router_std: float
    skew_alpha: float       # 0 = no bias (near-uniform routing)
    seed: int = 0
    description: str = ""

    @property
    def shape_tuple(self):
        return (self.hidden, self.inter, self.n_experts, self.top_k, self.n_shared,
                self.inter_shared, self.n_slots, self.n_blocks)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _dsv3(name, tokens, alpha, n_slots=256, description=""):
    return Workload(name=name, tokens=tokens, hidden=7168, inter=2048, n_experts=256, top_k=8,
                    n_shared=2, inter_shared=2048, n_slots=n_slots, n_blocks=8,
                    router_std=0.02, skew_alpha=alpha, description=description)


WORKLOADS = {
    "tiny": Workload(name="tiny", tokens=16, hidden=64, inter=32, n_experts=8, top_k=2,
                     n_shared=1, inter_shared=32, n_slots=8, n_blocks=8, router_std=0.02,
                     skew_alpha=0.0,
                     description="tiny layer: T=16, hidden 64, 8 experts, inter 32, top-2, 1 shared"),
    "decode_t32": _dsv3("decode_t32", 32, 0.0,
                        description="DeepSeek-V3 MoE layer decode step, T=32, near-uniform routing"),
    "decode_t256_skew": _dsv3("decode_t256_skew", 256, 1.5,
                              description="decode T=256, long-tail routing bias 1.5*log(1/(rank+1))"),
    # the same batch with the bias calibrated to the pages' load picture (about 30% of
    # the experts take about 60% of the assignments); the literal 1.5 gives ~98%
    "decode_t256_skew_a05": _dsv3("decode_t256_skew_a05", 256, 0.5,
                                  description="decode T=256, routing bias 0.5*log(1/(rank+1)): ~30% of "
                                              "the experts take ~60% of the assignments"),
    "prefill_t4096": _dsv3("prefill_t4096", 4096, 0.0,
                           description="prefill T=4096 (one 4k-token prompt), uniform routing"),
    "redundant_t1024": _dsv3("redundant_t1024", 1024, 1.5, n_slots=264,
                             description="T=1024 skewed routing, 256+8 slots, 8 hottest experts replicated"),
    # more experts of the same shape (the group-limited routing row's 512/1024-expert scaling)
    "decode_t32_e512": Workload(name="decode_t32_e512", tokens=32, hidden=7168, inter=2048, n_experts=512,
                                top_k=8, n_shared=2, inter_shared=2048, n_slots=512, n_blocks=8,
                                router_std=0.02, skew_alpha=0.0,
                                description="decode T=32, DeepSeek-V3 expert shapes, 512 experts (8 blocks of 64)"),
    "decode_t32_e1024": Workload(name="decode_t32_e1024", tokens=32, hidden=7168, inter=2048, n_experts=1024,
                                 top_k=8, n_shared=2, inter_shared=2048, n_slots=1024, n_blocks=8,
                                 router_std=0.02, skew_alpha=0.0,
                                 description="decode T=32, DeepSeek-V3 expert shapes, 1024 experts (8 blocks of 128)"),
    # profiling cases: the same per-expert shapes and rows per expert with 32 experts
    # (2.8 GB of expert weights), small enough for multi-pass hardware-counter captures
    "decode_t32_e32": Workload(name="decode_t32_e32", tokens=32, hidden=7168, inter=2048, n_experts=32,
                               top_k=8, n_shared=2, inter_shared=2048, n_slots=32, n_blocks=8,
                               router_std=0.02, skew_alpha=0.0,
                               description="profiling case: DeepSeek-V3 expert shapes, 32 experts, T=32"),
    "prefill_t512_e32": Workload(name="prefill_t512_e32", tokens=512, hidden=7168, inter=2048, n_experts=32,
                                 top_k=8, n_shared=2, inter_shared=2048, n_slots=32, n_blocks=8,
                                 router_std=0.02, skew_alpha=0.0,
                                 description="profiling case: DeepSeek-V3 expert shapes, 32 experts, "
                                             "T=512 (128 rows per expert, as prefill T=4096)"),
    "decode_t128_e32": Workload(name="decode_t128_e32", tokens=128, hidden=7168, inter=2048, n_experts=32,
                                top_k=8, n_shared=2, inter_shared=2048, n_slots=32, n_blocks=8,
                                router_std=0.02, skew_alpha=0.0,
                                description="profiling case: DeepSeek-V3 expert shapes, 32 experts, "
                                            "T=128 (32 rows per expert, as T=1024 over 256 experts)"),
}

# the skewed decode workload whose histogram chooses the 8 replicated experts
REPLICA_PLAN_SOURCE = "decode_t256_skew"
N_REPLICAS = 8


def expert_ranking(n_experts: int, seed: int) -> np.ndarray:
    """Seeded random ranking of the experts: rank[e] in 0..E-1."""
    rng = np.random.Generator(np.random.PCG64([seed, 0x5EED]))
    perm = rng.permutation(n_experts)
    rank = np.empty(n_experts, dtype=np.int64)
    rank[perm] = np.arange(n_experts)
    return rank


def router_bias(w: Workload) -> Optional[np.ndarray]:
    """Per-expert logit bias b_e = alpha*log(1/(rank_e+1)) (fp32), or None."""
    if w.skew_alpha == 0.0:
        return None
    rank = expert_ranking(w.n_experts, w.seed)
    return (w.skew_alpha * np.log(1.0 / (rank + 1.0))).astype(np.float32)


def hidden_states(w: Workload, device="cpu", rows: Optional[slice] = None) -> torch.Tensor:
    """x [T, H] bf16 ~ N(0,1); ``rows`` regenerates a row range only."""
    if rows is None:
        return normal_bf16((w.tokens, w.hidden), 1.0, w.seed, TID_X, 0, device)
    r0, r1 = rows.start, rows.stop
    return normal_bf16((r1 - r0, w.hidden), 1.0, w.seed, TID_X, 0, device, offset=r0 * w.hidden)


def with_outliers(x: torch.Tensor, seed: int, per_row: int = 2, lo: float = 8.0, hi: float = 20.0) -> torch.Tensor:
    """A copy of x [T, H] (unit-variance rows) with per_row seeded entries of every
    row replaced by outliers of magnitude lo..hi (in units of the row's standard
    deviation, 1) and random sign, rounded to bf16: heavy tails the bounded
    generator (+-3.45 sigma) never produces."""
    T, H = x.shape
    rng = np.random.Generator(np.random.PCG64([seed, 0x0D7]))
    cols = np.stack([rng.choice(H, size=per_row, replace=False) for _ in range(T)])
    mag = rng.uniform(lo, hi, size=(T, per_row)) * rng.choice([-1.0, 1.0], size=(T, per_row))
    out = x.clone()
    rows = torch.arange(T)[:, None].expand(T, per_row)
    out[rows, torch.from_numpy(cols)] = torch.from_numpy(mag).to(torch.float32).to(torch.bfloat16).to(x.device)
    return out


def router_weight(w: Workload, device="cpu") -> torch.Tensor:
    """W_r stored [E, H] (row e = expert e's router vector), bf16 ~ N(0, 0.02**2)."""
    return normal_bf16((w.n_experts, w.hidden), w.router_std, w.seed, TID_ROUTER, 0, device)


def expert_weights(w: Workload, expert: int, device="cpu"):
    """(gate [I,H], up [I,H], down [H,I]) bf16 of logical expert ``expert``.

    nn.Linear layout [out, in]; std 1/sqrt(fan_in).
    """
    H, I = w.hidden, w.inter
    g = normal_bf16((I, H), 1.0 / math.sqrt(H), w.seed, TID_GATE, expert, device)
    u = normal_bf16((I, H), 1.0 / math.sqrt(H), w.seed, TID_UP, expert, device)
    d = normal_bf16((H, I), 1.0 / math.sqrt(I), w.seed, TID_DOWN, expert, device)
    return g, u, d


def shared_weights(w: Workload, j: int, device="cpu"):
    H, I = w.hidden, w.inter_shared
    g = normal_bf16((I, H), 1.0 / math.sqrt(H), w.seed, TID_SH_GATE, j, device)
    u = normal_bf16((I, H), 1.0 / math.sqrt(H), w.seed, TID_SH_UP, j, device)
    d = normal_bf16((H, I), 1.0 / math.sqrt(I), w.seed, TID_SH_DOWN, j, device)
    return g, u, d


def home_slot(w: Workload, e: int) -> int:
    """Slot of expert e's own copy: blocks keep experts in order, replica slots last."""
    epb = w.n_experts // w.n_blocks
    spb = w.n_slots // w.n_blocks
    return (e // epb) * spb + (e % epb)


def slot_experts(w: Workload, replica_of: Optional[np.ndarray]) -> np.ndarray:
    """Logical expert held by each slot (-1 for an unused replica slot)."""
    se = np.full(w.n_slots, -1, dtype=np.int64)
    for e in range(w.n_experts):
        se[home_slot(w, e)] = e
    if replica_of is not None:
        for e in range(w.n_experts):
            if replica_of[e] >= 0:
                se[int(replica_of[e])] = e
    return se


def stacked_expert_weights(w: Workload, replica_of: Optional[np.ndarray] = None, device="cpu",
                           slots=None):
    """Slot-major weights W_g[S,I,H], W_u[S,I,H], W_d[S,H,I] (bf16).

    A replica slot holds a byte copy of its source expert; an unused slot is
    zero.  ``slots`` restricts generation to a subset (others stay zero).
    """
    S, H, I = w.n_slots, w.hidden, w.inter
    device = torch.device(device)
    wg = torch.zeros((S, I, H), dtype=torch.bfloat16, device=device)
    wu = torch.zeros((S, I, H), dtype=torch.bfloat16, device=device)
    wd = torch.zeros((S, H, I), dtype=torch.bfloat16, device=device)
    se = slot_experts(w, replica_of)
    todo = [s for s in range(S) if se[s] >= 0 and (slots is None or s in slots)]
    # several experts per generator call on a GPU (fewer launches), one at a time on the host
    batch = max(1, min(16, (1 << 27) // max(1, H * I))) if device.type == "cuda" else 1
    for i in range(0, len(todo), batch):
        sl = todo[i:i + batch]
        ex = [int(se[s]) for s in sl]
        idx = torch.tensor(sl, dtype=torch.int64, device=device)
        wg.index_copy_(0, idx, normal_bf16_experts((I, H), 1.0 / math.sqrt(H), w.seed, TID_GATE, ex, device))
        wu.index_copy_(0, idx, normal_bf16_experts((I, H), 1.0 / math.sqrt(H), w.seed, TID_UP, ex, device))
        wd.index_copy_(0, idx, normal_bf16_experts((H, I), 1.0 / math.sqrt(I), w.seed, TID_DOWN, ex, device))
    return wg, wu, wd


def stacked_shared_weights(w: Workload, device="cpu"):
    """Shared experts Ws_g[n_sh,I_sh,H], Ws_u[n_sh,I_sh,H], Ws_d[n_sh,H,I_sh] (bf16)."""
    gs, us, ds = zip(*(shared_weights(w, j, device) for j in range(w.n_shared)))
    return torch.stack(gs), torch.stack(us), torch.stack(ds)


def fp32_logits(w: Workload, device="cpu") -> torch.Tensor:
    """Synthetic fp32 router logits [T, E] for the route-from-logits path.

    Values lie on a coarse grid (multiples of 2**-10 in [-4, 4)) so that exact
    ties occur and the tie rule is exercised; the skew bias is added.
    """
    u = uniform_f32((w.tokens, w.n_experts), -4.0, 4.0, w.seed, TID_LOGITS, 0, device)
    u = torch.floor(u * 1024.0) / 1024.0
    b = router_bias(w)
    if b is not None:
        u = u + torch.from_numpy(b).to(device)
    return u.contiguous()
