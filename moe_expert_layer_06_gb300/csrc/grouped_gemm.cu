// Grouped swap-AB GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA: the expert FFN of the MoE layer (gate/up + SwiGLU, and down) and
// the router linear.
//
// Expert-parallel layer of the blog post "专家并行(EP)", section 2.2, step 3:
// every expert computes its FFN on the token rows dispatched to it.  The
// weights are the large operand (88 MB per expert; a decode step touches
// ~160 experts), tokens the small one (a few to a few hundred rows per
// expert).  So the weight matrix is the UMMA "A" operand (M = 128 output
// rows per tile) and the expert's token rows the "B" operand (N = up to BN
// rows, rounded up to 16): each weight tile streams from HBM once per token
// chunk.  BN is 32 at decode (five 36 KB pipeline stages) and 160 above 32
// tokens (four 52 KB stages), which covers every expert of a 4096-token
// batch with uniform routing in one chunk; the chunks of one expert that
// needs more run at the same time on different SMs and share its weights
// through L2.
//
// Work item = (matrix, 128-row block of outputs, token chunk[, K split]);
// a gate/up item carries the gate and the up tile of the same rows, a down
// item two consecutive 128-row tiles.  E4M3 modes use 128-element K chunks.
// The item list is derived on the device from the dispatch offsets, so no
// host synchronisation is needed.  A persistent CTA per SM takes items
// round-robin; warp roles:
//   warp 0      TMA producer (one elected lane)   smem ring of STAGES stages
//   warp 1      MMA issuer   (one elected lane)   TMEM accumulators: two when they
//                                                 fit; the 160-row E4M3 down rotates
//                                                 three one-tile slots instead
//   warps 2..17 epilogue: tcgen05.ld -> SwiGLU / dequantise / E4M3 payload ->
//               global stores (bf16 as two-row words, payload codes as words)
// Every mbarrier wait is bounded; on expiry the kernel raises the status word,
// drains its own copies and MMAs (bounded) and frees its TMEM.
#include <cuda_fp8.h>

#include <type_traits>

#include "e4m3.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kEpiWarps = 16;          // 4 per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kABytes = 128 * 64 * 2;  // one 128x64 bf16 weight tile
constexpr int kMaxSlots = 1024;

struct Item {
    int shared;  // 0: routed or router, 1: shared expert
    int z;       // slot | shared expert | 0
    int m0;      // first output row of the A tile
    int row0;    // first B row
    int nrows;   // valid B rows (<= BN)
    int kc0, kc1;
    int ks;      // router K split
    int shared_a;  // the A tile is also read by other token chunks (keep it in L2 for them)
};

// Gate/up items carry the gate and the up tile of the same 128 rows; down items
// carry two consecutive 128-row tiles of W_d (256 output rows); router items one
// tile.  Two weight tiles per stage keep twice the weight bytes in flight per
// token-chunk byte.
template <int MODE>
struct Traits {
    static constexpr bool kF8 = (MODE == kGateUpF8 || MODE == kDownF8 || MODE == kDownF8Q);  // E4M3 operands
    static constexpr bool kDownLike = (MODE == kDown || MODE == kDownF8 || MODE == kDownF8Q);
    static constexpr bool kDownF8Like = (MODE == kDownF8 || MODE == kDownF8Q);
    static constexpr bool kGateUpLike = (MODE == kGateUp || MODE == kGateUpF8);
    static constexpr int NA = (MODE == kRouter) ? 1 : 2;
    static constexpr int kRowsPerItem = kDownLike ? 256 : 128;
    // elements of K per 128-byte smem row (one pipeline chunk)
    static constexpr int kChunkK = kF8 ? 128 : 64;
};

__host__ __device__ constexpr int pow2_at_least(int v) {
    int p = 32;
    while (p < v) p <<= 1;
    return p;
}

template <int MODE, int BN, int STAGES>
struct Config {
    static constexpr int NA = Traits<MODE>::NA;
    static constexpr int kBBytes = BN * 64 * 2;
    static constexpr int kStageBytes = NA * kABytes + kBBytes;
    static constexpr int kAccCols = NA * BN;
    // E4M3 down items whose two tiles' accumulators cannot be double-buffered rotate
    // three one-tile slots instead: tile u = 2 * (item ordinal) + half goes to slot
    // u % 3, so the next item's first tile starts at once and its second tile waits
    // only for the first half of the previous item's epilogue.  An E4M3 down item is
    // 16 K chunks, so its epilogue is a large share of it (4096 tokens, 160-row
    // chunks: 957 against 1010 us); the bf16 down item is twice as long and was
    // slower with the rotation (1446 against 1392 us), so it keeps one accumulator.
    static constexpr bool kRot = Traits<MODE>::kDownF8Like && 2 * kAccCols > 512 && 3 * BN <= 512;
    static constexpr int kNumAcc = kRot ? 3 : (2 * kAccCols <= 512) ? 2 : 1;
    static constexpr int kTmemCols = pow2_at_least(kRot ? 3 * BN : kNumAcc * kAccCols);
    static constexpr int kBarBytes = (2 * STAGES + 2 * kNumAcc + 1) * 8;
    static constexpr int kTableBytes = (kMaxSlots + 4) * 4;
    // column groups of 16 tokens one epilogue warp drains per item
    static constexpr int kMaxG = (BN / 16 + kEpiWarps / 4 - 1) / (kEpiWarps / 4);
    // kDownF8Q: per-warp column maxima exchanged by the four warps that share columns
    // (two mbarriers per group of four warps, then the maxima)
    static constexpr int kXchgBytes = MODE == kDownF8Q ? 64 + (kEpiWarps / 4) * 4 * kMaxG * 2 * 16 * 4 : 0;
    static constexpr int kSmemBytes = 1024 + STAGES * kStageBytes + kBarBytes + 16 + kTableBytes + kXchgBytes;
    static_assert(kTmemCols <= 512, "TMEM overflow");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory overflow");
    static_assert(BN <= 15 * 16, "token chunk must be at most 15 groups of 16 rows");
};

// Shared-memory table of the routed items of this launch.
struct Table {
    int* pre;   // [S+1] exclusive prefix of routed items per slot
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

template <int MODE, int BN>
__device__ __forceinline__ Item decode_item(int i, const GemmArgs& a, const Table& tb, int n_sh_items) {
    Item it;
    it.ks = 0;
    if (MODE == kRouter) {
        const int chunks = cdiv(a.T, BN);
        it.shared = 0;
        it.z = 0;
        it.ks = i % a.ksplit;
        const int r = i / a.ksplit;
        const int c = r % chunks;
        it.m0 = (r / chunks) * 128;
        it.row0 = c * BN;
        it.nrows = min(BN, a.T - it.row0);
        it.kc0 = it.ks * a.kc_split;
        it.kc1 = min(a.kc_routed, it.kc0 + a.kc_split);
        it.shared_a = chunks > 1;
        return it;
    }
    constexpr int RPI = Traits<MODE>::kRowsPerItem;
    if (i < n_sh_items) {
        const int chunks = cdiv(a.T, BN);
        const int mb = cdiv(a.m_shared, RPI);
        it.shared = 1;
        int r = i;
        if (Traits<MODE>::kGateUpLike) {
            it.z = r / (mb * chunks);
            r -= it.z * mb * chunks;
        } else {
            it.z = 0;
        }
        it.m0 = (r / chunks) * RPI;
        it.row0 = (r % chunks) * BN;
        it.nrows = min(BN, a.T - it.row0);
        it.kc0 = 0;
        it.kc1 = a.kc_shared;
        it.shared_a = chunks > 1;
        return it;
    }
    i -= n_sh_items;
    // slot s: the last slot with pre[s] <= i (pre is non-decreasing)
    int lo = 0, hi = a.n_slots - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tb.pre[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int l = i - tb.pre[s];
    const int off = __ldg(a.offsets + s);
    const int cnt = __ldg(a.offsets + s + 1) - off;
    const int chunks = cdiv(cnt, BN);
    const int c = l % chunks;
    it.shared = 0;
    it.z = s;
    it.m0 = (l / chunks) * RPI;
    it.row0 = off + c * BN;
    it.nrows = min(BN, cnt - c * BN);
    it.kc0 = 0;
    it.kc1 = a.kc_routed;
    it.shared_a = chunks > 1;
    return it;
}

// SwiGLU gate.  h is rounded to bf16 right after, 2^14 times coarser than the
// approximate division's error, so the fast divide is enough.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

template <int MODE, int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmArgs a) {
    pdl_launch_dependents();
    using C = Config<MODE, BN, STAGES>;
    constexpr int NA = C::NA;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + C::kNumAcc;
    uint64_t* mma_done = tempty + C::kNumAcc;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    Table tb{reinterpret_cast<int*>(tmem_slot + 4)};
    // kDownF8Q exchange: xfull[p] / xfree[p] (four warps arrive on each), then the maxima
    uint64_t* xbar = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(tmem_slot + 4) + C::kTableBytes);
    float* xchg = reinterpret_cast<float*>(xbar + 8);
    (void)xchg;
    constexpr int RPI = Traits<MODE>::kRowsPerItem;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long limit = a.st.limit_ns;

    // ---- setup (reads nothing a predecessor writes): barriers, descriptors, TMEM
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int s = 0; s < C::kNumAcc; ++s) {
            mbar_init(smem_u32(&tfull[s]), 1);
            mbar_init(smem_u32(&tempty[s]), kEpiWarps);
        }
        mbar_init(smem_u32(mma_done), 1);
        if (MODE == kDownF8Q)
            for (int p = 0; p < 8; ++p) mbar_init(smem_u32(&xbar[p]), 4);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&a.a0);
        tma_prefetch_desc(&a.b[0]);
        if (NA == 2) tma_prefetch_desc(&a.a1);
        if (MODE != kRouter && a.n_shared > 0) {
            tma_prefetch_desc(&a.sa0);
            tma_prefetch_desc(&a.sb[0]);
            if (NA == 2) tma_prefetch_desc(&a.sa1);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    // ---- everything below reads the predecessor's results (offsets, activations)
    pdl_wait();

    // ---- work list: shared items first, then routed items slot by slot
    int n_sh_items = 0;
    if (MODE != kRouter && a.n_shared > 0) {
        const int chunks = cdiv(a.T, BN);
        const int mb = cdiv(a.m_shared, RPI);
        n_sh_items = (Traits<MODE>::kGateUpLike ? a.n_shared : 1) * mb * chunks;
    }
    int n_items;
    if (MODE == kRouter) {
        n_items = cdiv(a.m_routed, 128) * cdiv(a.T, BN) * a.ksplit;
    } else {
        if (warp == 0) {
            const int S = a.n_slots;
            const int per = cdiv(S, 32);
            const int s0 = min(S, lane * per), s1 = min(S, s0 + per);
            const int mb = cdiv(a.m_routed, RPI);
            int sum = 0;
            for (int s = s0; s < s1; ++s) sum += cdiv(a.offsets[s + 1] - a.offsets[s], BN) * mb;
            int incl = sum;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += v;
            }
            int run = incl - sum;
            for (int s = s0; s < s1; ++s) {
                tb.pre[s] = run;
                run += cdiv(a.offsets[s + 1] - a.offsets[s], BN) * mb;
            }
            if (lane == 31) tb.pre[S] = incl;
        }
        __syncthreads();
        n_items = n_sh_items + tb.pre[a.n_slots];
    }
    if ((int)blockIdx.x >= n_items) {  // uniform across the CTA: nothing to do
        if (warp == 1) tmem_dealloc(tbase, C::kTmemCols);
        return;
    }

    if (warp == 0) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            // weights stream through L2 once (evict first) unless other token chunks of
            // the same rows will read them too (evict normal, so those chunks hit)
            const uint64_t pol_w1 = policy_evict_first();
            const uint64_t pol_wn = policy_evict_normal();
            const uint64_t pol_x = policy_evict_last();
            uint32_t armed[STAGES];
            for (int s = 0; s < STAGES; ++s) armed[s] = 2;  // 2 = never armed
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
                const Item it = decode_item<MODE, BN>(i, a, tb, n_sh_items);
                const CUtensorMap* ma0 = it.shared ? &a.sa0 : &a.a0;
                const CUtensorMap* ma1 = it.shared ? &a.sa1 : &a.a1;
                const CUtensorMap* mb = it.shared ? a.sb : a.b;
                const uint64_t pol_w = it.shared_a ? pol_wn : pol_w1;
                // the chunk's rows rounded up to 16, one box per set bit of the 16-row count
                const int nb = (it.nrows + 15) >> 4;
                const uint32_t bytes = NA * kABytes + nb * 2048;
                for (int kc = it.kc0; kc < it.kc1; ++kc) {
                    if (*abort_flag || !mbar_wait(smem_u32(&empty[stage]), phase ^ 1, limit)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * C::kStageBytes;
                    uint8_t* sb = sa + NA * kABytes;
                    const uint32_t fb = smem_u32(&full[stage]);
                    mbar_arrive_expect_tx(fb, bytes);
                    armed[stage] = phase;
                    constexpr int CK = Traits<MODE>::kChunkK;
                    int ka = kc * CK, kb = kc * CK, za = it.z, bmid = 0;
                    if (MODE == kDown && it.shared) {
                        za = kc / a.kc_per_sh;
                        ka = (kc - za * a.kc_per_sh) * 64;
                        kb = ka;
                        bmid = za;
                    }
                    tma_load_3d(smem_u32(sa), ma0, fb, ka, it.m0, za, pol_w);
                    if (Traits<MODE>::kGateUpLike)
                        tma_load_3d(smem_u32(sa + kABytes), ma1, fb, ka, it.m0, za, pol_w);
                    if (Traits<MODE>::kDownLike)
                        tma_load_3d(smem_u32(sa + kABytes), ma0, fb, ka, it.m0 + 128, za, pol_w);
                    for (int bit = 3, off = 0; bit >= 0; --bit) {
                        if (nb & (1 << bit)) {
                            tma_load_3d(smem_u32(sb + off * 2048), mb + bit, fb, kb, bmid, it.row0 + off * 16, pol_x);
                            off += 1 << bit;
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                raise_status(a.st, kStatusWaitTimeout);
            }
            // drain: every copy this thread issued has landed before the CTA exits
            for (int s = 0; s < STAGES; ++s)
                if (armed[s] != 2) mbar_wait(smem_u32(&full[s]), armed[s], limit);
        }
    } else if (warp == 1) {
        // =========================== MMA issuer =============================
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
                const Item it = decode_item<MODE, BN>(i, a, tb, n_sh_items);
                const int nb = (it.nrows + 15) >> 4;
                const uint32_t idesc =
                    Traits<MODE>::kF8 ? umma_idesc_e4m3(128, nb * 16) : umma_idesc_bf16(128, nb * 16);
                if (C::kRot) {
                    // one tile's four MMAs of the chunk in stage st (32 bytes of K each)
                    auto issue = [&](uint32_t d, int st, int tile, bool first) {
                        const uint32_t sa = smem_u32(smem + st * C::kStageBytes);
                        const uint64_t adesc = umma_desc_sw128(sa + tile * kABytes);
                        const uint64_t bdesc = umma_desc_sw128(sa + NA * kABytes);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t accum = (!first || kk > 0) ? 1u : 0u;
                            if (Traits<MODE>::kF8) umma_e4m3(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, accum);
                            else umma_bf16(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, accum);
                        }
                    };
                    // slots of the two tiles and the parities of their current use
                    const int s0 = acc, s1 = acc == 2 ? 0 : acc + 1;
                    const uint32_t p0 = acc_phase, p1 = acc == 2 ? acc_phase ^ 1 : acc_phase;
                    acc += 2;
                    if (acc >= 3) {
                        acc -= 3;
                        acc_phase ^= 1;
                    }
                    if (*abort_flag || !mbar_wait(smem_u32(&tempty[s0]), p0 ^ 1, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // The first tile runs ahead over the stages in flight; a stage is released
                    // once the second tile has consumed it too, so the second tile's MMAs follow
                    // as soon as its slot is drained.
                    const int nk = it.kc1 - it.kc0;
                    int st1 = stage;
                    int k0 = 0, k1 = 0;
                    bool t1 = false;
                    while (k1 < nk) {
                        if (!t1 && mbar_test_wait(smem_u32(&tempty[s1]), p1 ^ 1)) {
                            tc_fence_after();
                            t1 = true;
                        }
                        if (t1 && k1 < k0) {
                            issue(tbase + s1 * BN, st1, 1, k1 == 0);
                            umma_commit(smem_u32(&empty[st1]));
                            if (++st1 == STAGES) st1 = 0;
                            ++k1;
                        } else if (k0 < nk && k0 - k1 < STAGES) {
                            if (*abort_flag || !mbar_wait(smem_u32(&full[stage]), phase, limit)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue(tbase + s0 * BN, stage, 0, k0 == 0);
                            if (++stage == STAGES) {
                                stage = 0;
                                phase ^= 1;
                            }
                            if (++k0 == nk) umma_commit(smem_u32(&tfull[s0]));
                        } else {
                            if (*abort_flag || !mbar_wait(smem_u32(&tempty[s1]), p1 ^ 1, limit)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            t1 = true;
                        }
                    }
                    if (!ok) break;
                    umma_commit(smem_u32(&tfull[s1]));
                    continue;
                }
                if (*abort_flag || !mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tbase + acc * C::kAccCols;
                for (int kc = it.kc0; kc < it.kc1; ++kc) {
                    if (*abort_flag || !mbar_wait(smem_u32(&full[stage]), phase, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
                    const uint64_t adesc0 = umma_desc_sw128(sa);
                    const uint64_t adesc1 = umma_desc_sw128(sa + kABytes);
                    const uint64_t bdesc = umma_desc_sw128(sa + NA * kABytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t accum = (kc > it.kc0 || kk > 0) ? 1u : 0u;
                        // 32 bytes of K per instruction: 16 bf16 or 32 e4m3 elements
                        if (Traits<MODE>::kF8) {
                            umma_e4m3(d0, adesc0 + 2 * kk, bdesc + 2 * kk, idesc, accum);
                            umma_e4m3(d0 + BN, adesc1 + 2 * kk, bdesc + 2 * kk, idesc, accum);
                        } else {
                            umma_bf16(d0, adesc0 + 2 * kk, bdesc + 2 * kk, idesc, accum);
                            if (NA == 2) umma_bf16(d0 + BN, adesc1 + 2 * kk, bdesc + 2 * kk, idesc, accum);
                        }
                    }
                    umma_commit(smem_u32(&empty[stage]));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(smem_u32(&tfull[acc]));
                if (++acc == C::kNumAcc) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                raise_status(a.st, kStatusWaitTimeout);
            }
            // drain: all MMAs issued by this thread are complete before TMEM is freed
            umma_commit(smem_u32(mma_done));
            mbar_wait(smem_u32(mma_done), 0, limit);
        }
    } else {
        // =========================== epilogue ================================
        const int ew = warp - 2;
        const int q = warp & 3;           // TMEM lane quarter this warp may access
        const int part = ew >> 2;         // column groups part, part+4, ...
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t xph = 0;  // kDownF8Q: exchanges done by this warp
        bool ok = true;
        // Rotating slots (kRot): drain one half of a down item (one 128-row output
        // block) from the TMEM slot at tl.  Routed rows leave as bf16 y (E4M3 operands
        // dequantised first), shared rows as fp32 y_shared.
        auto plain_half = [&](const Item& it, int hh, uint32_t tl, int nb, int mlim) {
            const int row = it.m0 + hh * 128 + q * 32 + lane;
            const bool live = row < mlim;
            float sw = 0.0f;
            if (Traits<MODE>::kDownF8Like && live)
                sw = it.shared ? __ldg(a.sa0_scale + row) : __ldg(a.a0_scale + (size_t)it.z * a.m_routed + row);
#pragma unroll 1
            for (int g = part; g < nb; g += kEpiWarps / 4) {
                float v[16];
                tmem_ld16(tl + g * 16, v);
                tmem_ld_wait();
                if (!live) continue;
                if (Traits<MODE>::kDownF8Like) {
                    const float* sbp = (it.shared ? a.sb_scale : a.b_scale) + it.row0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int col = g * 16 + j;
                        v[j] *= sw * (col < it.nrows ? __ldg(sbp + col) : 0.0f);
                    }
                }
                if (it.shared) {
                    float* dst = reinterpret_cast<float*>(a.out_sh) + row;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int col = g * 16 + j;
                        if (col < it.nrows) dst[(size_t)(it.row0 + col) * a.out_sh_ld] = v[j];
                    }
                } else {
                    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.out) + row;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int col = g * 16 + j;
                        if (col < it.nrows) dst[(size_t)(it.row0 + col) * a.out_ld] = __float2bfloat16_rn(v[j]);
                    }
                }
            }
        };
        // Rotating slots, E4M3 combine payload: one half is one block of 128 output rows,
        // so its scales need only this half's maxima.  Pass 1: bf16 y, warp maxima of |y|
        // per column into shared memory; the four warps of these columns meet; pass 2:
        // the block scale of each column, codes, stores.
        // sxg[gi]: lane l's token scale of column group gi (column g*16 + l%16), sw: the
        // weight-row scale of this lane's row; both loaded before the accumulator wait.
        auto payload_half = [&](const Item& it, int hh, uint32_t tl, int nb, int mlim,
                                const float (&sxg)[C::kMaxG], float sw) -> bool {
            constexpr int kMaxG = C::kMaxG;
            const int blk = (it.m0 >> 7) + hh;
            float* xw = xchg + (size_t)(part * 4 + q) * kMaxG * 2 * 16;
            const float* xp = xchg + (size_t)part * 4 * kMaxG * 2 * 16;
            const uint32_t xfull = smem_u32(&xbar[part]), xfree = smem_u32(&xbar[4 + part]);
            // y of column group g: the fp32 value the plain E4M3 down rounds to bf16
            auto load_y = [&](int g, float sxl, float (&v)[16]) {
                tmem_ld16(tl + g * 16, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] *= sw * __shfl_sync(0xffffffffu, sxl, j);
            };
            // the four warps have read the previous exchange's maxima
            if (xph > 0 && !mbar_wait(xfree, (xph - 1) & 1, limit)) return false;
            // bf16 y of this warp's column groups, packed and kept for pass 2 where the
            // registers allow it (the 160-row rotating-slot kernel: 95 registers; the
            // 128-row kernel spilled and reloads the accumulator instead)
            constexpr bool kKeepY = C::kRot;
            uint32_t yb[kMaxG][8];
#pragma unroll
            for (int gi = 0; gi < kMaxG; ++gi) {
                const int g = part + gi * (kEpiWarps / 4);
                if (g < nb) {
                    float v[16];
                    load_y(g, sxg[gi], v);
                    // rounding is monotone: the bf16 of the largest |y| is the largest bf16 |y|
                    float mine = 0.0f;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const uint32_t mx = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v[j])));
                        if (lane == j) mine = __uint_as_float(mx);
                    }
                    if (lane < 16) xw[(gi * 2 + hh) * 16 + lane] = __bfloat162float(__float2bfloat16_rn(mine));
                    if constexpr (kKeepY) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const __nv_bfloat162 p2 = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
                            yb[gi][j] = *reinterpret_cast<const uint32_t*>(&p2);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(xfull);
            if (!mbar_wait(xfull, xph & 1, limit)) return false;
#pragma unroll
            for (int gi = 0; gi < kMaxG; ++gi) {
                const int g = part + gi * (kEpiWarps / 4);
                if (g >= nb) continue;
                // lane l < 16: scale of column l from the four warps' maxima
                const int o = (gi * 2 + hh) * 16 + (lane & 15);
                const float amax = fmaxf(fmaxf(xp[o], xp[kMaxG * 32 + o]),
                                         fmaxf(xp[2 * kMaxG * 32 + o], xp[3 * kMaxG * 32 + o]));
                const float sl = row_scale(amax);
                const int col_l = g * 16 + lane;
                if (q == 0 && lane < 16 && col_l < it.nrows)
                    a.out8_scale[(size_t)(it.row0 + col_l) * a.n_blk + blk] = sl;
                const RowDiv dl = row_div(sl);
                if constexpr (!kKeepY) {
                    float v[16];
                    load_y(g, sxg[gi], v);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const __nv_bfloat162 p2 = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
                        yb[gi][j] = *reinterpret_cast<const uint32_t*>(&p2);
                    }
                }
                // codes of the 16 columns, four to a word (byte c of word b: column 4b + c)
                uint32_t w[4];
                auto encode = [&](auto all_fast) {
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        float qv[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            RowDiv d;
                            d.s = __shfl_sync(0xffffffffu, dl.s, j + u);
                            d.r = __shfl_sync(0xffffffffu, dl.r, j + u);
                            const uint32_t yw = yb[gi][j >> 1];
                            const float yv = __uint_as_float(u ? (yw & 0xffff0000u) : (yw << 16));
                            if (decltype(all_fast)::value) qv[u] = div_rn<true>(d, yv);
                            else qv[u] = d.s >= 0x1p-96f ? div_rn<true>(d, yv) : div_rn<false>(d, yv);
                        }
                        const uint32_t c2 =
                            __nv_cvt_float2_to_fp8x2(make_float2(qv[0], qv[1]), __NV_SATFINITE, __NV_E4M3) & 0xffffu;
                        if (j & 2) w[j >> 2] |= c2 << 16;
                        else w[j >> 2] = c2;
                    }
                };
                // the reciprocal path for every column unless a scale of this group is
                // below 2^-96 (lanes 16-31 repeat columns 0-15)
                if (__all_sync(0xffffffffu, dl.fast)) encode(std::true_type{});
                else encode(std::false_type{});
                // 4x4 byte transpose inside each quad of lanes: lane 4m+c ends with column
                // 4b+c of rows 4m..4m+3, one aligned word (H % 8 == 0, codes 16-byte aligned)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const uint32_t o2 = __shfl_xor_sync(0xffffffffu, w[b], 2);
                    w[b] = __byte_perm(w[b], o2, (lane & 2) ? 0x3276 : 0x5410);
                    const uint32_t o1 = __shfl_xor_sync(0xffffffffu, w[b], 1);
                    w[b] = __byte_perm(w[b], o1, (lane & 1) ? 0x3715 : 0x6240);
                }
                const int row4 = it.m0 + hh * 128 + q * 32 + (lane & ~3);
                if (row4 < mlim) {
                    uint8_t* dst8 = a.out8 + row4;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const int col = g * 16 + 4 * b + (lane & 3);
                        if (col < it.nrows)
                            *reinterpret_cast<uint32_t*>(dst8 + (size_t)(it.row0 + col) * a.out_ld) = w[b];
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(xfree);  // this warp's reads of the maxima are done
            ++xph;
            return true;
        };
        // E4M3 payload: lane l's token scale of each of this warp's column groups
        // (column g*16 + l%16) and the weight-row scales of its rows in both halves
        auto payload_scales = [&](const Item& it, int mlim, float (&sxg)[C::kMaxG], float (&swh)[2]) {
#pragma unroll
            for (int gi = 0; gi < C::kMaxG; ++gi) {
                const int col = (part + gi * (kEpiWarps / 4)) * 16 + (lane & 15);
                sxg[gi] = col < it.nrows ? __ldg(a.b_scale + it.row0 + col) : 0.0f;
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = it.m0 + hh * 128 + q * 32 + lane;
                swh[hh] = row < mlim ? __ldg(a.a0_scale + (size_t)it.z * a.m_routed + row) : 0.0f;
            }
        };
        for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
            const Item it = decode_item<MODE, BN>(i, a, tb, n_sh_items);
            const int nb = (it.nrows + 15) >> 4;
            if (C::kRot) {
                // the two halves in turn, each from its own slot, each slot freed when drained
                const int sA = acc, sB = acc == 2 ? 0 : acc + 1;
                const uint32_t pA = acc_phase, pB = acc == 2 ? acc_phase ^ 1 : acc_phase;
                acc += 2;
                if (acc >= 3) {
                    acc -= 3;
                    acc_phase ^= 1;
                }
                const int mlim = it.shared ? a.m_shared : a.m_routed;
                // E4M3 payload: the token and weight-row scales, loaded while the MMAs run
                float sxg[C::kMaxG], swh[2];
                if (MODE == kDownF8Q && !it.shared) payload_scales(it, mlim, sxg, swh);
#pragma unroll 1
                for (int hh = 0; hh < 2 && ok; ++hh) {
                    const int sl = hh ? sB : sA;
                    if (*abort_flag || !mbar_wait(smem_u32(&tfull[sl]), hh ? pB : pA, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // a half past the last output row (H not a multiple of 256) holds no block
                    if (it.m0 + hh * 128 < mlim) {
                        const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16) + sl * BN;
                        if (MODE == kDownF8Q && !it.shared) ok = payload_half(it, hh, tl, nb, mlim, sxg, swh[hh]);
                        else plain_half(it, hh, tl, nb, mlim);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&tempty[sl]));
                }
                if (!ok) break;
                continue;
            }
            const int mlim = it.shared ? a.m_shared : a.m_routed;
            float sxg[C::kMaxG], swh[2];
            if (MODE == kDownF8Q && !it.shared) payload_scales(it, mlim, sxg, swh);
            if (MODE == kGateUpF8) {
                // token scales (one per lane and column group) and the gate and up row
                // scales of this lane's row, loaded while the MMAs run
                const float* sbp = (it.shared ? a.sb_scale : a.b_scale) + it.row0;
#pragma unroll
                for (int gi = 0; gi < C::kMaxG; ++gi) {
                    const int col = (part + gi * (kEpiWarps / 4)) * 16 + (lane & 15);
                    sxg[gi] = col < it.nrows ? __ldg(sbp + col) : 0.0f;
                }
                const int r = it.m0 + q * 32 + lane;
                const size_t zo = (size_t)it.z * (it.shared ? a.m_shared : a.m_routed);
                swh[0] = r < mlim ? __ldg((it.shared ? a.sa0_scale : a.a0_scale) + zo + r) : 0.0f;
                swh[1] = r < mlim ? __ldg((it.shared ? a.sa1_scale : a.a1_scale) + zo + r) : 0.0f;
            }
            if (*abort_flag || !mbar_wait(smem_u32(&tfull[acc]), acc_phase, limit)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int mrow = it.m0 + q * 32 + lane;
            const bool row_ok = mrow < mlim;
            (void)row_ok;
            const uint32_t tl = tbase + ((uint32_t)(q * 32) << 16) + acc * C::kAccCols;
            if (Traits<MODE>::kGateUpLike) {
                // SwiGLU per column group into packed bf16 registers, then free the
                // accumulator (the next item's MMAs may start) and store
                constexpr int kMaxG = C::kMaxG;
                uint32_t hp[kMaxG][8];
#pragma unroll
                for (int gi = 0; gi < kMaxG; ++gi) {
                    const int g = part + gi * (kEpiWarps / 4);
                    if (g < nb) {
                        float v0[16], v1[16];
                        tmem_ld16(tl + g * 16, v0);
                        tmem_ld16(tl + BN + g * 16, v1);
                        tmem_ld_wait();
                        if (MODE == kGateUpF8) {
                            // dequantise: weight-row scale x token scale (both factor out of the K sum)
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const float sx = __shfl_sync(0xffffffffu, sxg[gi], j);
                                v0[j] *= swh[0] * sx;
                                v1[j] *= swh[1] * sx;
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const __nv_bfloat162 p2 = __floats2bfloat162_rn(silu_f(v0[2 * j]) * v1[2 * j],
                                                                            silu_f(v0[2 * j + 1]) * v1[2 * j + 1]);
                            hp[gi][j] = *reinterpret_cast<const uint32_t*>(&p2);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
                {
                    // h as words of two rows: lanes 2m and 2m+1 swap half their columns, so
                    // the even lane holds the even columns of rows (2m, 2m+1) and the odd lane
                    // the odd ones (I % 8 == 0: both rows of a pair are valid together)
                    const bool odd = lane & 1;
                    const int row2 = mrow & ~1;
                    // the down projection reads h next: keep it in L2 ahead of the streamed weights
                    const uint64_t pol_h = policy_evict_last();
                    uint32_t* dst;
                    int ldw;
                    if (it.shared) {
                        dst = reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(a.out_sh) +
                                                          (size_t)it.z * a.sh_col_stride + row2);
                        ldw = a.out_sh_ld >> 1;
                    } else {
                        dst = reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(a.out) + row2);
                        ldw = a.out_ld >> 1;
                    }
#pragma unroll
                    for (int gi = 0; gi < kMaxG; ++gi) {
                        const int g = part + gi * (kEpiWarps / 4);
                        if (g < nb) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const uint32_t o = __shfl_xor_sync(0xffffffffu, hp[gi][i], 1);
                                const uint32_t w = __byte_perm(hp[gi][i], o, odd ? 0x3276 : 0x5410);
                                const int col = g * 16 + 2 * i + (odd ? 1 : 0);
                                if (row_ok && col < it.nrows) st_hint(dst + (size_t)(it.row0 + col) * ldw, w, pol_h);
                            }
                        }
                    }
                }
                if (++acc == C::kNumAcc) {
                    acc = 0;
                    acc_phase ^= 1;
                }
                continue;
            }
            if (MODE == kDownF8Q && !it.shared) {
                // E4M3 payload, both halves from this accumulator, which is freed after both
#pragma unroll 1
                for (int hh = 0; hh < 2 && ok; ++hh)
                    if (it.m0 + hh * 128 < mlim) ok = payload_half(it, hh, tl + hh * BN, nb, mlim, sxg, swh[hh]);
                if (!ok) break;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
                if (++acc == C::kNumAcc) {
                    acc = 0;
                    acc_phase ^= 1;
                }
                continue;
            }
            for (int g = part; g < nb; g += kEpiWarps / 4) {
                float v0[16], v1[16];
                tmem_ld16(tl + g * 16, v0);
                if (NA == 2) tmem_ld16(tl + BN + g * 16, v1);
                tmem_ld_wait();
                // FP8 down: the token-row scales of this column group
                float sxv[16];
                if (Traits<MODE>::kDownF8Like) {
                    const float* sbp = (it.shared ? a.sb_scale : a.b_scale) + it.row0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int col = g * 16 + j;
                        sxv[j] = col < it.nrows ? __ldg(sbp + col) : 0.0f;
                    }
                }
                // NA consecutive 128-row output blocks (down: rows m0.. and m0+128..)
#pragma unroll
                for (int hh = 0; hh < NA; ++hh) {
                    const int row = mrow + hh * 128;
                    if (MODE == kDown && !it.shared) {
                        // bf16 y as words of two rows: lanes 2m and 2m+1 swap half their
                        // columns, so the even lane holds the even columns of rows (row,
                        // row+1) and the odd lane the odd ones (H % 8 == 0: both rows of a
                        // pair are valid together, and every word is 4-byte aligned)
                        const bool odd = lane & 1;
                        uint32_t* dst = reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(a.out) + (row & ~1));
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float* vv = hh ? v1 : v0;
                            const __nv_bfloat162 p2 = __floats2bfloat162_rn(vv[2 * i], vv[2 * i + 1]);
                            const uint32_t p = *reinterpret_cast<const uint32_t*>(&p2);
                            const uint32_t o = __shfl_xor_sync(0xffffffffu, p, 1);
                            const uint32_t w = __byte_perm(p, o, odd ? 0x3276 : 0x5410);
                            const int col = g * 16 + 2 * i + (odd ? 1 : 0);
                            if (row < mlim && col < it.nrows) dst[(size_t)(it.row0 + col) * (a.out_ld >> 1)] = w;
                        }
                        continue;
                    }
                    if (row >= mlim) continue;
                    if (Traits<MODE>::kDownF8Like) {
                        // dequantise: weight-row scale x intermediate-row scale
                        const float sw = it.shared ? __ldg(a.sa0_scale + row)
                                                   : __ldg(a.a0_scale + (size_t)it.z * a.m_routed + row);
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            if (hh) v1[j] *= sw * sxv[j];
                            else v0[j] *= sw * sxv[j];
                        }
                    }
                    if (MODE == kRouter) {
                        float* dst = reinterpret_cast<float*>(a.out) + (size_t)it.ks * a.T * a.out_ld + row;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int col = g * 16 + j;
                            if (col < it.nrows) dst[(size_t)(it.row0 + col) * a.out_ld] = hh ? v1[j] : v0[j];
                        }
                    } else if (it.shared) {
                        float* dst = reinterpret_cast<float*>(a.out_sh) + row;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int col = g * 16 + j;
                            if (col < it.nrows) dst[(size_t)(it.row0 + col) * a.out_sh_ld] = hh ? v1[j] : v0[j];
                        }
                    } else {
                        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.out) + row;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int col = g * 16 + j;
                            if (col < it.nrows)
                                dst[(size_t)(it.row0 + col) * a.out_ld] = __float2bfloat16_rn(hh ? v1[j] : v0[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
            if (++acc == C::kNumAcc) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            raise_status(a.st, kStatusWaitTimeout);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, C::kTmemCols);
}

template <int MODE, int BN, int STAGES>
cudaError_t launch_one(const GemmArgs& args, int grid, cudaStream_t stream) {
    using C = Config<MODE, BN, STAGES>;
    auto kern = grouped_gemm_kernel<MODE, BN, STAGES>;
    static std::atomic<uint64_t> configured{0};
    const cudaError_t e = configure_once(configured, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    });
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), C::kSmemBytes, stream, args);
}

}  // namespace

int gemm_max_slots() { return kMaxSlots; }

cudaError_t launch_gemm(GemmMode mode, int bn, const GemmArgs& args, int grid, cudaStream_t stream) {
    if (grid <= 0) return cudaSuccess;
    if (bn == 32) {
        switch (mode) {
            case kGateUpF8: return launch_one<kGateUpF8, 32, 5>(args, grid, stream);
            case kGateUp: return launch_one<kGateUp, 32, 5>(args, grid, stream);
            case kDown: return launch_one<kDown, 32, 5>(args, grid, stream);
            case kDownF8: return launch_one<kDownF8, 32, 5>(args, grid, stream);
            case kDownF8Q: return launch_one<kDownF8Q, 32, 5>(args, grid, stream);
            case kRouter: return launch_one<kRouter, 32, 8>(args, grid, stream);
        }
    } else if (bn == kMidBN) {
        if (mode == kDownF8) return launch_one<kDownF8, kMidBN, 4>(args, grid, stream);
        if (mode == kDownF8Q) return launch_one<kDownF8Q, kMidBN, 4>(args, grid, stream);
    } else if (bn == kPrefillBN) {
        switch (mode) {
            case kGateUpF8: return launch_one<kGateUpF8, kPrefillBN, 4>(args, grid, stream);
            case kGateUp: return launch_one<kGateUp, kPrefillBN, 4>(args, grid, stream);
            case kDown: return launch_one<kDown, kPrefillBN, 4>(args, grid, stream);
            case kDownF8: return launch_one<kDownF8, kPrefillBN, 4>(args, grid, stream);
            case kDownF8Q: return launch_one<kDownF8Q, kPrefillBN, 4>(args, grid, stream);
            case kRouter: return launch_one<kRouter, kPrefillBN, 5>(args, grid, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe
