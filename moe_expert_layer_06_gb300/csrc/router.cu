// Router in one launch: GEMM + bias + softmax + top-k.
//
// Blog post "专家并行(EP)", section 2.2 step 1: logits = x W_r^T over the
// router linear [hidden, E], top-k of the E logits; step 5 weights each
// selected expert by softmax(logits)[i] over all E (not renormalised); ties
// go to the lower expert index.
//
// One thread-block cluster of C CTAs (16 for chunks of 32 tokens, 8 for 128)
// takes a chunk of BN tokens; CTA r of the cluster takes the r-th slice of the
// K (hidden) dimension and every expert (two 128-row tiles of W_r):
//   1. TMA streams W_r and x slices, tcgen05.mma accumulates the partial
//      logits [256 x BN] in TMEM (warp 0 producer, warp 1 issuer);
//   2. warps 2-5 move the partial to shared memory, token-major;
//   3. cluster barrier; CTA r sums experts [r*256/C, (r+1)*256/C) over the C
//      partials through distributed shared memory, in rank order, and adds
//      the bias;
//   4. cluster barrier; each warp of CTA r takes one of the chunk's tokens
//      r, r + C, ...: gathers its E logits from the C CTAs (8 a lane), softmax
//      statistics by warp reductions in a fixed order, then k arg-max rounds
//      (larger logit first, equal logits by lower expert index);
//   5. cluster barrier before any CTA's shared memory goes away.
// Every mbarrier wait is bounded; on expiry a CTA raises the status word and
// skips its remaining work but still meets every cluster barrier.
#include "kernels.h"

namespace moe {
namespace {

constexpr int kRThreads = 256;   // 8 warps
constexpr int kRStages = 4;
constexpr int kRExperts = 256;   // two 128-row tiles
constexpr int kRTileBytes = 128 * 64 * 2;

template <int BN>
struct RCfg {
    static constexpr int kBBytes = BN * 128;
    static constexpr int kStageBytes = 2 * kRTileBytes + kBBytes;
    static constexpr int kRingBytes = kRStages * kStageBytes;
    static constexpr int kPartBytes = BN * kRExperts * 4;        // token-major partial, reuses the ring
    static constexpr int kLocBytes = BN * 32 * 4;                // reduced logits of this CTA's experts (<= 32)
    static constexpr int kSmemBytes = 1024 + kRingBytes + kLocBytes + (2 * kRStages + 2) * 8 + 16;
    static_assert(kPartBytes <= kRingBytes, "partial must fit the ring");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory overflow");
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

struct RouterArgs {
    CUtensorMap w;       // W_r [E, H] as {H, E, 1}, box {64, 128, 1}
    CUtensorMap x;       // x [T, H] as {H, 1, T}, box {64, 1, BN}
    const float* bias;   // [E] or null
    int T, E, H, k;
    float* logits_out;   // [T, E] or null
    int32_t* topk_idx;   // [T, k]
    float* topk_w;       // [T, k]
    DevStatus st;
};

template <int BN>
__global__ void __launch_bounds__(kRThreads, 1) router_topk_kernel(const __grid_constant__ RouterArgs a) {
    pdl_launch_dependents();
    using C = RCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* part = reinterpret_cast<float*>(smem);                       // [BN][256], after the MMAs
    float* loc = reinterpret_cast<float*>(smem + C::kRingBytes);        // [BN][epc]
    uint64_t* bars = reinterpret_cast<uint64_t*>(loc + BN * 32);
    uint64_t* full = bars;
    uint64_t* empty = bars + kRStages;
    uint64_t* tfull = bars + 2 * kRStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kRStages + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank(), ncta = cluster_size();
    const int chunk = blockIdx.x / ncta;
    const int t0 = chunk * BN;
    const int nk = (a.H + 63) / 64;
    const int kc0 = (int)((long)rank * nk / ncta), kc1 = (int)((long)(rank + 1) * nk / ncta);
    const int epc = kRExperts / (int)ncta;  // experts reduced by this CTA (16 or 32)
    const unsigned long long limit = a.st.limit_ns;
    constexpr uint32_t kCols = (2 * BN < 32) ? 32 : 2 * BN;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kRStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(tfull), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&a.w);
        tma_prefetch_desc(&a.x);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    pdl_wait();

    // ---- 1. partial logits of this CTA's K slice
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_normal();  // every token chunk's cluster reads W_r
            const uint64_t pol_x = policy_evict_first();
            uint32_t armed[kRStages];
            for (int s = 0; s < kRStages; ++s) armed[s] = 2;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int kc = kc0; kc < kc1; ++kc) {
                if (*abort_flag || !mbar_wait(smem_u32(&empty[stage]), phase ^ 1, limit)) {
                    ok = false;
                    break;
                }
                uint8_t* sa = smem + stage * C::kStageBytes;
                const uint32_t fb = smem_u32(&full[stage]);
                mbar_arrive_expect_tx(fb, C::kStageBytes);
                armed[stage] = phase;
                tma_load_3d(smem_u32(sa), &a.w, fb, kc * 64, 0, 0, pol_w);
                tma_load_3d(smem_u32(sa + kRTileBytes), &a.w, fb, kc * 64, 128, 0, pol_w);
                tma_load_3d(smem_u32(sa + 2 * kRTileBytes), &a.x, fb, kc * 64, 0, t0, pol_x);
                if (++stage == kRStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                raise_status(a.st, kStatusWaitTimeout);
            }
            for (int s = 0; s < kRStages; ++s)
                if (armed[s] != 2) mbar_wait(smem_u32(&full[s]), armed[s], limit);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16(128, BN);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int kc = kc0; kc < kc1; ++kc) {
                if (*abort_flag || !mbar_wait(smem_u32(&full[stage]), phase, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
                const uint64_t a0 = umma_desc_sw128(sa), a1 = umma_desc_sw128(sa + kRTileBytes);
                const uint64_t b = umma_desc_sw128(sa + 2 * kRTileBytes);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acc = (kc > kc0 || kk > 0) ? 1u : 0u;
                    umma_bf16(tbase, a0 + 2 * kk, b + 2 * kk, idesc, acc);
                    umma_bf16(tbase + BN, a1 + 2 * kk, b + 2 * kk, idesc, acc);
                }
                umma_commit(smem_u32(&empty[stage]));
                if (++stage == kRStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                raise_status(a.st, kStatusWaitTimeout);
            }
            if (kc1 > kc0) umma_commit(smem_u32(tfull));  // arrives once every MMA issued above is done
            else mbar_arrive(smem_u32(tfull));            // no K chunk here: nothing to wait for
        }
    }
    // ---- 2. partial to shared memory, token-major (a CTA with no K chunk writes zeros)
    if (warp >= 2 && warp < 6) {
        const int q = warp & 3;
        const bool have = kc1 > kc0;
        if (!mbar_wait(smem_u32(tfull), 0, limit)) {
            *abort_flag = 1;
            if (lane == 0) raise_status(a.st, kStatusWaitTimeout);
        }
        tc_fence_after();
#pragma unroll
        for (int tile = 0; tile < 2; ++tile) {
            const int e = tile * 128 + q * 32 + lane;
#pragma unroll
            for (int g = 0; g < BN / 16; ++g) {
                float v[16];
                if (have && !*abort_flag) {
                    tmem_ld16(tbase + ((uint32_t)(q * 32) << 16) + tile * BN + g * 16, v);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0.0f;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) part[(g * 16 + j) * kRExperts + e] = v[j];
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    cluster_sync();  // every CTA's partial is in its shared memory

    // ---- 3. reduce this CTA's experts over the cluster, in rank order, plus the bias
    {
        const int e0 = (int)rank * epc;
        for (int o = threadIdx.x; o < BN * epc; o += kRThreads) {
            const int t = o / epc, el = o - t * epc, e = e0 + el;
            const uint32_t off = smem_u32(part + t * kRExperts + e);
            float v[16];  // every peer's partial first (the loads overlap), then the sum in rank order
#pragma unroll
            for (int r = 0; r < 16; ++r) v[r] = r < (int)ncta ? ld_cluster(peer_addr(off, (uint32_t)r)) : 0.0f;
            float s = 0.0f;
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (r < (int)ncta) s += v[r];
            if (a.bias && e < a.E) s += __ldg(a.bias + e);
            loc[t * epc + el] = s;
        }
    }
    __syncthreads();
    cluster_sync();  // every CTA's reduced logits are ready

    // ---- 4. softmax and top-k, one warp per token: tokens rank, rank + C, ... of the chunk
    const int E = a.E;
    for (int tt = (int)rank + warp * (int)ncta; tt < BN; tt += 8 * (int)ncta) {
        const int t = t0 + tt;
        if (t >= a.T) break;
        float v[8];
        uint32_t valid = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = i * 32 + lane;
            v[i] = 0.0f;
            if (e < E) {
                v[i] = ld_cluster(peer_addr(smem_u32(loc + tt * epc + (e % epc)), (uint32_t)(e / epc)));
                valid |= 1u << i;
            }
        }
        if (a.logits_out) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (valid & (1u << i)) a.logits_out[(size_t)t * E + i * 32 + lane] = v[i];
        }
        // softmax statistics over all E (fixed reduction order)
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (valid & (1u << i)) mx = fmaxf(mx, v[i]);
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
        float den = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (valid & (1u << i)) den += expf(v[i] - mx);
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) den += __shfl_xor_sync(0xffffffffu, den, d);
        const float inv_den = 1.0f / den;
        // k arg-max rounds: larger logit first, equal logits by lower expert index
        uint32_t avail = valid;
        for (int j = 0; j < a.k; ++j) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = i * 32 + lane;
                if ((avail & (1u << i)) && (bi == 0x7fffffff || v[i] > bv || (v[i] == bv && e < bi))) {
                    bv = v[i];
                    bi = e;
                }
            }
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, d);
                if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (bi != 0x7fffffff && (bi & 31) == lane) avail &= ~(1u << (bi >> 5));
            if (lane == 0) {
                a.topk_idx[(size_t)t * a.k + j] = bi;
                a.topk_w[(size_t)t * a.k + j] = expf(bv - mx) * inv_den;
            }
        }
    }
    cluster_sync();  // no CTA leaves while a peer may still read its shared memory
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, kCols);
}

template <int BN>
cudaError_t launch_router_bn(const RouterArgs& args, int cluster, cudaStream_t stream) {
    using C = RCfg<BN>;
    auto kern = router_topk_kernel<BN>;
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = configure_once(configured, [&] {
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (r == cudaSuccess) r = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        return r;
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(((args.T + BN - 1) / BN) * cluster));
    cfg.blockDim = dim3(kRThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

// The cluster size per token chunk width on the calling thread's device: for 32
// tokens 16 CTAs (else 8), for 128 tokens 8 (else 16), whichever first has at
// least one resident cluster; 0 if none (the two-launch router is used then).
// Measured on one GB300: 16-CTA clusters for 128-token chunks cost the
// 4096-token prefill 70 us (fewer clusters fit a GPC at once); with these
// choices every bench workload times as with the two-launch router.
template <int BN>
int cluster_for(int dev) {
    static std::atomic<int> cached[64];
    if (dev < 0 || dev >= 64) return 0;
    int v = cached[dev].load(std::memory_order_acquire);
    if (v != 0) return v > 0 ? v : 0;
    using C = RCfg<BN>;
    auto kern = router_topk_kernel<BN>;
    int best = -1;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) == cudaSuccess &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        for (int c : (BN == 32 ? std::initializer_list<int>{16, 8} : std::initializer_list<int>{8, 16})) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)c);
            cfg.blockDim = dim3(kRThreads);
            cfg.dynamicSmemBytes = C::kSmemBytes;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = c;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= 1) {
                best = c;
                break;
            }
        }
    }
    cudaGetLastError();  // a refused attribute or query leaves no error behind
    cached[dev].store(best, std::memory_order_release);
    return best > 0 ? best : 0;
}

}  // namespace

int router_fused_supported(int n_experts, int top_k) { return n_experts <= kRExperts && top_k <= 32 ? 1 : 0; }

int router_fused_bn(int T) { return T <= 32 ? 32 : 128; }

cudaError_t launch_router_fused(const CUtensorMap& w, const CUtensorMap& x, const float* bias, int T, int E, int H,
                                int k, float* logits_out, int32_t* topk_idx, float* topk_w, const DevStatus& st,
                                cudaStream_t stream, bool* launched) {
    *launched = false;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int bn = router_fused_bn(T);
    const int cl = bn == 32 ? cluster_for<32>(dev) : cluster_for<128>(dev);
    if (cl == 0) return cudaSuccess;
    RouterArgs a;
    a.w = w;
    a.x = x;
    a.bias = bias;
    a.T = T;
    a.E = E;
    a.H = H;
    a.k = k;
    a.logits_out = logits_out;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.st = st;
    *launched = true;
    return bn == 32 ? launch_router_bn<32>(a, cl, stream) : launch_router_bn<128>(a, cl, stream);
}

}  // namespace moe
