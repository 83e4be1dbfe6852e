// Router tail: sum of the router GEMM's K-split partial logits (fixed order),
// bias, softmax over all experts and top-k selection, one warp per token.
//
// Blog post "专家并行(EP)", section 2.2: step 1 picks the top-8 of the 256
// router logits; step 5 weights each selected expert's output by
// softmax(logits)[i].  The softmax runs over all E logits and the selected
// probabilities are not renormalised.  Selection is by value, ties broken by
// the lower expert index: by warp-shuffle arg-max rounds, or, for a decode
// batch of at most 256 experts, by each thread ranking its expert against all.
#include "kernels.h"

namespace moe {
namespace {

// a ranks before b: larger value, or equal value and lower index.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

// tpc (1..8) tokens per CTA, grid-stride: all threads sum the K-split partials
// of the CTA's tokens (coalesced over experts, eight loads in flight) into
// shared memory, then warp w runs the softmax and the k arg-max rounds of
// token w.  Up to a few hundred tokens use one token per CTA; up to 64 tokens
// (decode) the CTA has groups = 4 x 256 threads and each logit's partials are
// summed by 4 threads (group g takes splits g, g + 4, ... in order) whose sums
// are added in group order, so the result does not depend on scheduling.
constexpr int kTokPerCta = 8;
// up to 64 tokens (one token per 1024-thread CTA) and at most this many
// experts: selection by ranks (measured ~1 us faster than the warp's k
// arg-max rounds there; slower at 256 tokens, where 256-thread CTAs keep the
// warp rounds)
constexpr int kRankMaxExperts = 256;
constexpr int kMaxGroups = 4;

// sum of p[ks * slice] for ks = first, first + stride, ... < ksplit, in that
// order; eight loads in flight, the last block predicated
__device__ __forceinline__ float sum_partials(const float* p, int first, int stride, int ksplit, size_t slice) {
    float s = 0.0f;
    for (int ks = first; ks < ksplit; ks += 8 * stride) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = ks + u * stride < ksplit ? __ldg(p + (size_t)(ks + u * stride) * slice) : 0.0f;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (ks + u * stride < ksplit) s += v[u];
    }
    return s;
}

template <int EPL>  // logits per lane; expert e = i*32 + lane
__global__ void __launch_bounds__(1024) topk_kernel(const float* __restrict__ partials, int ksplit,
                                                   const float* __restrict__ bias, int T, int E, int k,
                                                   float* __restrict__ logits_out,
                                                   int32_t* __restrict__ topk_idx,
                                                   float* __restrict__ topk_w, int tpc, int groups,
                                                   int n_groups, int topk_groups) {
    pdl_begin();
    __shared__ __align__(16) float lg[kTokPerCta][EPL * 32];
    __shared__ float red[32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const size_t slice = (size_t)T * E;
    for (int t0 = blockIdx.x * tpc; t0 < T; t0 += gridDim.x * tpc) {
        const int nt = min(tpc, T - t0);
        if (tpc == 1) {
            // one token: group g of the CTA sums splits g, g + groups, ... into lg[g]
            for (int q = threadIdx.x; q < groups * E; q += blockDim.x) {
                const int g = q / E, e = q - g * E;
                lg[g][e] = sum_partials(partials + (size_t)t0 * E + e, g, groups, ksplit, slice);
            }
            __syncthreads();
            for (int e = threadIdx.x; e < E; e += blockDim.x) {
                float s = lg[0][e];
                for (int g = 1; g < groups && g < ksplit; ++g) s += lg[g][e];
                if (bias) s += bias[e];
                lg[0][e] = s;
                if (logits_out) logits_out[(size_t)t0 * E + e] = s;
            }
        } else {
            for (int q = threadIdx.x; q < nt * E; q += blockDim.x) {
                const int tt = q / E, e = q - tt * E;
                float s = sum_partials(partials + (size_t)(t0 + tt) * E + e, 0, 1, ksplit, slice);
                if (bias) s += bias[e];
                lg[tt][e] = s;
                if (logits_out) logits_out[(size_t)(t0 + tt) * E + e] = s;
            }
        }
        __syncthreads();
        if (groups > 1 && topk_groups >= n_groups && E <= kRankMaxExperts && E <= (int)blockDim.x) {
            // one token, plain top-k: thread e ranks expert e against all E
            // (larger logit first, equal logits by lower index); ranks below
            // k are the selection in order.  Softmax statistics by block
            // reductions in a fixed order.
            const int e = threadIdx.x;
            const int nw = (E + 31) / 32;  // warps that hold experts
            const float v = e < E ? lg[0][e] : -INFINITY;
            float m_ = v;
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) m_ = fmaxf(m_, __shfl_xor_sync(0xffffffffu, m_, d));
            if (lane == 0 && warp < nw) red[warp] = m_;
            __syncthreads();
            float mx = red[0];
            for (int w = 1; w < nw; ++w) mx = fmaxf(mx, red[w]);
            const float ex = e < E ? expf(v - mx) : 0.0f;
            float sum = ex;
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
            __syncthreads();  // every thread has read the maxima
            if (lane == 0 && warp < nw) red[warp] = sum;
            __syncthreads();
            float den = 0.0f;
            for (int w = 0; w < nw; ++w) den += red[w];
            if (e < E) {
                // four logits per (broadcast) shared-memory read, several reads in flight
                const float4* row4 = reinterpret_cast<const float4*>(lg[0]);
                int rank = 0, j = 0;
#pragma unroll 4
                for (; j + 4 <= E; j += 4) {
                    const float4 u = row4[j >> 2];
                    rank += (u.x > v || (u.x == v && j < e)) ? 1 : 0;
                    rank += (u.y > v || (u.y == v && j + 1 < e)) ? 1 : 0;
                    rank += (u.z > v || (u.z == v && j + 2 < e)) ? 1 : 0;
                    rank += (u.w > v || (u.w == v && j + 3 < e)) ? 1 : 0;
                }
                for (; j < E; ++j) {
                    const float u = lg[0][j];
                    rank += (u > v || (u == v && j < e)) ? 1 : 0;
                }
                if (rank < k) {
                    topk_idx[(size_t)t0 * k + rank] = e;
                    topk_w[(size_t)t0 * k + rank] = ex * (1.0f / den);
                }
            }
            __syncthreads();  // lg and red are rewritten for the next token
            continue;
        }
        if (warp < nt) {
            const int t = t0 + warp;
            float v[EPL];
            uint32_t valid = 0;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = i * 32 + lane;
                v[i] = 0.0f;
                if (e < E) {
                    v[i] = lg[warp][e];
                    valid |= 1u << i;
                }
            }
            // softmax statistics over all E (fixed reduction order)
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (valid & (1u << i)) mx = fmaxf(mx, v[i]);
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
            float den = 0.0f;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (valid & (1u << i)) den += expf(v[i] - mx);
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) den += __shfl_xor_sync(0xffffffffu, den, d);
            const float inv_den = 1.0f / den;

            uint32_t avail = valid;
            if (topk_groups < n_groups) {
                // group-limited routing: keep the topk_groups groups with the best
                // maximum logit (ties -> lower group), then select experts in them
                const int gs = E / n_groups;
                float gv = -INFINITY;
                int gi = 0x7fffffff;
                if (lane < n_groups) {
                    gv = lg[warp][lane * gs];
                    for (int e = lane * gs + 1; e < (lane + 1) * gs; ++e) gv = fmaxf(gv, lg[warp][e]);
                    gi = lane;
                }
                uint32_t kept = 0;
                for (int r = 0; r < topk_groups; ++r) {
                    float bv = (kept >> lane) & 1u ? -INFINITY : gv;
                    int bi = (kept >> lane) & 1u ? 0x7fffffff : gi;
#pragma unroll
                    for (int d = 16; d > 0; d >>= 1) {
                        const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
                        const int oi = __shfl_xor_sync(0xffffffffu, bi, d);
                        if (oi != 0x7fffffff && (bi == 0x7fffffff || better(ov, oi, bv, bi))) {
                            bv = ov;
                            bi = oi;
                        }
                    }
                    kept |= 1u << bi;
                }
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const int e = i * 32 + lane;
                    if (e < E && !((kept >> (e / gs)) & 1u)) avail &= ~(1u << i);
                }
            }
            for (int j = 0; j < k; ++j) {
                float bv = -INFINITY;
                int bi = 0x7fffffff;
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    if (avail & (1u << i)) {
                        const int e = i * 32 + lane;
                        if (bi == 0x7fffffff || better(v[i], e, bv, bi)) {
                            bv = v[i];
                            bi = e;
                        }
                    }
                }
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, d);
                    if (oi != 0x7fffffff && (bi == 0x7fffffff || better(ov, oi, bv, bi))) {
                        bv = ov;
                        bi = oi;
                    }
                }
                if (bi != 0x7fffffff && (bi & 31) == lane) avail &= ~(1u << (bi >> 5));
                if (lane == 0) {
                    topk_idx[(size_t)t * k + j] = bi;
                    topk_w[(size_t)t * k + j] = expf(bv - mx) * inv_den;
                }
            }
        }
        __syncthreads();
    }
}

template <int EPL>
cudaError_t launch_epl(const float* partials, int ksplit, const float* bias, int T, int E, int k,
                       float* logits_out, int32_t* topk_idx, float* topk_w, int n_groups, int topk_groups,
                       cudaStream_t stream) {
    const int tpc = T <= 4 * num_sms() ? 1 : kTokPerCta;
    const int groups = T <= 64 ? kMaxGroups : 1;
    const int threads = 256 * groups;
    int blocks = (T + tpc - 1) / tpc;
    const int cap = num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(topk_kernel<EPL>, dim3(blocks), dim3(threads), 0, stream, partials, ksplit, bias, T, E, k,
                      logits_out, topk_idx, topk_w, tpc, groups, n_groups, topk_groups);
}

}  // namespace

cudaError_t launch_topk(const float* partials, int ksplit, const float* bias, int T, int E, int k,
                        float* logits_out, int32_t* topk_idx, float* topk_w, int n_groups, int topk_groups,
                        const DevStatus& st, cudaStream_t stream) {
    (void)st;
    if (n_groups <= 0) n_groups = topk_groups = 1;
    const int epl = (E + 31) / 32;
    if (epl <= 1) return launch_epl<1>(partials, ksplit, bias, T, E, k, logits_out, topk_idx, topk_w, n_groups, topk_groups, stream);
    if (epl <= 2) return launch_epl<2>(partials, ksplit, bias, T, E, k, logits_out, topk_idx, topk_w, n_groups, topk_groups, stream);
    if (epl <= 4) return launch_epl<4>(partials, ksplit, bias, T, E, k, logits_out, topk_idx, topk_w, n_groups, topk_groups, stream);
    if (epl <= 8) return launch_epl<8>(partials, ksplit, bias, T, E, k, logits_out, topk_idx, topk_w, n_groups, topk_groups, stream);
    if (epl <= 16) return launch_epl<16>(partials, ksplit, bias, T, E, k, logits_out, topk_idx, topk_w, n_groups, topk_groups, stream);
    if (epl <= 32) return launch_epl<32>(partials, ksplit, bias, T, E, k, logits_out, topk_idx, topk_w, n_groups, topk_groups, stream);
    return cudaErrorInvalidValue;
}

}  // namespace moe
