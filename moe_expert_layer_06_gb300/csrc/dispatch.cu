// Dispatch of the MoE layer on one device: replica remap, per-slot histogram,
// per-block loads, exclusive offsets, a stable counting-sort permutation, and
// the row scatter into the per-slot contiguous dispatch buffer.
//
// Blog post "专家并行(EP)": section 2.2 step 2 sends each token's hidden
// state to the owner of each expert it selected (here: a permutation into one
// buffer whose slot segments sit in block order, the per-rank send segments
// of section 2.1's contiguous layout); section 6.2 monitors per-expert
// arrivals and per-rank load sums; section 6.3 lets a token use any replica
// of its expert (here: odd tokens use the replica).
#include "kernels.h"

namespace moe {
namespace {

constexpr int kIdxThreads = 1024;
constexpr int kMaxSlots = 1024;
// chunked index pass: from this many assignments, chunks of kIndexChunk
// (more per chunk beyond kMaxIndexChunks chunks)
constexpr int kChunkedIndexMin = 4096;
constexpr int kIndexChunk = 512;
constexpr int kMaxIndexChunks = 128;

__device__ __forceinline__ int home_slot(int e, int E, int S, int n_blocks) {
    const int epb = E / n_blocks, spb = S / n_blocks;
    return (e / epb) * spb + (e % epb);
}

// Slot of assignment x = t*k + j: the replica for odd tokens of a replicated
// expert, else the expert's home slot; S (the invalid bucket) for a bad id.
__device__ __forceinline__ int slot_of_assignment(const DispatchArgs& a, int x, bool& bad) {
    const int t = x / a.k;
    const int e = a.topk_idx[x];
    if (e < 0 || e >= a.E) {
        bad = true;
        return a.S;
    }
    int slot = home_slot(e, a.E, a.S, a.n_blocks);
    if (a.replica_of && (t & 1)) {
        const int r = a.replica_of[e];
        if (r >= 0) {
            if (r < a.S) slot = r;
            else { slot = a.S; bad = true; }
        }
    }
    return slot;
}

// Pass 1 of a warp over its contiguous assignment range [r0, r1): slot of
// each assignment (stored to slot_of when given) and this warp's count per
// slot in mine[] (match_any groups equal slots within a step).
__device__ __forceinline__ void warp_count_range(const DispatchArgs& a, int r0, int r1, int* mine, bool& bad) {
    const int lane = threadIdx.x & 31;
    for (int x0 = r0; x0 < r1; x0 += 32) {
        const int x = x0 + lane;
        const bool valid = x < r1;
        int slot = -1;
        if (valid) {
            slot = slot_of_assignment(a, x, bad);
            if (a.slot_of) a.slot_of[x] = slot;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, slot);
        if (valid && (__ffs(peers) - 1) == lane) mine[slot] += __popc(peers);
        __syncwarp();
    }
}

// Pass 2 over the same range in order: mine[slot] holds the next row of this
// warp in each slot; rows are handed out in assignment order.
__device__ __forceinline__ void warp_rank_range(const DispatchArgs& a, int r0, int r1, int* mine) {
    const int lane = threadIdx.x & 31;
    const unsigned lt_mask = (1u << lane) - 1u;
    bool unused = false;
    for (int x0 = r0; x0 < r1; x0 += 32) {
        const int x = x0 + lane;
        const bool valid = x < r1;
        const int slot = valid ? slot_of_assignment(a, x, unused) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, slot);
        if (valid) {
            const int row = mine[slot] + __popc(peers & lt_mask);
            a.perm[row] = x;
            a.inv_perm[x] = row;
        }
        __syncwarp();
        if (valid && (__ffs(peers) - 1) == lane) mine[slot] += __popc(peers);
        __syncwarp();
    }
}

// From the per-slot totals cnt[NS]: counts, block loads and (when offsets is
// given) the exclusive prefix base[0..NS] over slots and the invalid bucket,
// written to offsets.  Called by every thread of the CTA.
__device__ __forceinline__ void finish_counts(const DispatchArgs& a, const int* cnt, int* base, int NS) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < NS; i += blockDim.x) a.counts[i] = cnt[i];
    if (a.block_counts) {
        const int spb = a.S / a.n_blocks;
        for (int b = tid; b < a.n_blocks; b += blockDim.x) {
            int sum = 0;
            for (int s = b * spb; s < (b + 1) * spb; ++s) sum += cnt[s];
            a.block_counts[b] = sum;
        }
    }
    if (!a.offsets) return;
    if (warp == 0) {
        const int ps = (NS + 31) / 32;
        const int s0 = min(NS, lane * ps), s1 = min(NS, s0 + ps);
        int sum = 0;
        for (int s = s0; s < s1; ++s) sum += cnt[s];
        int incl = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        int r = incl - sum;
        for (int s = s0; s < s1; ++s) {
            base[s] = r;
            r += cnt[s];
        }
        if (lane == 31) base[NS] = incl;
    }
    __syncthreads();
    for (int i = tid; i <= NS; i += blockDim.x) a.offsets[i] = base[i];
}

// One CTA: index work for all T*k assignments (a = t*k + j).  Warp w owns the
// contiguous range [w*per, (w+1)*per) of assignments, so warp order is
// assignment order.  Pass 1 counts per warp and slot; a scan over warps gives
// each warp its first rank in every slot; pass 2 walks the range again in
// order and hands out ranks.
__global__ void __launch_bounds__(kIdxThreads, 1) index_pass_kernel(const DispatchArgs a) {
    pdl_begin();
    extern __shared__ int sm[];
    const int NS = a.S + 1;    // slots + invalid bucket
    int* cnt = sm;             // [NS]
    int* base = cnt + NS;      // [NS + 1]
    int* wc = base + NS + 1;   // [32][NS]: per-warp counts, then per-warp next rank
    const int tid = threadIdx.x, warp = tid >> 5;
    const int n = a.T * a.k;
    // warps that own assignments: one 32-wide step each while there are few
    const int nw = min(32, max(1, (n + 31) / 32));
    const int per = (n + nw - 1) / nw;
    const int r0 = warp < nw ? min(n, warp * per) : n, r1 = warp < nw ? min(n, r0 + per) : n;
    int* mine = wc + min(warp, nw - 1) * NS;  // warps >= nw have empty ranges

    for (int i = tid; i < nw * NS; i += kIdxThreads) wc[i] = 0;
    __syncthreads();
    bool bad = false;
    warp_count_range(a, r0, r1, mine, bad);
    if (bad) raise_status(a.st, kStatusInvalidExpert);
    __syncthreads();

    // per slot: exclusive prefix over warps; totals are the counts
    for (int s = tid; s < NS; s += kIdxThreads) {
        int run = 0;
        for (int w = 0; w < nw; ++w) {
            const int c = wc[w * NS + s];
            wc[w * NS + s] = run;
            run += c;
        }
        cnt[s] = run;
    }
    __syncthreads();
    finish_counts(a, cnt, base, NS);
    if (!a.offsets) return;  // histogram only
    for (int s = tid; s < NS; s += kIdxThreads)
        for (int w = 0; w < nw; ++w) wc[w * NS + s] += base[s];
    __syncthreads();
    warp_rank_range(a, r0, r1, mine);
}

// ---- many assignments: the same counting sort over chunks of kChunk
// assignments, one CTA each, in three launches.  hist [chunks][NS] (the
// caller's workspace) holds each chunk's count per slot, then the chunk's
// first rank in each slot.
constexpr int kChunkThreads = 256;
constexpr int kChunkWarps = kChunkThreads / 32;

__device__ __forceinline__ void chunk_range(int n, int chunk, int& lo, int& hi) {
    lo = min(n, (int)blockIdx.x * chunk);
    hi = min(n, lo + chunk);
}

// launch 1: per-chunk slot histograms (and slot_of)
__global__ void __launch_bounds__(kChunkThreads) index_hist_kernel(const DispatchArgs a, int chunk,
                                                                   int32_t* __restrict__ hist) {
    pdl_begin();
    extern __shared__ int sm[];
    const int NS = a.S + 1;
    int* cnt = sm;  // [NS]
    for (int i = threadIdx.x; i < NS; i += kChunkThreads) cnt[i] = 0;
    __syncthreads();
    int lo, hi;
    chunk_range(a.T * a.k, chunk, lo, hi);
    bool bad = false;
    for (int x = lo + (int)threadIdx.x; x < hi; x += kChunkThreads) {
        const int slot = slot_of_assignment(a, x, bad);
        if (a.slot_of) a.slot_of[x] = slot;
        atomicAdd(&cnt[slot], 1);
    }
    if (bad) raise_status(a.st, kStatusInvalidExpert);
    __syncthreads();
    for (int i = threadIdx.x; i < NS; i += kChunkThreads) hist[(size_t)blockIdx.x * NS + i] = cnt[i];
}

// launch 2 (one CTA): per slot, exclusive prefix over chunks (in place) and the
// totals; then counts, block loads and offsets
__global__ void __launch_bounds__(kIdxThreads, 1) index_scan_kernel(const DispatchArgs a, int n_chunks,
                                                                    int32_t* __restrict__ hist) {
    pdl_begin();
    extern __shared__ int sm[];
    const int NS = a.S + 1;
    int* cnt = sm;          // [NS]
    int* base = cnt + NS;   // [NS + 1]
    for (int s = threadIdx.x; s < NS; s += kIdxThreads) {
        int run = 0;
        for (int c0 = 0; c0 < n_chunks; c0 += 8) {
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = c0 + u < n_chunks ? hist[(size_t)(c0 + u) * NS + s] : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (c0 + u < n_chunks) {
                    hist[(size_t)(c0 + u) * NS + s] = run;
                    run += v[u];
                }
            }
        }
        cnt[s] = run;
    }
    __syncthreads();
    finish_counts(a, cnt, base, NS);
}

// launch 3: ranks within each chunk (per-warp ranges as in the one-CTA pass),
// offset by the slot's offset and the chunk's first rank in the slot
__global__ void __launch_bounds__(kChunkThreads) index_rank_kernel(const DispatchArgs a, int chunk,
                                                                   const int32_t* __restrict__ hist) {
    pdl_begin();
    extern __shared__ int sm[];
    const int NS = a.S + 1;
    int* wc = sm;  // [kChunkWarps][NS]
    const int tid = threadIdx.x, warp = tid >> 5;
    int lo, hi;
    chunk_range(a.T * a.k, chunk, lo, hi);
    const int per = (hi - lo + kChunkWarps - 1) / kChunkWarps;
    const int r0 = min(hi, lo + warp * per), r1 = min(hi, r0 + per);
    int* mine = wc + warp * NS;
    for (int i = tid; i < kChunkWarps * NS; i += kChunkThreads) wc[i] = 0;
    __syncthreads();
    bool unused = false;
    warp_count_range(a, r0, r1, mine, unused);
    __syncthreads();
    for (int s = tid; s < NS; s += kChunkThreads) {
        int run = a.offsets[s] + hist[(size_t)blockIdx.x * NS + s];
        for (int w = 0; w < kChunkWarps; ++w) {
            const int c = wc[w * NS + s];
            wc[w * NS + s] = run;
            run += c;
        }
    }
    __syncthreads();
    warp_rank_range(a, r0, r1, mine);
}

// x_disp[row] = x[perm[row] / k] in 16-byte vectors.  A row is spread over
// tpr threads (a multiple of 32) that each issue all of their (at most
// kCopyVpt) loads before storing; blockDim.x / tpr rows per CTA.
constexpr int kCopyVpt = 8;
constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) scatter_rows_kernel(const uint4* __restrict__ x,
                                                                    const int32_t* __restrict__ perm, int n_rows,
                                                                    int k, int vec_per_row, int tpr,
                                                                    uint4* __restrict__ x_disp) {
    pdl_begin();
    const int rows_per_cta = blockDim.x / tpr;
    const int sub = threadIdx.x / tpr;
    const int t0 = threadIdx.x - sub * tpr;
    for (int r0 = blockIdx.x * rows_per_cta; r0 < n_rows; r0 += gridDim.x * rows_per_cta) {
        const int row = r0 + sub;
        if (row >= n_rows) continue;
        const int t = __ldg(perm + row) / k;
        const uint4* src = x + (size_t)t * vec_per_row;
        uint4* dst = x_disp + (size_t)row * vec_per_row;
        for (int c0 = 0; c0 < vec_per_row; c0 += kCopyVpt * tpr) {
            uint4 v[kCopyVpt];
#pragma unroll
            for (int j = 0; j < kCopyVpt; ++j) {
                const int c = c0 + t0 + j * tpr;
                if (c < vec_per_row) v[j] = __ldg(src + c);
            }
#pragma unroll
            for (int j = 0; j < kCopyVpt; ++j) {
                const int c = c0 + t0 + j * tpr;
                if (c < vec_per_row) dst[c] = v[j];
            }
        }
    }
}

}  // namespace

int dispatch_max_slots() { return kMaxSlots; }

cudaError_t launch_index_pass(const DispatchArgs& a, cudaStream_t stream) {
    const int NS = a.S + 1;
    const size_t smem = (size_t)(NS + (NS + 1) + NS + 32 * NS) * sizeof(int);
    static std::atomic<uint64_t> configured{0};
    const cudaError_t e = configure_once(configured, [] {
        return cudaFuncSetAttribute(index_pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)((kMaxSlots + 1) * 35 + 8) * (int)sizeof(int));
    });
    if (e != cudaSuccess) return e;
    return launch_pdl(index_pass_kernel, dim3(1), dim3(kIdxThreads), smem, stream, a);
}

int index_chunks(int n) {
    if (n < kChunkedIndexMin) return 0;
    int chunk = kIndexChunk;
    if ((n + chunk - 1) / chunk > kMaxIndexChunks) chunk = (n + kMaxIndexChunks - 1) / kMaxIndexChunks;
    return (n + chunk - 1) / chunk;
}

size_t index_workspace_bytes(int n, int n_slots) {
    return (size_t)index_chunks(n) * (size_t)(n_slots + 1) * sizeof(int32_t);
}

cudaError_t launch_index_chunked(const DispatchArgs& a, int32_t* hist, cudaStream_t stream) {
    const int n = a.T * a.k;
    const int n_chunks = index_chunks(n);
    const int chunk = (n + n_chunks - 1) / n_chunks;
    const int NS = a.S + 1;
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = configure_once(configured, [] {
        return cudaFuncSetAttribute(index_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)(kChunkWarps * (kMaxSlots + 1) * sizeof(int)));
    });
    if (e != cudaSuccess) return e;
    e = launch_pdl(index_hist_kernel, dim3(n_chunks), dim3(kChunkThreads), NS * sizeof(int), stream, a, chunk, hist);
    if (e != cudaSuccess) return e;
    e = launch_pdl(index_scan_kernel, dim3(1), dim3(kIdxThreads), (2 * NS + 1) * sizeof(int), stream, a, n_chunks, hist);
    if (e != cudaSuccess) return e;
    return launch_pdl(index_rank_kernel, dim3(n_chunks), dim3(kChunkThreads), kChunkWarps * NS * sizeof(int), stream, a,
                      chunk, static_cast<const int32_t*>(hist));
}

cudaError_t launch_scatter_rows(const uint16_t* x, const int32_t* perm, int n_rows, int k, int hidden,
                                uint16_t* x_disp, cudaStream_t stream) {
    if (n_rows <= 0) return cudaSuccess;
    const int vec = hidden / 8;
    int tpr = 32;  // the fewest warps that cover the row in one round of loads (at most the CTA)
    while (tpr * kCopyVpt < vec && tpr < kCopyThreads) tpr <<= 1;
    const int rows_per_cta = kCopyThreads / tpr;
    int blocks = (n_rows + rows_per_cta - 1) / rows_per_cta;
    const int cap = num_sms() * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(scatter_rows_kernel, dim3(blocks), dim3(kCopyThreads), 0, stream,
                      reinterpret_cast<const uint4*>(x), perm, n_rows, k, vec, tpr, reinterpret_cast<uint4*>(x_disp));
}

}  // namespace moe
