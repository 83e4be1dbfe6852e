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

__device__ __forceinline__ int home_slot(int e, int E, int S, int n_blocks) {
    const int epb = E / n_blocks, spb = S / n_blocks;
    return (e / epb) * spb + (e % epb);
}

// One CTA: index work for all T*k assignments (a = t*k + j).
__global__ void __launch_bounds__(kIdxThreads, 1) index_pass_kernel(const DispatchArgs a) {
    extern __shared__ int sm[];
    const int NS = a.S + 1;  // slots + invalid bucket
    int* cnt = sm;           // [NS]
    int* base = cnt + NS;    // [NS + 1]
    int* run = base + NS + 1;  // [NS]
    int* wcnt = run + NS;    // [32][NS]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = a.T * a.k;

    for (int i = tid; i < NS; i += kIdxThreads) {
        cnt[i] = 0;
        run[i] = 0;
    }
    __syncthreads();

    // replica remap + histogram (shared-memory atomics: the counts do not depend on order)
    bool bad = false;
    for (int x = tid; x < n; x += kIdxThreads) {
        const int t = x / a.k;
        const int e = a.topk_idx[x];
        int slot;
        if (e < 0 || e >= a.E) {
            slot = a.S;
            bad = true;
        } else {
            slot = home_slot(e, a.E, a.S, a.n_blocks);
            if (a.replica_of && (t & 1)) {
                const int r = a.replica_of[e];
                if (r >= 0) {
                    if (r < a.S) slot = r;
                    else { slot = a.S; bad = true; }
                }
            }
        }
        if (a.slot_of) a.slot_of[x] = slot;
        atomicAdd(&cnt[slot], 1);
    }
    if (bad) raise_status(a.st, kStatusInvalidExpert);
    __syncthreads();

    for (int i = tid; i < NS; i += kIdxThreads) a.counts[i] = cnt[i];
    if (a.block_counts) {
        const int spb = a.S / a.n_blocks;
        for (int b = tid; b < a.n_blocks; b += kIdxThreads) {
            int sum = 0;
            for (int s = b * spb; s < (b + 1) * spb; ++s) sum += cnt[s];
            a.block_counts[b] = sum;
        }
    }
    if (!a.offsets) return;  // histogram only

    // exclusive prefix of counts over slots and the invalid bucket
    if (warp == 0) {
        const int per = (NS + 31) / 32;
        const int s0 = min(NS, lane * per), s1 = min(NS, s0 + per);
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
    for (int i = tid; i <= NS; i += kIdxThreads) a.offsets[i] = base[i];

    // stable ranks: tiles of 1024 assignments in order; within a tile, rank =
    // earlier same-slot lanes of the warp + same-slot counts of earlier warps
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int tile = 0; tile < n; tile += kIdxThreads) {
        const int x = tile + tid;
        const bool valid = x < n;
        const int slot = valid ? a.slot_of[x] : -1;
        for (int i = tid; i < 32 * NS; i += kIdxThreads) wcnt[i] = 0;
        __syncthreads();
        const unsigned peers = __match_any_sync(0xffffffffu, slot);
        const int lane_rank = __popc(peers & lt_mask);
        const bool leader = (__ffs(peers) - 1) == lane;
        const bool lane_last = (31 - __clz(peers)) == lane;
        if (valid && leader) wcnt[warp * NS + slot] = __popc(peers);
        __syncthreads();
        int before = 0, after = 0, r0 = 0;
        if (valid) {
            for (int w = 0; w < warp; ++w) before += wcnt[w * NS + slot];
            for (int w = warp + 1; w < 32; ++w) after += wcnt[w * NS + slot];
            r0 = run[slot];
            const int row = base[slot] + r0 + before + lane_rank;
            a.perm[row] = x;
            a.inv_perm[x] = row;
        }
        __syncthreads();
        if (valid && lane_last && after == 0) run[slot] = r0 + before + lane_rank + 1;
    }
}

// x_disp[row] = x[perm[row] / k], 16-byte vectors, one warp per row.
__global__ void __launch_bounds__(256) scatter_rows_kernel(const uint4* __restrict__ x,
                                                           const int32_t* __restrict__ perm, int n_rows,
                                                           int k, int vec_per_row, uint4* __restrict__ x_disp) {
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    for (int row = blockIdx.x * wpb + (threadIdx.x >> 5); row < n_rows; row += gridDim.x * wpb) {
        const int t = perm[row] / k;
        const uint4* src = x + (size_t)t * vec_per_row;
        uint4* dst = x_disp + (size_t)row * vec_per_row;
        for (int v = lane; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
    }
}

}  // namespace

int dispatch_max_slots() { return kMaxSlots; }

cudaError_t launch_index_pass(const DispatchArgs& a, cudaStream_t stream) {
    const int NS = a.S + 1;
    const size_t smem = (size_t)(NS + (NS + 1) + NS + 32 * NS) * sizeof(int);
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(index_pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)((kMaxSlots + 1) * 35 + 8) * (int)sizeof(int));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    index_pass_kernel<<<1, kIdxThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_scatter_rows(const uint16_t* x, const int32_t* perm, int n_rows, int k, int hidden,
                                uint16_t* x_disp, cudaStream_t stream) {
    if (n_rows <= 0) return cudaSuccess;
    const int wpb = 8;
    int blocks = (n_rows + wpb - 1) / wpb;
    const int cap = num_sms() * 16;
    if (blocks > cap) blocks = cap;
    scatter_rows_kernel<<<blocks, wpb * 32, 0, stream>>>(reinterpret_cast<const uint4*>(x), perm, n_rows, k,
                                                         hidden / 8, reinterpret_cast<uint4*>(x_disp));
    return cudaGetLastError();
}

}  // namespace moe
