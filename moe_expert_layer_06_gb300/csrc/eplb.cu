// Online expert-parallel load balancing (EPLB) on one device.
//
// Blog post "专家并行(EP)", section 6.2: monitor per-expert arrivals over a
// recent window and each rank's load (the sum over its experts), trigger a
// rebalance when max/mean rank load exceeds a threshold (1.2 in the post),
// copy hot experts to lightly loaded ranks, then switch the routing table
// without stopping inference, old work finishing on the old table (RCU).
//
// Here the window is a ring of the last W batches' per-slot counts in a
// caller-owned device buffer, updated by one small kernel per batch (no host
// synchronisation).  The migration helpers copy replica weights with
// device-to-device copies on a caller stream and compute the "stable" table
// (the replicas that stay valid while others are being overwritten) that the
// caller serves with until the copies have landed.
#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 1024;

struct WindowHeader {
    int32_t head;    // ring row the next batch goes to
    int32_t filled;  // rows holding a batch (<= window)
    int32_t pad[2];
};

// State layout: header | ring [window][S+1] int32 | sums [S+1] int64 (8-byte aligned).
__host__ __device__ inline size_t sum_offset(int window, int S) {
    const size_t ring_end = sizeof(WindowHeader) + (size_t)window * (S + 1) * sizeof(int32_t);
    return (ring_end + 15) & ~size_t(15);
}

__device__ __forceinline__ int home_slot_dev(int e, int E, int S, int B) {
    const int epb = E / B, spb = S / B;
    return (e / epb) * spb + (e % epb);
}

// One CTA: push one batch's slot counts into the ring, refresh the window sums
// and derive block loads, expert loads, the imbalance ratio and the trigger.
__global__ void __launch_bounds__(kThreads, 1) window_push_kernel(uint8_t* state, int window, int S, int E, int B,
                                                                  const int32_t* __restrict__ counts,
                                                                  const int32_t* __restrict__ replica_of,
                                                                  double threshold, int64_t* block_load,
                                                                  int64_t* expert_load, double* ratio,
                                                                  int32_t* trigger) {
    pdl_begin();
    __shared__ int64_t s_block[1024];
    WindowHeader* hdr = reinterpret_cast<WindowHeader*>(state);
    int32_t* ring = reinterpret_cast<int32_t*>(state + sizeof(WindowHeader));
    int64_t* sum = reinterpret_cast<int64_t*>(state + sum_offset(window, S));
    const int NS = S + 1;
    const int head = hdr->head;
    for (int s = threadIdx.x; s < NS; s += blockDim.x) {
        const int32_t nw = counts[s];
        int32_t* cell = ring + (size_t)head * NS + s;
        const int32_t old = *cell;  // zero until the ring has wrapped (reset clears it)
        *cell = nw;
        sum[s] += (int64_t)nw - (int64_t)old;
    }
    __syncthreads();
    const int spb = S / B;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        int64_t acc = 0;
        for (int s = b * spb; s < (b + 1) * spb; ++s) acc += sum[s];
        s_block[b] = acc;
        if (block_load) block_load[b] = acc;
    }
    if (expert_load) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            int64_t acc = sum[home_slot_dev(e, E, S, B)];
            if (replica_of) {
                const int r = replica_of[e];
                if (r >= 0 && r < S) acc += sum[r];
            }
            expert_load[e] = acc;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t mx = 0, total = 0;
        for (int b = 0; b < B; ++b) {
            total += s_block[b];
            if (s_block[b] > mx) mx = s_block[b];
        }
        if (ratio) *ratio = total > 0 ? (double)mx * (double)B / (double)total : 0.0;
        if (trigger) *trigger = (double)mx * (double)B > threshold * (double)total ? 1 : 0;
        hdr->head = (head + 1) % window;
        hdr->filled = hdr->filled < window ? hdr->filled + 1 : window;
    }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_eplb_window_bytes(const moe_shape_t* shape, int window) {
    if (api_check_shape(shape, 0) != MOE_OK || window < 1) return 0;
    return sum_offset(window, shape->n_slots) + (size_t)(shape->n_slots + 1) * sizeof(int64_t);
}

int moe_eplb_window_reset(const moe_shape_t* shape, int window, void* state, size_t state_bytes, void* stream) {
    int rc = api_check_shape(shape, 0);
    if (rc) return rc;
    if (window < 1) return api_fail(MOE_ERR_INVALID_ARG, "window %d < 1", window);
    if (!state || (reinterpret_cast<uintptr_t>(state) & 15u))
        return api_fail(MOE_ERR_INVALID_ARG, "window state is NULL or not 16-byte aligned");
    const size_t need = moe_eplb_window_bytes(shape, window);
    if (state_bytes < need) return api_fail(MOE_ERR_WORKSPACE, "window state %zu < %zu bytes", state_bytes, need);
    const cudaError_t e = cudaMemsetAsync(state, 0, need, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return api_fail(MOE_ERR_CUDA, "window reset: %s", cudaGetErrorString(e));
    return MOE_OK;
}

int moe_eplb_window_push(const moe_shape_t* shape, int window, void* state, size_t state_bytes,
                         const int32_t* counts, const int32_t* replica_of, double threshold, int64_t* block_load,
                         int64_t* expert_load, double* ratio, int32_t* trigger, void* stream) {
    int rc = api_check_shape(shape, 0);
    if (rc) return rc;
    if (window < 1) return api_fail(MOE_ERR_INVALID_ARG, "window %d < 1", window);
    if (shape->n_blocks > 1024) return api_fail(MOE_ERR_UNSUPPORTED, "n_blocks %d > 1024", shape->n_blocks);
    if (!state || (reinterpret_cast<uintptr_t>(state) & 15u))
        return api_fail(MOE_ERR_INVALID_ARG, "window state is NULL or not 16-byte aligned");
    if (state_bytes < moe_eplb_window_bytes(shape, window))
        return api_fail(MOE_ERR_WORKSPACE, "window state too small");
    if (!counts) return api_fail(MOE_ERR_INVALID_ARG, "counts is NULL");
    if (!(threshold > 0.0)) return api_fail(MOE_ERR_INVALID_ARG, "threshold must be > 0");
    const cudaError_t le = launch_pdl(window_push_kernel, dim3(1), dim3(kThreads), 0,
                                      reinterpret_cast<cudaStream_t>(stream), static_cast<uint8_t*>(state), window,
                                      shape->n_slots, shape->n_experts, shape->n_blocks, counts, replica_of, threshold,
                                      block_load, expert_load, ratio, trigger);
    if (le != cudaSuccess) return api_fail(MOE_ERR_CUDA, "window push launch: %s", cudaGetErrorString(le));
    return MOE_OK;
}

int moe_eplb_stable_table(const moe_shape_t* shape, const int32_t* host_old, const int32_t* host_new,
                          int32_t* host_out) {
    int rc = api_check_shape(shape, 0);
    if (rc) return rc;
    if (!host_new || !host_out) return api_fail(MOE_ERR_INVALID_ARG, "NULL host table");
    for (int e = 0; e < shape->n_experts; ++e) {
        const int32_t o = host_old ? host_old[e] : -1;
        host_out[e] = (o >= 0 && o == host_new[e]) ? o : -1;
    }
    return MOE_OK;
}

int moe_eplb_copy_replicas(const moe_shape_t* shape, const int32_t* host_old, const int32_t* host_new, void* w_gate,
                           void* w_up, void* w_down, void* stream) {
    int rc = api_check_shape(shape, 0);
    if (rc) return rc;
    if (!host_new || !w_gate || !w_up || !w_down) return api_fail(MOE_ERR_INVALID_ARG, "NULL argument");
    const int E = shape->n_experts, S = shape->n_slots, B = shape->n_blocks;
    const int epb = E / B, spb = S / B;
    // validate the whole plan before enqueuing anything
    for (int e = 0; e < E; ++e) {
        const int32_t r = host_new[e];
        if (r < 0) continue;
        if (r >= S || (r % spb) < epb)
            return api_fail(MOE_ERR_INVALID_ARG, "slot %d given to expert %d is not a replica slot", r, e);
        for (int f = e + 1; f < E; ++f)
            if (host_new[f] == r) return api_fail(MOE_ERR_INVALID_ARG, "replica slot %d assigned twice", r);
    }
    const size_t mat = (size_t)shape->inter * shape->hidden * 2;  // bytes of one slot's gate (= up = down)
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* bases[3] = {static_cast<uint8_t*>(w_gate), static_cast<uint8_t*>(w_up), static_cast<uint8_t*>(w_down)};
    for (int e = 0; e < E; ++e) {
        const int32_t r = host_new[e];
        if (r < 0 || (host_old && host_old[e] == r)) continue;  // unchanged replicas keep their weights
        const int home = (e / epb) * spb + (e % epb);
        for (int j = 0; j < 3; ++j) {
            const cudaError_t err = cudaMemcpyAsync(bases[j] + (size_t)r * mat, bases[j] + (size_t)home * mat, mat,
                                                    cudaMemcpyDeviceToDevice, st);
            if (err != cudaSuccess) return api_fail(MOE_ERR_CUDA, "replica copy: %s", cudaGetErrorString(err));
        }
    }
    return MOE_OK;
}

}  // extern "C"
