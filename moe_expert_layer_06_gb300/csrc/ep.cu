// Expert parallelism across GPUs: the bookkeeping of the two all-to-alls.
//
// Blog post "专家并行(EP)", section 2.1: EP rank g holds the experts of block g
// (32 of 256, or 33 slots with a replica); section 2.2 steps 2 and 4: a token's
// hidden state goes to the ranks that hold its experts (dispatch all-to-all)
// and the expert outputs come back (combine all-to-all); section 2.3: the
// volume is 2 x top-k x hidden x 2 bytes per token each way.
//
// On the sending rank the dispatch buffer is already grouped by slot and so by
// block: the rows for rank g are the contiguous segment of block g's slots.
// The receiving rank gets, from every source rank s in turn, that source's
// rows for its own slots, slot by slot ("source-major").  Its expert GEMMs
// want each slot's rows together ("slot-major": slot j's rows from source 0,
// then source 1, ...).  moe_ep_plan derives the row counts of both
// all-to-alls and the two permutations between the layouts from the exchanged
// per-slot counts; moe_gather_rows applies a permutation on the device.  The
// combine all-to-all sends each rank's expert outputs back along the same
// segments in reverse, so they land in the sender's dispatch-buffer order.
#include <string.h>

#include "kernels.h"

extern "C" {

int moe_ep_plan(const moe_shape_t* shape, int world, const int32_t* counts, const int32_t* recv_counts,
                int32_t* send_rows, int32_t* recv_rows, int32_t* local_offsets, int32_t* slot_from_src,
                int32_t* src_from_slot, int32_t rows_cap, int32_t* rows_out) {
    using namespace moe;
    int rc = api_check_shape(shape, 1);
    if (rc != MOE_OK) return rc;
    if (world < 1 || shape->n_blocks != world)
        return api_fail(MOE_ERR_INVALID_ARG, "moe_ep_plan: world %d must equal n_blocks %d", world, shape->n_blocks);
    if (!counts || !recv_counts || !send_rows || !recv_rows || !local_offsets || !rows_out)
        return api_fail(MOE_ERR_INVALID_ARG, "moe_ep_plan: null argument");
    const int S = shape->n_slots;
    const int spb = S / world;
    // rows this rank sends to each rank: the counts of that rank's slots
    for (int g = 0; g < world; ++g) {
        long sum = 0;
        for (int j = 0; j < spb; ++j) {
            const int32_t c = counts[g * spb + j];
            if (c < 0) return api_fail(MOE_ERR_INVALID_ARG, "moe_ep_plan: negative count at slot %d", g * spb + j);
            sum += c;
        }
        if (sum > INT32_MAX) return api_fail(MOE_ERR_UNSUPPORTED, "moe_ep_plan: more than 2^31 rows");
        send_rows[g] = (int32_t)sum;
    }
    // rows received from each source and the slot-major offsets of the local slots
    long total = 0;
    for (int s = 0; s < world; ++s) {
        long sum = 0;
        for (int j = 0; j < spb; ++j) {
            const int32_t c = recv_counts[(size_t)s * spb + j];
            if (c < 0) return api_fail(MOE_ERR_INVALID_ARG, "moe_ep_plan: negative received count");
            sum += c;
        }
        recv_rows[s] = (int32_t)sum;
        total += sum;
    }
    if (total > INT32_MAX) return api_fail(MOE_ERR_UNSUPPORTED, "moe_ep_plan: more than 2^31 rows");
    const int32_t R = (int32_t)total;
    *rows_out = R;
    int32_t run = 0;
    for (int j = 0; j < spb; ++j) {
        local_offsets[j] = run;
        for (int s = 0; s < world; ++s) run += recv_counts[(size_t)s * spb + j];
    }
    local_offsets[spb] = run;
    local_offsets[spb + 1] = run;
    if (!slot_from_src && !src_from_slot) return MOE_OK;
    if (R > rows_cap)
        return api_fail(MOE_ERR_INVALID_ARG, "moe_ep_plan: %d received rows exceed the map capacity %d", R,
                        rows_cap);
    // source-major position p of (source s, local slot j, i-th row) against its
    // slot-major position q
    int32_t p = 0;
    for (int s = 0; s < world; ++s) {
        for (int j = 0; j < spb; ++j) {
            int32_t q = local_offsets[j];
            for (int s2 = 0; s2 < s; ++s2) q += recv_counts[(size_t)s2 * spb + j];
            const int32_t c = recv_counts[(size_t)s * spb + j];
            for (int i = 0; i < c; ++i, ++p) {
                if (slot_from_src) slot_from_src[q + i] = p;
                if (src_from_slot) src_from_slot[p] = q + i;
            }
        }
    }
    return MOE_OK;
}

int moe_gather_rows(int n_rows, int row_bytes, const void* src, const int32_t* index, void* dst, void* stream) {
    using namespace moe;
    if (n_rows < 0 || row_bytes <= 0 || row_bytes % 16)
        return api_fail(MOE_ERR_INVALID_ARG, "moe_gather_rows: n_rows >= 0 and row_bytes %% 16 == 0 required");
    if (n_rows == 0) return MOE_OK;
    if (!src || !index || !dst) return api_fail(MOE_ERR_INVALID_ARG, "moe_gather_rows: null argument");
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u)
        return api_fail(MOE_ERR_INVALID_ARG, "moe_gather_rows: src and dst must be 16-byte aligned");
    PdlScope pdl(n_rows);
    // dst[i] = src[index[i]]: the dispatch scatter with one copy per row
    const cudaError_t e = launch_scatter_rows(static_cast<const uint16_t*>(src), index, n_rows, 1, row_bytes / 2,
                                              static_cast<uint16_t*>(dst), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return api_fail(MOE_ERR_CUDA, "moe_gather_rows launch: %s", cudaGetErrorString(e));
    return MOE_OK;
}

}  // extern "C"
