/*
 * libmoe — forward pass of a DeepSeek-V3-style Mixture-of-Experts layer on one
 * GB300 GPU (sm_103a), as a C ABI.
 *
 * The layer is the expert-parallel MoE layer of the blog post "专家并行(EP)"
 * (expert parallelism).  Its section 2.2 follows one token through five steps:
 *   1. router linear [hidden, n_experts] -> logits -> top-k experts;
 *   2. dispatch: the token's hidden state goes to each selected expert;
 *   3. each expert computes its FFN on the rows it received;
 *   4. combine: the expert outputs return to the token;
 *   5. output = sum over the top-k of softmax(logits)[i] * expert_output[i]
 *      plus the shared expert output.
 * Section 2.1 lays the routed experts out in contiguous blocks (one per EP
 * rank) with the shared experts replicated; section 6.2 monitors per-expert
 * arrivals and per-rank load; section 6.3 adds redundant expert slots.
 * On one device the two all-to-alls become permutations in device memory:
 * the dispatch buffer holds the rows of every slot contiguously, slot after
 * slot, so the rows of each EP block are contiguous too.
 *
 * Conventions (all entry points)
 *   - "bf16" arrays are raw 16-bit bfloat16 values (passed as void*).
 *   - Device pointers are owned by the caller; the library never allocates,
 *     frees or retains them.  Unless stated otherwise every pointer is a
 *     device pointer, 16-byte aligned, row-major and densely packed.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device
 *     work is enqueued asynchronously on it; the call returns once enqueued.
 *   - Every call returns an int status (MOE_OK = 0).  Nothing aborts, traps
 *     or prints.  Arguments are validated before anything is enqueued; on an
 *     error nothing is enqueued and moe_last_error_string() says why.
 *   - Errors found on the device (an expert id outside [0, E), a bounded
 *     wait that expired) set a device status word instead of faulting;
 *     moe_check_status() synchronises the stream, reads and clears it.
 *   - T = 0 is valid and enqueues nothing.
 *   - Every *_workspace_size(shape, T) is non-decreasing in T: a workspace
 *     sized for the largest batch serves every smaller one.
 *   - Any number of host threads may call concurrently, each on its own
 *     stream and buffers: the library's per-device set-up is done once under
 *     atomics, the error text is per thread, and the device status word is
 *     shared (one thread's moe_check_status may report and clear another's
 *     error).  moe_expert_ffn_noalloc calls must not overlap (one scratch).
 *   - Calls enqueue kernels only.  moe_forward and moe_forward_fp8 replay
 *     from a captured CUDA graph (tested).  The first use of each kernel on
 *     a device sets its shared-memory attribute (cudaFuncSetAttribute, a
 *     host-side setting, not a graph node): make the same call (same entry
 *     point, shape and T) once before capturing it, as a warm-up does.
 *   - Calls of at most 8192 token-expert assignments (T*k) launch their
 *     kernels with programmatic dependent launch: a kernel may be scheduled
 *     while its predecessor in the stream finishes and waits for it before
 *     touching memory, so results and memory order are those of plain stream
 *     order (a caller's own kernel before it is waited for the same way).
 *
 * Notation: T tokens, H hidden, I routed intermediate, E routed experts,
 * k top-k, S slots (E, or E + redundant replicas), B blocks (EP ranks),
 * n_sh shared experts of intermediate I_sh.  Slot layout: block b owns slots
 * [b*S/B, (b+1)*S/B); its experts b*E/B .. (b+1)*E/B-1 sit in its first E/B
 * slots in order (home slots), its remaining slots hold replicas.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1     /* null/misaligned pointer, bad size, inconsistent shape */
#define MOE_ERR_UNSUPPORTED 2     /* valid shape outside the library's kernel limits */
#define MOE_ERR_CUDA 3            /* a CUDA runtime call or launch failed */
#define MOE_ERR_DEVICE_TIMEOUT 4  /* a kernel's bounded wait expired (moe_check_status) */
#define MOE_ERR_DEVICE_STATUS 5   /* a kernel flagged invalid data, e.g. expert id out of range */
#define MOE_ERR_WORKSPACE 6       /* workspace null or smaller than the *_workspace_size() answer */

/* Expert FFN kernel variant: token chunk of 32 rows (decode: weights streamed
 * once per 32 rows of an expert) or 160 rows (prefill).  AUTO picks 32 when
 * T <= 32 and 160 above, except the E4M3 down projection (moe_expert_down_fp8,
 * and inside moe_forward_fp8) when the batch averages at most 32 rows per slot
 * (T*k <= 32*S), which takes a 128-row chunk with double-buffered
 * accumulators.  Results are identical up to fp32 summation order. */
#define MOE_FFN_AUTO 0
#define MOE_FFN_DECODE 1
#define MOE_FFN_PREFILL 2

/* Layer shape.  Limits of the library: 1 <= k <= min(E, 32); E <= 1024;
 * S <= 1024; E and S divisible by B with S/B >= E/B; H, I, I_sh multiples of 8. */
typedef struct {
    int32_t hidden;        /* H */
    int32_t inter;         /* I */
    int32_t n_experts;     /* E */
    int32_t top_k;         /* k */
    int32_t n_shared;      /* n_sh (0 = no shared expert) */
    int32_t inter_shared;  /* I_sh */
    int32_t n_slots;       /* S */
    int32_t n_blocks;      /* B */
} moe_shape_t;

/* Text of the last error raised on the calling thread ("" if none). */
MOE_API const char* moe_last_error_string(void);

/* Library ABI version (increments on any signature change). */
MOE_API int moe_abi_version(void);

/* Synchronise `stream`, read and clear the current device's status word.
 * Returns MOE_OK, MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_DEVICE_STATUS. */
MOE_API int moe_check_status(void* stream);

/* Bound (nanoseconds of device time) of every spin wait in later launches on
 * any device; default 2e9.  Returns MOE_ERR_INVALID_ARG for 0. */
MOE_API int moe_set_wait_limit_ns(uint64_t ns);

/* Launch one kernel whose bounded wait is on a barrier nothing completes: it
 * gives up after the current wait limit and sets the timeout status, which
 * moe_check_status() then reports.  For tests of the failure path only. */
MOE_API int moe_debug_expire_wait(void* stream);

/* ---------------------------------------------------------------- step 1: route
 * "专家并行(EP)" section 2.2 step 1 (router linear, top-k) and step 5 (the
 * combine weight softmax(logits)[i]).
 *   logits[t,e] = sum_h x[t,h] * w_router[e,h] (+ bias[e]), fp32 accumulation
 *     on the tensor cores (router GEMM split over K, partials summed in a fixed
 *     order);
 *   topk_idx[t,0..k-1]: the k largest logits, descending, equal values ->
 *     lower expert index first;
 *   topk_w[t,j] = softmax over all E logits at topk_idx[t,j] (fp32, not
 *     renormalised over the top-k).
 * x [T,H] bf16; w_router [E,H] bf16 (one row per expert); bias [E] fp32 or
 * NULL.  logits_in [T,E] fp32 or NULL: when given, the GEMM is skipped and the
 * selection runs on these final logits (bias must then be NULL; x, w_router
 * may be NULL).  logits_out [T,E] fp32 or NULL receives the logits used.
 * The GEMM sums K in splits whose number follows T and the device's SM
 * count, added in a fixed order: results repeat bit for bit on one GPU model
 * and may differ in the last bits of the logits on another.
 * Outputs topk_idx [T,k] int32, topk_w [T,k] fp32.  ws: device workspace of
 * at least moe_route_workspace_size() bytes (may be NULL if that is 0). */
MOE_API size_t moe_route_workspace_size(const moe_shape_t* shape, int T);
MOE_API int moe_route(const moe_shape_t* shape, int T, const void* x, const void* w_router, const float* bias,
              const float* logits_in, float* logits_out, int32_t* topk_idx, float* topk_w, void* ws,
              size_t ws_bytes, void* stream);

/* Group-limited routing (the post's summary section names routing by expert
 * group first and by expert second as a direction for larger expert counts).
 * The E experts form n_groups contiguous groups of E/n_groups (with
 * n_groups = B these are the EP blocks); a group scores its largest logit;
 * the topk_groups best groups are kept (ties -> lower group); topk_idx is the
 * top-k of the kept groups' experts (same order and tie rule as moe_route);
 * topk_w is still softmax over all E logits.  1 <= n_groups <= 32,
 * n_groups divides E, 1 <= topk_groups <= n_groups, k <= topk_groups*E/n_groups.
 * Other arguments, workspace and outputs as moe_route. */
MOE_API int moe_route_grouped(const moe_shape_t* shape, int T, int n_groups, int topk_groups, const void* x,
                              const void* w_router, const float* bias, const float* logits_in, float* logits_out,
                              int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- EPLB monitor
 * "专家并行(EP)" section 6.2 ("monitor": tokens arriving at each expert; a
 * rank's load = sum over its experts) for one batch, and section 6.3 (a token
 * may use any replica of its expert).
 *   slot(t,j) = replica_of[e] if replica_of != NULL, replica_of[e] >= 0 and t
 *               is odd; else e's home slot  (e = topk_idx[t,j]);
 *   counts[s] = number of assignments to slot s (s < S); counts[S] = number of
 *               expert ids outside [0,E) (these also set the device status);
 *   block_counts[b] = sum of counts over block b's slots (NULL to skip).
 * topk_idx [T,k] int32; replica_of [E] int32 or NULL (values -1 or a slot in
 * [0,S)); counts [S+1] int32; block_counts [B] int32. */
MOE_API int moe_expert_histogram(const moe_shape_t* shape, int T, const int32_t* topk_idx, const int32_t* replica_of,
                         int32_t* counts, int32_t* block_counts, void* stream);

/* Imbalance of per-block loads (host arrays): max / mean, 0 if all are zero.
 * Section 6.2 rebalances when it exceeds a threshold (typically 1.2). */
MOE_API double moe_eplb_imbalance(const int32_t* host_block_counts, int n_blocks);

/* Redundant-expert placement (host-only, section 6.2 "copy the overloaded
 * rank's hottest experts to an idle rank", section 6.3 "8 redundant experts").
 * From per-expert counts host_expert_counts[E]: the n_rep hottest experts
 * (count descending, ties -> lower id) each get one replica.  A block's load
 * starts as the sum of its experts' counts with a hot expert's count halved;
 * in hot order, each replica goes to the least-loaded block (ties -> lower
 * block) that has a free replica slot and is not the expert's home block,
 * else to its home block if that has one free; the block's load then grows by
 * half the expert's count, and the replica takes that block's first free
 * replica slot.  Output host_replica_of[E]: slot or -1.
 * The caller copies the source expert's weights into each replica slot. */
MOE_API int moe_eplb_plan_replicas(const moe_shape_t* shape, const int32_t* host_expert_counts, int n_rep,
                           int32_t* host_replica_of);

/* ---------------------------------------------------------------- EPLB online loop
 * Section 6.2: monitor arrivals over a recent window, detect when the most
 * loaded rank exceeds the mean by a threshold (1.2 in the post), copy hot
 * experts to other ranks and switch the routing table without stopping
 * inference.  The window is the last `window` batches (a reading: the post
 * speaks of a time span such as 100 ms).
 *
 * moe_eplb_window_bytes / _reset: size and zeroing of the caller-owned device
 * state (ring of `window` rows of S+1 int32 slot counts + S+1 int64 sums).
 * moe_eplb_window_push: one small kernel per batch, no host synchronisation.
 * Pushes counts [S+1] (as written by moe_dispatch / moe_expert_histogram),
 * dropping the oldest row once full, then writes (each output may be NULL,
 * all device pointers):
 *   block_load[B]  = windowed counts summed over the block's slots (int64);
 *   expert_load[E] = windowed count of e's home slot + its replica slot under
 *                    replica_of (may be NULL) (int64);
 *   ratio[1]       = max(block_load) * B / sum(block_load), 0 if the sum is 0;
 *   trigger[1]     = 1 if max * B > threshold * sum (evaluated in double).
 * Calls on one state must be stream-ordered. */
MOE_API size_t moe_eplb_window_bytes(const moe_shape_t* shape, int window);
MOE_API int moe_eplb_window_reset(const moe_shape_t* shape, int window, void* state, size_t state_bytes,
                                  void* stream);
MOE_API int moe_eplb_window_push(const moe_shape_t* shape, int window, void* state, size_t state_bytes,
                                 const int32_t* counts, const int32_t* replica_of, double threshold,
                                 int64_t* block_load, int64_t* expert_load, double* ratio, int32_t* trigger,
                                 void* stream);

/* Migration without stopping inference (host helpers, RCU-like switch).
 * A new plan (moe_eplb_plan_replicas) overwrites replica slots that the old
 * plan may still be using.  Safe order on one device:
 *   1. moe_eplb_stable_table(old, new, stable): stable[e] = old[e] where the
 *      old and new plans agree, else -1 (home slot only); upload it and use it
 *      for every batch enqueued from now on;
 *   2. on a copy stream that waits for the last batch using `old`, call
 *      moe_eplb_copy_replicas(old, new, ...): for every expert whose replica
 *      slot changes, 3 device-to-device copies (gate, up, down) from its home
 *      slot into the new replica slot (no allocation);
 *   3. make the compute stream wait for the copies, then use `new`.
 * Every batch sees a table whose replica slots hold the right weights, so the
 * layer output is unchanged throughout (replicas are byte copies).  host_old
 * may be NULL (no replicas before).  Weights are slot-major [S,I,H] / [S,H,I]. */
MOE_API int moe_eplb_stable_table(const moe_shape_t* shape, const int32_t* host_old, const int32_t* host_new,
                                  int32_t* host_out);
MOE_API int moe_eplb_copy_replicas(const moe_shape_t* shape, const int32_t* host_old, const int32_t* host_new,
                                   void* w_gate, void* w_up, void* w_down, void* stream);

/* ---------------------------------------------------------------- step 2: dispatch
 * Section 2.2 step 2.  Slot map and histogram as moe_expert_histogram, then
 *   offsets[s] = sum_{s'<s} counts[s'] for s <= S+1 (offsets[S+1] = T*k; the
 *     rows of out-of-range ids sit in [offsets[S], offsets[S+1]));
 *   rows of slot s: [offsets[s], offsets[s+1]), in ascending a = t*k + j;
 *   perm[row] = a, inv_perm[a] = row;
 *   x_disp[row,:] = x[perm[row] / k, :]  (16-byte vector copies).
 * The buffer is exactly T*k*H*2 bytes; with the equally sized combine payload
 * that is 2*k*H*2 bytes per token (229,376 B at k=8, H=7168, section 2.3).
 * x [T,H] bf16; topk_idx [T,k]; replica_of [E] or NULL; outputs slot_of [T*k],
 * counts [S+1], block_counts [B] (or NULL), offsets [S+2], perm [T*k],
 * inv_perm [T*k] int32, x_disp [T*k,H] bf16.  ws: device scratch of
 * moe_dispatch_workspace_size(shape, T) bytes, 16-byte aligned (the size is 0,
 * and ws may be NULL, below 4096 assignments; above, the index pass runs in
 * chunks of 512 assignments with their histograms in ws), else
 * MOE_ERR_WORKSPACE. */
MOE_API size_t moe_dispatch_workspace_size(const moe_shape_t* shape, int T);
MOE_API int moe_dispatch(const moe_shape_t* shape, int T, const void* x, const int32_t* topk_idx,
                 const int32_t* replica_of, int32_t* slot_of, int32_t* counts, int32_t* block_counts,
                 int32_t* offsets, int32_t* perm, int32_t* inv_perm, void* x_disp, void* ws, size_t ws_bytes,
                 void* stream);

/* ---------------------------------------------------------------- step 3: expert FFN
 * Section 2.2 step 3 (each expert's FFN on its rows) with the SwiGLU form
 * h = silu(X W_g^T) * (X W_u^T), y = h W_d^T; the shared experts (section 2.1)
 * run on all T rows of x.  Grouped tcgen05 GEMMs, fp32 accumulation, h rounded
 * to bf16.
 * moe_expert_gate_up:
 *   h_disp[row, :] = silu(x_disp[row] . W_g[s]^T) * (x_disp[row] . W_u[s]^T),
 *     rows of slot s = [offsets[s], offsets[s+1]);
 *   h_shared[t, j*I_sh + :] = the same with shared expert j on x[t].
 * moe_expert_down:
 *   y_disp[row, :] = bf16(h_disp[row] . W_d[s]^T);
 *   y_shared[t, :] = sum_j h_shared[t, j*I_sh:(j+1)*I_sh] . Ws_d[j]^T (fp32).
 * moe_expert_ffn = gate_up then down, h in the workspace.
 * Layouts: w_gate, w_up [S,I,H]; w_down [S,H,I]; ws_gate, ws_up [n_sh,I_sh,H];
 * ws_down [n_sh,H,I_sh] (bf16, one nn.Linear [out,in] matrix per slot).
 * x [T,H]; x_disp, y_disp [T*k,H]; h_disp [T*k,I]; h_shared [T,n_sh*I_sh] bf16;
 * y_shared [T,H] fp32; offsets [S+2] from moe_dispatch.  Shared pointers may be
 * NULL when n_sh = 0.  Rows of out-of-range ids are not computed. */
MOE_API int moe_expert_gate_up(const moe_shape_t* shape, int T, const void* x, const void* x_disp,
                       const int32_t* offsets, const void* w_gate, const void* w_up, const void* ws_gate,
                       const void* ws_up, void* h_disp, void* h_shared, int mode, void* stream);
MOE_API int moe_expert_down(const moe_shape_t* shape, int T, const void* h_disp, const void* h_shared,
                    const int32_t* offsets, const void* w_down, const void* ws_down, void* y_disp,
                    float* y_shared, int mode, void* stream);
MOE_API size_t moe_ffn_workspace_size(const moe_shape_t* shape, int T);
MOE_API int moe_expert_ffn(const moe_shape_t* shape, int T, const void* x, const void* x_disp, const int32_t* offsets,
                   const void* w_gate, const void* w_up, const void* w_down, const void* ws_gate,
                   const void* ws_up, const void* ws_down, void* y_disp, float* y_shared, int mode, void* ws,
                   size_t ws_bytes, void* stream);

/* Capacity of the fixed device scratch used by moe_expert_ffn_noalloc (bytes). */
#define MOE_FFN_NOALLOC_SCRATCH_BYTES (8u << 20)

/* moe_expert_ffn without a workspace, for callers that cannot allocate device
 * memory (for instance a plugin whose host program owns every allocation and
 * passes it only inputs and outputs, or a latency-critical path where
 * cudaMalloc's implicit device synchronisation is not acceptable).  The
 * expert-parallel post has no counterpart to this entry point.
 * Same arguments, layouts and results as moe_expert_ffn, minus ws/ws_bytes:
 * the SwiGLU intermediate (T*k*I*2 bytes rounded up to 256, plus
 * T*n_sh*I_sh*2) lives in a fixed array of MOE_FFN_NOALLOC_SCRATCH_BYTES in
 * the library's device memory, which every GPU that loads the library holds
 * until the process exits.  Larger T returns MOE_ERR_UNSUPPORTED (8 MiB holds
 * T <= 204 at the DeepSeek-V3 shape, k=8, I=2048, two shared experts of 2048).
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress); make that first call before any stream
 * capture.  All calls share the array and each leaves its contents there:
 * calls whose work may overlap on the GPU (other streams, other threads on the
 * same device) race on it and must be serialised by the caller.  Allocates
 * nothing (no cudaMalloc, cudaFree or allocating library call). */
MOE_API int moe_expert_ffn_noalloc(const moe_shape_t* shape, int T, const void* x, const void* x_disp,
                                   const int32_t* offsets, const void* w_gate, const void* w_up,
                                   const void* w_down, const void* ws_gate, const void* ws_up,
                                   const void* ws_down, void* y_disp, float* y_shared, int mode, void* stream);

/* ---------------------------------------------------------------- FP8 path
 * Section 2.3: FP8 communication halves the per-token dispatch + combine
 * volume.  Format E4M3 (OCP 8-bit float: 4 exponent bits, bias 7, 3 mantissa
 * bits, largest finite 448).  A row is stored as codes plus one fp32 scale:
 * scale = amax(|row|) / 448 (1 for an all-zero row), code = e4m3(x / scale)
 * rounded to nearest even with saturation (the division in fp32); its value
 * is decode(code) * scale.
 *
 * moe_quantize_rows_fp8: rows x cols bf16 -> codes [rows, cols] u8 and
 * scale [rows] fp32 (cols % 16 == 0).  Use it once on the expert gate and up
 * weights ([S*I, H] and [n_sh*I_sh, H]: one scale per output row).
 * moe_dispatch_fp8: moe_dispatch (same workspace), except that each token is quantised once
 * (x8 [T,H] u8, x_scale [T]) and its dispatched copies carry its codes and
 * scale (x_disp8 [T*k,H] u8, x_disp_scale [T*k]): the dispatch buffer is
 * T*k*H bytes, half of the bf16 one (57,344 B per token at k=8, H=7168).
 * moe_expert_gate_up_fp8: moe_expert_gate_up with E4M3 operands on the FP8
 * tensor cores; h = silu(g) * u with g = sx*sg[i]*sum(qx*qg) (fp32 accumulate),
 * u likewise; h out in bf16, as for moe_expert_gate_up.  hidden % 16 == 0.
 * moe_expert_down_fp8: the down projection with E4M3 operands.  The bf16
 * intermediate is quantised with moe_quantize_rows_fp8: h_disp [T*k, I] rows
 * give h8 [T*k, I] + h_scale [T*k]; the shared experts' intermediate
 * h_shared [T, n_sh*I_sh] gives one row per token, hs8 + hs_scale [T].
 * Routed down weights qd [S, H, I] codes with one scale per output row
 * sd [S*H] (quantise w_down viewed as [S*H, I]).  The shared experts' outputs
 * are summed, so their down weights form one matrix [H, n_sh*I_sh] (expert
 * j's [H, I_sh] in columns j*I_sh...) quantised per row: qsd [H, n_sh*I_sh],
 * ssd [H].  y_disp[row, o] = bf16(h_scale[row] * sd[slot*H+o] * sum_i
 * h8*qd); y_shared[t, o] = hs_scale[t] * ssd[o] * sum_i hs8*qsd in fp32.
 * inter % 16 == 0 and n_sh*I_sh % 16 == 0.
 * moe_expert_down_fp8_payload: moe_expert_down_fp8 whose routed outputs
 * leave as the E4M3 combine payload (section 2.3 halves the combine volume
 * too): each row's bf16 value (the y_disp of moe_expert_down_fp8) is cut into
 * blocks of MOE_PAYLOAD_BLOCK columns (the last one shorter when hidden is
 * not a multiple), each block quantised with its own fp32 scale as above:
 * y_disp8 [T*k, H] u8 codes, y_disp_scale [T*k, ceil(H/MOE_PAYLOAD_BLOCK)].
 * Per token the payload is k*H bytes plus k*ceil(H/128)*4 bytes of scales
 * (59,136 B at k=8, H=7168).  y_shared as moe_expert_down_fp8 (fp32, local).
 * moe_combine_fp8: moe_combine on that payload; an expert output element is
 * decode(code) * the scale of its block, in fp32.  hidden % 16 == 0.
 * moe_forward_fp8: route (bf16 router), moe_dispatch_fp8,
 * moe_expert_gate_up_fp8, the two intermediate quantisations,
 * moe_expert_down_fp8_payload, moe_combine_fp8, intermediates in a workspace
 * of moe_workspace_size_fp8() bytes.  Every expert matrix is E4M3, and so are
 * the dispatch and the combine payloads. */
#define MOE_PAYLOAD_BLOCK 128
MOE_API int moe_quantize_rows_fp8(int rows, int cols, const void* x, uint8_t* codes, float* scale, void* stream);
MOE_API int moe_dispatch_fp8(const moe_shape_t* shape, int T, const void* x, const int32_t* topk_idx,
                             const int32_t* replica_of, int32_t* slot_of, int32_t* counts, int32_t* block_counts,
                             int32_t* offsets, int32_t* perm, int32_t* inv_perm, uint8_t* x8, float* x_scale,
                             uint8_t* x_disp8, float* x_disp_scale, void* ws, size_t ws_bytes,
                             void* stream);
MOE_API int moe_expert_gate_up_fp8(const moe_shape_t* shape, int T, const uint8_t* x8, const float* x_scale,
                                   const uint8_t* x_disp8, const float* x_disp_scale, const int32_t* offsets,
                                   const uint8_t* qg, const float* sg, const uint8_t* qu, const float* su,
                                   const uint8_t* qsg, const float* ssg, const uint8_t* qsu, const float* ssu,
                                   void* h_disp, void* h_shared, int mode, void* stream);
MOE_API int moe_expert_down_fp8(const moe_shape_t* shape, int T, const uint8_t* h8, const float* h_scale,
                                const uint8_t* hs8, const float* hs_scale, const int32_t* offsets, const uint8_t* qd,
                                const float* sd, const uint8_t* qsd, const float* ssd, void* y_disp, float* y_shared,
                                int mode, void* stream);
MOE_API int moe_expert_down_fp8_payload(const moe_shape_t* shape, int T, const uint8_t* h8, const float* h_scale,
                                        const uint8_t* hs8, const float* hs_scale, const int32_t* offsets,
                                        const uint8_t* qd, const float* sd, const uint8_t* qsd, const float* ssd,
                                        uint8_t* y_disp8, float* y_disp_scale, float* y_shared, int mode,
                                        void* stream);
MOE_API int moe_combine_fp8(const moe_shape_t* shape, int T, const uint8_t* y_disp8, const float* y_disp_scale,
                            const int32_t* inv_perm, const float* topk_w, const float* y_shared, void* out,
                            void* stream);
MOE_API size_t moe_workspace_size_fp8(const moe_shape_t* shape, int T);
MOE_API int moe_forward_fp8(const moe_shape_t* shape, int T, const void* x, const void* w_router, const float* bias,
                            const int32_t* replica_of, const uint8_t* qg, const float* sg, const uint8_t* qu,
                            const float* su, const uint8_t* qd, const float* sd, const uint8_t* qsg,
                            const float* ssg, const uint8_t* qsu, const float* ssu, const uint8_t* qsd,
                            const float* ssd, void* out,
                            int32_t* topk_idx_out, float* topk_w_out, int32_t* counts_out, int32_t* block_counts_out,
                            int mode, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- steps 4-5: combine
 * Section 2.2 steps 4-5 (shared expert gate taken as 1):
 *   out[t,:] = bf16( sum_{j<k} topk_w[t,j] * y_disp[inv_perm[t*k+j], :] + y_shared[t,:] ),
 * fp32 accumulation in ascending j, then the shared term.  y_disp [T*k,H] bf16;
 * inv_perm [T*k]; topk_w [T,k] fp32; y_shared [T,H] fp32 or NULL; out [T,H] bf16. */
MOE_API int moe_combine(const moe_shape_t* shape, int T, const void* y_disp, const int32_t* inv_perm,
                const float* topk_w, const float* y_shared, void* out, void* stream);

/* ---------------------------------------------------------------- EP across GPUs
 * Section 2.1: EP rank g holds the slots of block g; section 2.2 steps 2 and 4:
 * the dispatch all-to-all sends a token's rows to the ranks holding its
 * experts, the combine all-to-all brings the expert outputs back (section 2.3:
 * 2 * k * hidden * 2 bytes per token).  The collectives themselves are the
 * caller's (NCCL, or torch.distributed over it); these calls do the
 * bookkeeping around them.  world = n_blocks ranks, spb = n_slots / world.
 *
 * moe_ep_plan (host only, no device memory):
 *   counts [n_slots+1]: this rank's dispatch counts (moe_dispatch);
 *   recv_counts [world*spb]: recv_counts[s*spb+j] = rows source rank s sends
 *     for local slot j (rank s's counts of this rank's slots, exchanged first);
 *   out: send_rows [world] (rows to each rank: the segment of its block in the
 *     dispatch buffer, in rank order), recv_rows [world] (rows from each source,
 *     received source-major, each source's rows in slot order),
 *   local_offsets [spb+2]: offsets of the local slots once regrouped
 *     slot-major (each slot's rows from source 0, 1, ...); [spb] = [spb+1] = R;
 *   slot_from_src [R] / src_from_slot [R] (either may be NULL): the
 *     source-major index of each slot-major row, and its inverse; rows_cap is
 *     their capacity; *rows_out = R, the rows this rank receives.
 *   Errors: MOE_ERR_INVALID_ARG (world != n_blocks, null, negative counts,
 *   R > rows_cap when a map is asked for), MOE_ERR_UNSUPPORTED (>= 2^31 rows).
 * moe_gather_rows: dst[i] = src[index[i]] for n_rows rows of row_bytes bytes
 *   (row_bytes % 16 == 0, src and dst 16-byte aligned, device pointers;
 *   index [n_rows] device int32, each in range of src: not checked), async on
 *   stream.  Regroups received rows slot-major (index = slot_from_src) and
 *   expert outputs back source-major (index = src_from_slot), for bf16 and
 *   E4M3 rows alike. */
MOE_API int moe_ep_plan(const moe_shape_t* shape, int world, const int32_t* counts, const int32_t* recv_counts,
                        int32_t* send_rows, int32_t* recv_rows, int32_t* local_offsets, int32_t* slot_from_src,
                        int32_t* src_from_slot, int32_t rows_cap, int32_t* rows_out);
MOE_API int moe_gather_rows(int n_rows, int row_bytes, const void* src, const int32_t* index, void* dst,
                            void* stream);

/* ---------------------------------------------------------------- whole layer
 * moe_route (from x), moe_dispatch, moe_expert_ffn, moe_combine on one stream
 * (7 kernel launches; capturable in a CUDA graph).  Intermediates live in the
 * workspace (moe_workspace_size() bytes).  Optional outputs (NULL to skip):
 * topk_idx_out [T,k], topk_w_out [T,k], counts_out [S+1], block_counts_out [B].
 * out [T,H] bf16. */
MOE_API size_t moe_workspace_size(const moe_shape_t* shape, int T);
MOE_API int moe_forward(const moe_shape_t* shape, int T, const void* x, const void* w_router, const float* bias,
                const int32_t* replica_of, const void* w_gate, const void* w_up, const void* w_down,
                const void* ws_gate, const void* ws_up, const void* ws_down, void* out, int32_t* topk_idx_out,
                float* topk_w_out, int32_t* counts_out, int32_t* block_counts_out, int mode, void* ws,
                size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
