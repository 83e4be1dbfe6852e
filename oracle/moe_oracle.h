/*
 * Plain fp64 CPU oracle of the DeepSeek-V3-style MoE layer forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares no source with
 * the CUDA library and must never sit on the product path.
 *
 * The method follows the blog post "专家并行(EP)" (expert parallelism):
 *   section 2.2 (a token's journey): router linear [7168,256] -> logits ->
 *     top-8 -> dispatch to the experts' owners -> per-expert FFN ->
 *     combine back -> output = sum_{i in top-8} softmax(logits)[i] *
 *     expert_output[i] + shared expert output;
 *   section 2.1: experts laid out in contiguous blocks, one per EP rank,
 *     shared experts replicated;
 *   section 6.2: per-expert arrival counts and per-rank load sums;
 *   section 6.3: redundant experts (256 + 8 slots, 33 per rank), a token may
 *     use any replica of its expert.
 * Readings where the post is silent (softmax over all experts without
 * renormalisation, SwiGLU form, shared gate = 1, tie rule, replica choice by
 * token parity, replica placement) are stated at each function.
 *
 * bf16 values are passed as their raw uint16 bit patterns; every arithmetic
 * step is in double precision.  All functions are single-threaded, pure
 * (no globals) and therefore safe to call from several threads at once.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t hidden;        /* H */
    int32_t inter;         /* I, routed expert SwiGLU width */
    int32_t n_experts;     /* E, logical routed experts */
    int32_t top_k;         /* k */
    int32_t n_shared;      /* shared experts */
    int32_t inter_shared;  /* I_sh */
    int32_t n_slots;       /* S = E or E + replicas */
    int32_t n_blocks;      /* EP blocks (ranks) */
} oracle_shape;

/* bf16 bit pattern -> double (exact). */
double oracle_bf16_to_double(uint16_t v);

/* logits[t,e] = sum_h x[t,h] * w_router[e,h] (+ bias[e]).  x [T,H], w_router [E,H]. */
void oracle_router_logits(const oracle_shape* s, int T, const uint16_t* x,
                          const uint16_t* w_router, const float* bias, double* logits);

/* Top-k by value (descending, equal values -> lower expert index first) and the
 * combine weight softmax(logits over all E)[idx], not renormalised. */
void oracle_topk_softmax(int T, int E, int k, const double* logits, int32_t* idx, double* weight);

/* Group-limited top-k (the summary section of the expert-parallelism post
 * names routing to an expert group first and to experts within it second as a
 * direction for larger expert counts).
 * Reading: the E experts form n_groups contiguous groups (the EP blocks); a
 * group's score is its largest logit; the topk_groups best groups are kept
 * (score descending, ties -> lower group); the top-k experts are then chosen
 * among the kept groups' experts only (same order and tie rule as
 * oracle_topk_softmax), and the combine weight is still softmax over all E. */
void oracle_topk_grouped(int T, int E, int k, int n_groups, int topk_groups, const double* logits,
                         int32_t* idx, double* weight);

/* Home slot of logical expert e (blocks keep their experts in order; with
 * replicas each block has trailing replica slots). */
int32_t oracle_home_slot(const oracle_shape* s, int32_t e);

/* slot_of[t*k+j]: replica of idx if the expert has one and t is odd, else home.
 * Returns the number of assignments with an expert id outside [0,E); they go
 * to slot S (the invalid bucket). */
int oracle_slot_map(const oracle_shape* s, int T, const int32_t* idx, const int32_t* replica_of,
                    int32_t* slot_of);

/* counts[S+1] (index S = invalid bucket) and per-block loads block_counts[n_blocks]. */
void oracle_histogram(const oracle_shape* s, int n_assign, const int32_t* slot_of, int32_t* counts,
                      int32_t* block_counts);

/* Counting-sort dispatch: offsets[S+2] exclusive prefix of counts (offsets[S+1] = T*k),
 * rows of a slot in ascending assignment order; perm[row] = a, inv_perm[a] = row;
 * x_disp[row] = x[a / k] (byte copy).  x_disp may be NULL. */
void oracle_dispatch(const oracle_shape* s, int T, const int32_t* slot_of, const int32_t* counts,
                     const uint16_t* x, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                     uint16_t* x_disp);

/* One SwiGLU FFN on one row: y = W_d (silu(W_g x) * (W_u x)).
 * w_gate/w_up [I,H] (row-major, nn.Linear), w_down [H,I]; y [H]. */
void oracle_swiglu_row(int H, int I, const uint16_t* x_row, const uint16_t* w_gate,
                       const uint16_t* w_up, const uint16_t* w_down, double* y);

/* Shared experts on one row: y = sum_j FFN_j(x) (shared gate taken as 1).
 * ws_* laid out [n_shared, I_sh, H] / [n_shared, H, I_sh]. */
void oracle_shared_row(const oracle_shape* s, const uint16_t* x_row, const uint16_t* ws_gate,
                       const uint16_t* ws_up, const uint16_t* ws_down, double* y);

/* Routed expert outputs of every dispatched row: y_disp[row] = FFN_{slot(row)}(x_disp[row]).
 * Routed weights slot-major [S,I,H], [S,I,H], [S,H,I]. */
void oracle_expert_ffn(const oracle_shape* s, int T, const int32_t* offsets, const uint16_t* x_disp,
                       const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                       double* y_disp);

/* out[t] = sum_{j<k} weight[t,j] * y_disp[inv_perm[t*k+j]] + y_shared[t]. */
void oracle_combine(const oracle_shape* s, int T, const double* y_disp, const int32_t* inv_perm,
                    const double* weight, const double* y_shared, double* out);

/* Whole layer.  Every output pointer may be NULL except out [T,H].
 * Returns the number of invalid expert ids met (0 on a well-formed input). */
int oracle_moe_forward(const oracle_shape* s, int T, const uint16_t* x, const uint16_t* w_router,
                       const float* bias, const int32_t* replica_of,
                       const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                       const uint16_t* ws_gate, const uint16_t* ws_up, const uint16_t* ws_down,
                       double* logits, int32_t* idx, double* weight, int32_t* slot_of,
                       int32_t* counts, int32_t* block_counts, int32_t* offsets, int32_t* perm,
                       int32_t* inv_perm, double* out);

/* One token's output from its routing: out = sum_j weight[j] * FFN(x; expert j's
 * weights at w_gate[j], w_up[j], w_down[j]) + shared.  For sampled checks at
 * full size, where only the experts a token uses are generated. */
void oracle_token_output(const oracle_shape* s, const uint16_t* x_row, int k,
                         const double* weight, const uint16_t* const* w_gate,
                         const uint16_t* const* w_up, const uint16_t* const* w_down,
                         const uint16_t* ws_gate, const uint16_t* ws_up, const uint16_t* ws_down,
                         double* out);

/* EPLB monitor and detection over a sliding window (section 6.2: per-expert
 * arrival rates over a recent window, per-rank load = sum over its experts,
 * rebalance when max/mean rank load exceeds a threshold such as 1.2).
 * Reading: the window is the last `window` batches (not a time span).
 * history [n_batches][S+1]: per-slot counts of each batch, oldest first.
 * slot_window[S+1] = sum of the last min(window, n_batches) rows;
 * block_load[B] = sum of slot_window over the block's slots;
 * expert_load[E] = slot_window of the expert's home slot plus that of its
 * replica slot (replica_of may be NULL);
 * ratio = max(block_load) * B / sum(block_load) (0 when the sum is 0);
 * trigger = max * B > threshold * sum, evaluated in double. */
void oracle_eplb_window(const oracle_shape* s, int n_batches, const int32_t* history, int window,
                        const int32_t* replica_of, double threshold, int64_t* slot_window,
                        int64_t* block_load, int64_t* expert_load, double* ratio, int* trigger);

/* ---- FP8 (section 2.3 of the post: FP8 communication halves the per-token
 * dispatch + combine bytes, 229 KB -> 115 KB).
 * E4M3 (OCP 8-bit floating point: 1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits; largest finite 448; code 0x7F/0xFF is NaN; no infinity).
 * Encoding rounds to nearest, ties to even, and saturates finite values
 * beyond 448 to +-448; NaN encodes as 0x7F. */
uint8_t oracle_e4m3_encode(float v);
double oracle_e4m3_decode(uint8_t code);

/* Per-row quantisation: scale[r] = amax(|row|) / 448 in fp32 (1 if the row is
 * all zero); codes[r][c] = e4m3(x[r][c] / scale[r]), the division in fp32.
 * Dequantised value = decode(code) * scale. */
void oracle_quantize_rows_e4m3(int rows, int cols, const uint16_t* x_bf16, uint8_t* codes, float* scale);

/* bf16 value nearest to v (ties to even), as a bit pattern.  The layer keeps
 * the SwiGLU intermediate h in bf16, so the FP8 down projection quantises the
 * bf16 h. */
uint16_t oracle_double_to_bf16(double v);

/* FP8 gate/up of one row: g_i = sx*sg[i] * sum_c qx_c*qg[i][c] (exact products
 * of decoded values in fp64), u likewise, h_i = silu(g_i)*u_i.  qg/qu [I,H]. */
void oracle_gate_up_row_fp8(int H, int I, const uint8_t* qx, float sx, const uint8_t* qg, const float* sg,
                            const uint8_t* qu, const float* su, double* h);

/* FP8 down projection of one row: y[o] = sh*sd[o] * sum_i qh_i*qd[o][i]
 * (decoded values), qh [K] codes of the intermediate with scale sh,
 * qd [H,K] codes with one scale per output row sd [H]. */
void oracle_down_row_fp8(int K, int H, const uint8_t* qh, float sh, const uint8_t* qd, const float* sd, double* y);

/* One routed expert on one token, all in FP8: oracle_gate_up_row_fp8, h
 * rounded to bf16 and quantised as one row (oracle_quantize_rows_e4m3), then
 * oracle_down_row_fp8.  qd [H,I] codes, sd [H]. */
void oracle_swiglu_row_fp8(int H, int I, const uint8_t* qx, float sx, const uint8_t* qg, const float* sg,
                           const uint8_t* qu, const float* su, const uint8_t* qd, const float* sd, double* y);

/* The shared experts on one token in FP8.  Their outputs are summed, so their
 * down matrices act as one matrix [H, n_sh*I_sh] (expert j's columns at
 * j*I_sh) applied to the concatenated intermediate [n_sh*I_sh]; that matrix
 * has one scale per output row (ssd [H]) and the concatenated intermediate
 * (bf16, as for a routed row) one scale per token.  qsg/qsu [n_sh,I_sh,H],
 * ssg/ssu [n_sh*I_sh], qsd [H, n_sh*I_sh]. */
void oracle_shared_row_fp8(const oracle_shape* s, const uint8_t* qx, float sx, const uint8_t* qsg, const float* ssg,
                           const uint8_t* qsu, const float* ssu, const uint8_t* qsd, const float* ssd, double* y);

/* Block quantisation: each row is cut into blocks of `block` columns (the
 * last one may be shorter) and each block is quantised as its own row by
 * oracle_quantize_rows_e4m3: scale[r][b] = amax(|block|) / 448 in fp32 (1 for
 * an all-zero block).  scale [rows, ceil(cols/block)]. */
void oracle_quantize_blocks_e4m3(int rows, int cols, int block, const uint16_t* x_bf16, uint8_t* codes,
                                 float* scale);

/* The E4M3 combine payload (section 2.3: FP8 communication halves the combine
 * bytes too).  An expert output row y (fp64) travels as its bf16 value (the
 * bf16 layer's payload) quantised in blocks of ORACLE_PAYLOAD_BLOCK columns;
 * y_deq = decode(code) * block scale, exact in fp64.  codes/scale may be NULL. */
#define ORACLE_PAYLOAD_BLOCK 128
void oracle_payload_e4m3(int rows, int cols, const double* y, double* y_deq, uint8_t* codes, float* scale);

/* Whole layer in FP8: routing as oracle_moe_forward (bf16 router), every
 * token quantised once per row (its k dispatched copies carry the same codes
 * and scale), routed experts by oracle_swiglu_row_fp8 (qg/qu [S,I,H] with
 * scales [S*I], qd [S,H,I] with [S*H]), their outputs carried back as the
 * E4M3 payload of oracle_payload_e4m3, shared experts by
 * oracle_shared_row_fp8 (local to the token, no payload), combine as
 * oracle_combine.  Returns the number of invalid expert ids. */
int oracle_moe_forward_fp8(const oracle_shape* s, int T, const uint16_t* x, const uint16_t* w_router,
                           const float* bias, const int32_t* replica_of, const uint8_t* qg, const float* sg,
                           const uint8_t* qu, const float* su, const uint8_t* qd, const float* sd,
                           const uint8_t* qsg, const float* ssg, const uint8_t* qsu, const float* ssu,
                           const uint8_t* qsd, const float* ssd, int32_t* idx, double* out);

/* oracle_moe_forward_fp8 that also returns the combine weights weight [T*k],
 * inv_perm [T*k] and the payload (y_codes [T*k, H] and y_scale [T*k,
 * ceil(H/ORACLE_PAYLOAD_BLOCK)], rows in dispatch order); any may be NULL. */
int oracle_moe_forward_fp8_payload(const oracle_shape* s, int T, const uint16_t* x, const uint16_t* w_router,
                                   const float* bias, const int32_t* replica_of, const uint8_t* qg, const float* sg,
                                   const uint8_t* qu, const float* su, const uint8_t* qd, const float* sd,
                                   const uint8_t* qsg, const float* ssg, const uint8_t* qsu, const float* ssu,
                                   const uint8_t* qsd, const float* ssd, int32_t* idx, double* out, double* weight,
                                   int32_t* inv_perm, uint8_t* y_codes, float* y_scale);

/* Replica placement for n_rep redundant slots from per-expert counts[E].
 * Hot list: the n_rep experts with the largest counts (ties -> lower id).
 * Each block initially carries the load of its experts, a hot expert's
 * count halved (half its tokens will use the replica).  For each hot expert
 * in order, the replica goes to the block with the smallest load among those
 * without a replica yet and other than its home block (ties -> lower block);
 * if only its home block is free, there.  The block's load grows by half the
 * expert's count and the replica takes that block's first free replica slot.
 * replica_of[E]: slot or -1.  Returns 0, or -1 if the shape has no room. */
int oracle_plan_replicas(const oracle_shape* s, const int32_t* counts, int n_rep,
                         int32_t* replica_of);

#ifdef __cplusplus
}
#endif
#endif
