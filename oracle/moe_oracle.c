/*
 * Plain fp64 CPU oracle of the DeepSeek-V3-style MoE layer forward pass.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  It shares no code
 * with the CUDA library.  Each function states the passage of the blog post
 * "专家并行(EP)" (expert parallelism) it follows, or the reading taken where
 * the post is silent.  No blocking, fusion or reordering: loops follow the
 * definitions in their plainest order.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no fast-math, so
 * x86-64 and aarch64 give identical results).
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

double oracle_bf16_to_double(uint16_t v) {
    /* bf16 is the upper half of an IEEE binary32. */
    uint32_t bits = ((uint32_t)v) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Section 2.2, step 1: "Router Linear: [7168, 256] -> logits: [1, 256]".
 * The router weight is stored [E, H] (one row per expert). */
void oracle_router_logits(const oracle_shape* s, int T, const uint16_t* x,
                          const uint16_t* w_router, const float* bias, double* logits) {
    const int H = s->hidden, E = s->n_experts;
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += oracle_bf16_to_double(x[(size_t)t * H + h]) *
                       oracle_bf16_to_double(w_router[(size_t)e * H + h]);
            if (bias) acc += (double)bias[e];
            logits[(size_t)t * E + e] = acc;
        }
    }
}

/* a ranks before b: larger value first, equal values -> lower index first. */
static int ranks_before(double va, int ia, double vb, int ib) {
    if (va > vb) return 1;
    if (va < vb) return 0;
    return ia < ib;
}

/* Section 2.2, step 1 ("Top-K: K=8") and step 5 ("output = sum softmax(logits[i]) x
 * expert_output[i], i in Top-8"): softmax is taken over all E logits and the
 * selected probabilities are used as they are (reading: not renormalised).
 * Selection: k passes, each taking the best remaining expert. */
void oracle_topk_softmax(int T, int E, int k, const double* logits, int32_t* idx, double* weight) {
    char* taken = (char*)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const double* l = logits + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
            }
            taken[best] = 1;
            idx[(size_t)t * k + j] = best;
        }
        double mx = l[0];
        for (int e = 1; e < E; ++e)
            if (l[e] > mx) mx = l[e];
        double denom = 0.0;
        for (int e = 0; e < E; ++e) denom += exp(l[e] - mx);
        if (weight)
            for (int j = 0; j < k; ++j)
                weight[(size_t)t * k + j] = exp(l[idx[(size_t)t * k + j]] - mx) / denom;
    }
    free(taken);
}

/* Summary section of the post: route by expert group first, then by expert.
 * Readings are stated in the header. */
void oracle_topk_grouped(int T, int E, int k, int n_groups, int topk_groups, const double* logits,
                         int32_t* idx, double* weight) {
    const int gs = E / n_groups;
    char* taken = (char*)malloc((size_t)E);
    char* group_kept = (char*)malloc((size_t)n_groups);
    double* gscore = (double*)malloc((size_t)n_groups * sizeof(double));
    for (int t = 0; t < T; ++t) {
        const double* l = logits + (size_t)t * E;
        for (int g = 0; g < n_groups; ++g) {
            double best = l[g * gs];
            for (int e = g * gs + 1; e < (g + 1) * gs; ++e)
                if (l[e] > best) best = l[e];
            gscore[g] = best;
            group_kept[g] = 0;
        }
        for (int r = 0; r < topk_groups; ++r) {
            int bg = -1;
            for (int g = 0; g < n_groups; ++g) {
                if (group_kept[g]) continue;
                if (bg < 0 || ranks_before(gscore[g], g, gscore[bg], bg)) bg = g;
            }
            group_kept[bg] = 1;
        }
        for (int e = 0; e < E; ++e) taken[e] = !group_kept[e / gs];
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
            }
            taken[best] = 1;
            idx[(size_t)t * k + j] = best;
        }
        double mx = l[0];
        for (int e = 1; e < E; ++e)
            if (l[e] > mx) mx = l[e];
        double denom = 0.0;
        for (int e = 0; e < E; ++e) denom += exp(l[e] - mx);
        if (weight)
            for (int j = 0; j < k; ++j)
                weight[(size_t)t * k + j] = exp(l[idx[(size_t)t * k + j]] - mx) / denom;
    }
    free(taken);
    free(group_kept);
    free(gscore);
}

/* Section 2.1: "each GPU holds a contiguous 1/N of the experts" (GPU g: experts
 * 32g..32g+31).  Section 6.3: with 8 redundant experts each of the 8 GPUs holds
 * 33.  Reading: a block keeps its own experts first, in order, and its replica
 * slots after them. */
int32_t oracle_home_slot(const oracle_shape* s, int32_t e) {
    const int epb = s->n_experts / s->n_blocks;
    const int spb = s->n_slots / s->n_blocks;
    return (e / epb) * spb + (e % epb);
}

/* Section 6.3: the router may send a token to any replica of its expert.
 * Reading: a deterministic choice, even tokens -> home slot, odd tokens -> replica. */
int oracle_slot_map(const oracle_shape* s, int T, const int32_t* idx, const int32_t* replica_of,
                    int32_t* slot_of) {
    const int k = s->top_k, E = s->n_experts;
    int invalid = 0;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            const int32_t e = idx[(size_t)t * k + j];
            int32_t slot;
            if (e < 0 || e >= E) {
                slot = s->n_slots;
                ++invalid;
            } else if (replica_of && replica_of[e] >= 0 && (t % 2) == 1) {
                slot = replica_of[e];
            } else {
                slot = oracle_home_slot(s, e);
            }
            slot_of[(size_t)t * k + j] = slot;
        }
    }
    return invalid;
}

/* Section 6.2, "monitor": tokens arriving at each expert, and each GPU's load =
 * the sum over its experts.  Here for one batch: counts per slot, block sums. */
void oracle_histogram(const oracle_shape* s, int n_assign, const int32_t* slot_of, int32_t* counts,
                      int32_t* block_counts) {
    const int S = s->n_slots;
    const int spb = S / s->n_blocks;
    for (int i = 0; i <= S; ++i) counts[i] = 0;
    for (int a = 0; a < n_assign; ++a) counts[slot_of[a]] += 1;
    if (block_counts) {
        for (int b = 0; b < s->n_blocks; ++b) {
            int32_t sum = 0;
            for (int i = b * spb; i < (b + 1) * spb; ++i) sum += counts[i];
            block_counts[b] = sum;
        }
    }
}

/* Section 2.2, step 2 (dispatch): each token's hidden state goes to the owner of
 * every expert it selected.  On one device this is a counting sort of the T*k
 * assignments by slot into one buffer whose slot segments sit in block order
 * (the per-rank send segments).  Reading: within a slot, ascending assignment
 * index a = t*k + j. */
void oracle_dispatch(const oracle_shape* s, int T, const int32_t* slot_of, const int32_t* counts,
                     const uint16_t* x, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                     uint16_t* x_disp) {
    const int S = s->n_slots, k = s->top_k, H = s->hidden;
    const int n = T * k;
    offsets[0] = 0;
    for (int i = 0; i <= S; ++i) offsets[i + 1] = offsets[i] + counts[i];
    int32_t* fill = (int32_t*)calloc((size_t)S + 1, sizeof(int32_t));
    for (int a = 0; a < n; ++a) {
        const int32_t slot = slot_of[a];
        const int32_t row = offsets[slot] + fill[slot];
        fill[slot] += 1;
        perm[row] = a;
        inv_perm[a] = row;
    }
    free(fill);
    if (x_disp)
        for (int row = 0; row < n; ++row)
            memcpy(x_disp + (size_t)row * H, x + (size_t)(perm[row] / k) * H,
                   (size_t)H * sizeof(uint16_t));
}

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* Section 2.2, step 3: each expert's FFN on its rows.  The post names the
 * gate/up projections [7168, 2048]; reading: SwiGLU, h = silu(x W_g^T) * (x W_u^T),
 * y = h W_d^T with W_d [7168 out, 2048 in]. */
void oracle_swiglu_row(int H, int I, const uint16_t* x_row, const uint16_t* w_gate,
                       const uint16_t* w_up, const uint16_t* w_down, double* y) {
    double* h = (double*)malloc((size_t)I * sizeof(double));
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            const double xv = oracle_bf16_to_double(x_row[c]);
            g += xv * oracle_bf16_to_double(w_gate[(size_t)i * H + c]);
            u += xv * oracle_bf16_to_double(w_up[(size_t)i * H + c]);
        }
        h[i] = silu(g) * u;
    }
    for (int o = 0; o < H; ++o) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += h[i] * oracle_bf16_to_double(w_down[(size_t)o * I + i]);
        y[o] = acc;
    }
    free(h);
}

/* Section 2.1: shared experts see every token and are not split across ranks.
 * Section 2.2, step 5 adds "shared_expert_output x shared_expert_gate"; reading:
 * the gate is 1 and the shared experts' outputs are summed. */
void oracle_shared_row(const oracle_shape* s, const uint16_t* x_row, const uint16_t* ws_gate,
                       const uint16_t* ws_up, const uint16_t* ws_down, double* y) {
    const int H = s->hidden, I = s->inter_shared;
    double* tmp = (double*)malloc((size_t)H * sizeof(double));
    for (int o = 0; o < H; ++o) y[o] = 0.0;
    for (int j = 0; j < s->n_shared; ++j) {
        oracle_swiglu_row(H, I, x_row, ws_gate + (size_t)j * I * H, ws_up + (size_t)j * I * H,
                          ws_down + (size_t)j * H * I, tmp);
        for (int o = 0; o < H; ++o) y[o] += tmp[o];
    }
    free(tmp);
}

void oracle_expert_ffn(const oracle_shape* s, int T, const int32_t* offsets, const uint16_t* x_disp,
                       const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                       double* y_disp) {
    const int S = s->n_slots, H = s->hidden, I = s->inter;
    (void)T;
    for (int slot = 0; slot < S; ++slot) {
        for (int row = offsets[slot]; row < offsets[slot + 1]; ++row) {
            oracle_swiglu_row(H, I, x_disp + (size_t)row * H, w_gate + (size_t)slot * I * H,
                              w_up + (size_t)slot * I * H, w_down + (size_t)slot * H * I,
                              y_disp + (size_t)row * H);
        }
    }
}

/* Section 2.2, steps 4-5: expert outputs come back to the token (combine) and
 * output = sum_{i in top-k} softmax(logits)[i] * expert_output[i] + shared. */
void oracle_combine(const oracle_shape* s, int T, const double* y_disp, const int32_t* inv_perm,
                    const double* weight, const double* y_shared, double* out) {
    const int H = s->hidden, k = s->top_k;
    for (int t = 0; t < T; ++t) {
        for (int o = 0; o < H; ++o) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                const int32_t row = inv_perm[(size_t)t * k + j];
                acc += weight[(size_t)t * k + j] * y_disp[(size_t)row * H + o];
            }
            out[(size_t)t * H + o] = acc + y_shared[(size_t)t * H + o];
        }
    }
}

int oracle_moe_forward(const oracle_shape* s, int T, const uint16_t* x, const uint16_t* w_router,
                       const float* bias, const int32_t* replica_of,
                       const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                       const uint16_t* ws_gate, const uint16_t* ws_up, const uint16_t* ws_down,
                       double* logits, int32_t* idx, double* weight, int32_t* slot_of,
                       int32_t* counts, int32_t* block_counts, int32_t* offsets, int32_t* perm,
                       int32_t* inv_perm, double* out) {
    const int H = s->hidden, E = s->n_experts, k = s->top_k, S = s->n_slots;
    const size_t n = (size_t)T * k;
    double* l_ = logits ? logits : (double*)malloc((size_t)T * E * sizeof(double));
    int32_t* idx_ = idx ? idx : (int32_t*)malloc(n * sizeof(int32_t));
    double* w_ = weight ? weight : (double*)malloc(n * sizeof(double));
    int32_t* so_ = slot_of ? slot_of : (int32_t*)malloc(n * sizeof(int32_t));
    int32_t* c_ = counts ? counts : (int32_t*)malloc(((size_t)S + 1) * sizeof(int32_t));
    int32_t* off_ = offsets ? offsets : (int32_t*)malloc(((size_t)S + 2) * sizeof(int32_t));
    int32_t* p_ = perm ? perm : (int32_t*)malloc(n * sizeof(int32_t));
    int32_t* ip_ = inv_perm ? inv_perm : (int32_t*)malloc(n * sizeof(int32_t));
    uint16_t* xd = (uint16_t*)malloc(n * H * sizeof(uint16_t));
    double* yd = (double*)calloc(n * H, sizeof(double));
    double* ysh = (double*)malloc((size_t)T * H * sizeof(double));

    oracle_router_logits(s, T, x, w_router, bias, l_);
    oracle_topk_softmax(T, E, k, l_, idx_, w_);
    const int invalid = oracle_slot_map(s, T, idx_, replica_of, so_);
    oracle_histogram(s, (int)n, so_, c_, block_counts);
    oracle_dispatch(s, T, so_, c_, x, off_, p_, ip_, xd);
    oracle_expert_ffn(s, T, off_, xd, w_gate, w_up, w_down, yd);
    for (int t = 0; t < T; ++t)
        oracle_shared_row(s, x + (size_t)t * H, ws_gate, ws_up, ws_down, ysh + (size_t)t * H);
    oracle_combine(s, T, yd, ip_, w_, ysh, out);

    if (!logits) free(l_);
    if (!idx) free(idx_);
    if (!weight) free(w_);
    if (!slot_of) free(so_);
    if (!counts) free(c_);
    if (!offsets) free(off_);
    if (!perm) free(p_);
    if (!inv_perm) free(ip_);
    free(xd);
    free(yd);
    free(ysh);
    return invalid;
}

void oracle_token_output(const oracle_shape* s, const uint16_t* x_row, int k,
                         const double* weight, const uint16_t* const* w_gate,
                         const uint16_t* const* w_up, const uint16_t* const* w_down,
                         const uint16_t* ws_gate, const uint16_t* ws_up, const uint16_t* ws_down,
                         double* out) {
    const int H = s->hidden, I = s->inter;
    double* y = (double*)malloc((size_t)H * sizeof(double));
    double* ysh = (double*)malloc((size_t)H * sizeof(double));
    for (int o = 0; o < H; ++o) out[o] = 0.0;
    for (int j = 0; j < k; ++j) {
        oracle_swiglu_row(H, I, x_row, w_gate[j], w_up[j], w_down[j], y);
        for (int o = 0; o < H; ++o) out[o] += weight[j] * y[o];
    }
    oracle_shared_row(s, x_row, ws_gate, ws_up, ws_down, ysh);
    for (int o = 0; o < H; ++o) out[o] += ysh[o];
    free(y);
    free(ysh);
}

/* Section 6.2 ("migrate": copy the overloaded GPU's hottest experts to an idle
 * GPU) and 6.3 (8 redundant experts, one more slot per GPU).  The post picks
 * targets by load only; the deterministic rule is stated in the header. */
int oracle_plan_replicas(const oracle_shape* s, const int32_t* counts, int n_rep,
                         int32_t* replica_of) {
    const int E = s->n_experts, B = s->n_blocks;
    const int epb = E / B, spb = s->n_slots / B;
    const int rep_per_block = spb - epb;
    for (int e = 0; e < E; ++e) replica_of[e] = -1;
    if (n_rep <= 0) return 0;
    if (rep_per_block <= 0 || n_rep > E || n_rep > rep_per_block * B) return -1;

    /* hot list: largest counts first, equal counts -> lower id */
    int32_t* hot = (int32_t*)malloc((size_t)n_rep * sizeof(int32_t));
    char* chosen = (char*)calloc((size_t)E, 1);
    for (int r = 0; r < n_rep; ++r) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (chosen[e]) continue;
            if (best < 0 || counts[e] > counts[best]) best = e;
        }
        chosen[best] = 1;
        hot[r] = best;
    }
    /* loads in half-token units: 2*count, a hot expert counted once (halved) */
    int64_t* load2 = (int64_t*)calloc((size_t)B, sizeof(int64_t));
    int* used = (int*)calloc((size_t)B, sizeof(int));
    for (int e = 0; e < E; ++e) load2[e / epb] += chosen[e] ? (int64_t)counts[e] : 2 * (int64_t)counts[e];
    int rc = 0;
    for (int r = 0; r < n_rep; ++r) {
        const int e = hot[r], home = e / epb;
        int target = -1;
        for (int b = 0; b < B; ++b) {
            if (b == home || used[b] >= rep_per_block) continue;
            if (target < 0 || load2[b] < load2[target]) target = b;
        }
        if (target < 0 && used[home] < rep_per_block) target = home;
        if (target < 0) { rc = -1; break; }
        replica_of[e] = target * spb + epb + used[target];
        used[target] += 1;
        load2[target] += counts[e];
    }
    free(hot);
    free(chosen);
    free(load2);
    free(used);
    return rc;
}

/* Section 6.2, monitor (arrival counts over a recent window, per-rank sums) and
 * detect (max/mean rank load against a threshold).  Readings in the header. */
void oracle_eplb_window(const oracle_shape* s, int n_batches, const int32_t* history, int window,
                        const int32_t* replica_of, double threshold, int64_t* slot_window,
                        int64_t* block_load, int64_t* expert_load, double* ratio, int* trigger) {
    const int S = s->n_slots, B = s->n_blocks, E = s->n_experts;
    const int spb = S / B;
    const int first = n_batches > window ? n_batches - window : 0;
    for (int i = 0; i <= S; ++i) {
        int64_t acc = 0;
        for (int b = first; b < n_batches; ++b) acc += history[(size_t)b * (S + 1) + i];
        slot_window[i] = acc;
    }
    int64_t mx = 0, total = 0;
    for (int b = 0; b < B; ++b) {
        int64_t acc = 0;
        for (int i = b * spb; i < (b + 1) * spb; ++i) acc += slot_window[i];
        block_load[b] = acc;
        total += acc;
        if (acc > mx) mx = acc;
    }
    for (int e = 0; e < E; ++e) {
        int64_t acc = slot_window[oracle_home_slot(s, e)];
        if (replica_of && replica_of[e] >= 0) acc += slot_window[replica_of[e]];
        expert_load[e] = acc;
    }
    *ratio = total > 0 ? (double)mx * (double)B / (double)total : 0.0;
    *trigger = (double)mx * (double)B > threshold * (double)total;
}

/* ---- FP8.  Section 2.3: FP8 communication halves the dispatch + combine
 * volume.  Format: OCP 8-bit floating point E4M3 (definition in the header). */
uint8_t oracle_e4m3_encode(float v) {
    if (isnan(v)) return 0x7F;
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7E;  /* saturate */
    if (a < ldexp(1.0, -6)) {
        /* subnormal grid: multiples of 2^-9; rounding up to 8 * 2^-9 gives the
         * smallest normal, whose code is 8 as well */
        const double m = rint(a * ldexp(1.0, 9)); /* default mode: nearest, ties to even */
        return sign | (uint8_t)m;
    }
    int ex;
    frexp(a, &ex);              /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;             /* a in [2^e, 2^(e+1)) */
    double m = rint((a * ldexp(1.0, -e) - 1.0) * 8.0);
    if (m == 8.0) {
        m = 0.0;
        e += 1;
    }
    return sign | (uint8_t)(((e + 7) << 3) | (int)m);
}

double oracle_e4m3_decode(uint8_t code) {
    const int e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return (code & 0x80) ? -mag : mag;
}

void oracle_quantize_rows_e4m3(int rows, int cols, const uint16_t* x_bf16, uint8_t* codes, float* scale) {
    for (int r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int c = 0; c < cols; ++c) {
            const float v = fabsf((float)oracle_bf16_to_double(x_bf16[(size_t)r * cols + c]));
            if (v > amax) amax = v;
        }
        const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
        scale[r] = s;
        for (int c = 0; c < cols; ++c)
            codes[(size_t)r * cols + c] = oracle_e4m3_encode((float)oracle_bf16_to_double(x_bf16[(size_t)r * cols + c]) / s);
    }
}

void oracle_quantize_blocks_e4m3(int rows, int cols, int block, const uint16_t* x_bf16, uint8_t* codes,
                                 float* scale) {
    const int nb = (cols + block - 1) / block;
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < nb; ++b) {
            const int c0 = b * block;
            const int w = cols - c0 < block ? cols - c0 : block;
            oracle_quantize_rows_e4m3(1, w, x_bf16 + (size_t)r * cols + c0, codes + (size_t)r * cols + c0,
                                      scale + (size_t)r * nb + b);
        }
}

void oracle_payload_e4m3(int rows, int cols, const double* y, double* y_deq, uint8_t* codes, float* scale) {
    const int nb = (cols + ORACLE_PAYLOAD_BLOCK - 1) / ORACLE_PAYLOAD_BLOCK;
    uint16_t* yb = (uint16_t*)malloc((size_t)cols * sizeof(uint16_t));
    uint8_t* q = (uint8_t*)malloc((size_t)cols);
    float* sc = (float*)malloc((size_t)nb * sizeof(float));
    for (int r = 0; r < rows; ++r) {
        const double* yr = y + (size_t)r * cols;
        for (int c = 0; c < cols; ++c) yb[c] = oracle_double_to_bf16(yr[c]);
        oracle_quantize_blocks_e4m3(1, cols, ORACLE_PAYLOAD_BLOCK, yb, q, sc);
        for (int c = 0; c < cols; ++c)
            y_deq[(size_t)r * cols + c] = oracle_e4m3_decode(q[c]) * (double)sc[c / ORACLE_PAYLOAD_BLOCK];
        if (codes) memcpy(codes + (size_t)r * cols, q, (size_t)cols);
        if (scale) memcpy(scale + (size_t)r * nb, sc, (size_t)nb * sizeof(float));
    }
    free(yb); free(q); free(sc);
}

uint16_t oracle_double_to_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    int ex;
    frexp(fabs(v), &ex);         /* |v| in [2^(ex-1), 2^ex) */
    if (ex < -125) ex = -125;    /* below 2^-126 the grid stays at 2^-133 (subnormals) */
    const double step = ldexp(1.0, ex - 8);   /* 8 significant bits */
    const double r = rint(v / step) * step;   /* nearest multiple, ties to even */
    const float f = (float)r;                 /* exact (or +-inf past the largest bf16) */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(bits >> 16);
}

/* Every code's value, from oracle_e4m3_decode: the row products below look
 * codes up here instead of decoding each element again (same values). */
static void e4m3_table(double* tab) {
    for (int c = 0; c < 256; ++c) tab[c] = oracle_e4m3_decode((uint8_t)c);
}

void oracle_gate_up_row_fp8(int H, int I, const uint8_t* qx, float sx, const uint8_t* qg, const float* sg,
                            const uint8_t* qu, const float* su, double* h) {
    double dec[256];
    e4m3_table(dec);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            const double xv = dec[qx[c]];
            g += xv * dec[qg[(size_t)i * H + c]];
            u += xv * dec[qu[(size_t)i * H + c]];
        }
        g *= (double)sx * (double)sg[i];
        u *= (double)sx * (double)su[i];
        h[i] = silu(g) * u;
    }
}

void oracle_down_row_fp8(int K, int H, const uint8_t* qh, float sh, const uint8_t* qd, const float* sd, double* y) {
    double dec[256];
    e4m3_table(dec);
    for (int o = 0; o < H; ++o) {
        double acc = 0.0;
        for (int i = 0; i < K; ++i) acc += dec[qh[i]] * dec[qd[(size_t)o * K + i]];
        y[o] = acc * (double)sh * (double)sd[o];
    }
}

/* h (fp64) -> bf16 -> one E4M3 row with its scale */
static void quantize_h_row(int K, const double* h, uint16_t* hb, uint8_t* qh, float* sh) {
    for (int i = 0; i < K; ++i) hb[i] = oracle_double_to_bf16(h[i]);
    oracle_quantize_rows_e4m3(1, K, hb, qh, sh);
}

void oracle_swiglu_row_fp8(int H, int I, const uint8_t* qx, float sx, const uint8_t* qg, const float* sg,
                           const uint8_t* qu, const float* su, const uint8_t* qd, const float* sd, double* y) {
    double* h = (double*)malloc((size_t)I * sizeof(double));
    uint16_t* hb = (uint16_t*)malloc((size_t)I * sizeof(uint16_t));
    uint8_t* qh = (uint8_t*)malloc((size_t)I);
    float sh;
    oracle_gate_up_row_fp8(H, I, qx, sx, qg, sg, qu, su, h);
    quantize_h_row(I, h, hb, qh, &sh);
    oracle_down_row_fp8(I, H, qh, sh, qd, sd, y);
    free(h); free(hb); free(qh);
}

void oracle_shared_row_fp8(const oracle_shape* s, const uint8_t* qx, float sx, const uint8_t* qsg, const float* ssg,
                           const uint8_t* qsu, const float* ssu, const uint8_t* qsd, const float* ssd, double* y) {
    const int H = s->hidden, Is = s->inter_shared, n_sh = s->n_shared;
    const int K = n_sh * Is;
    if (n_sh == 0) {
        for (int o = 0; o < H; ++o) y[o] = 0.0;
        return;
    }
    double* h = (double*)malloc((size_t)K * sizeof(double));
    uint16_t* hb = (uint16_t*)malloc((size_t)K * sizeof(uint16_t));
    uint8_t* qh = (uint8_t*)malloc((size_t)K);
    float sh;
    for (int j = 0; j < n_sh; ++j)
        oracle_gate_up_row_fp8(H, Is, qx, sx, qsg + (size_t)j * Is * H, ssg + (size_t)j * Is, qsu + (size_t)j * Is * H,
                               ssu + (size_t)j * Is, h + (size_t)j * Is);
    quantize_h_row(K, h, hb, qh, &sh);
    oracle_down_row_fp8(K, H, qh, sh, qsd, ssd, y);
    free(h); free(hb); free(qh);
}

int oracle_moe_forward_fp8(const oracle_shape* s, int T, const uint16_t* x, const uint16_t* w_router,
                           const float* bias, const int32_t* replica_of, const uint8_t* qg, const float* sg,
                           const uint8_t* qu, const float* su, const uint8_t* qd, const float* sd,
                           const uint8_t* qsg, const float* ssg, const uint8_t* qsu, const float* ssu,
                           const uint8_t* qsd, const float* ssd, int32_t* idx, double* out) {
    return oracle_moe_forward_fp8_payload(s, T, x, w_router, bias, replica_of, qg, sg, qu, su, qd, sd, qsg, ssg, qsu,
                                          ssu, qsd, ssd, idx, out, NULL, NULL, NULL, NULL);
}

int oracle_moe_forward_fp8_payload(const oracle_shape* s, int T, const uint16_t* x, const uint16_t* w_router,
                                   const float* bias, const int32_t* replica_of, const uint8_t* qg, const float* sg,
                                   const uint8_t* qu, const float* su, const uint8_t* qd, const float* sd,
                                   const uint8_t* qsg, const float* ssg, const uint8_t* qsu, const float* ssu,
                                   const uint8_t* qsd, const float* ssd, int32_t* idx, double* out, double* weight,
                                   int32_t* inv_perm, uint8_t* y_codes, float* y_scale) {
    const int H = s->hidden, E = s->n_experts, k = s->top_k, S = s->n_slots, I = s->inter;
    const size_t n = (size_t)T * k;
    double* logits = (double*)malloc((size_t)T * E * sizeof(double));
    double* w = (double*)malloc(n * sizeof(double));
    int32_t* so = (int32_t*)malloc(n * sizeof(int32_t));
    int32_t* cnt = (int32_t*)malloc(((size_t)S + 1) * sizeof(int32_t));
    int32_t* off = (int32_t*)malloc(((size_t)S + 2) * sizeof(int32_t));
    int32_t* perm = (int32_t*)malloc(n * sizeof(int32_t));
    int32_t* inv = (int32_t*)malloc(n * sizeof(int32_t));
    uint8_t* qx = (uint8_t*)malloc((size_t)T * H);
    float* sx = (float*)malloc((size_t)T * sizeof(float));
    double* yd = (double*)calloc(n * H, sizeof(double));
    double* ysh = (double*)calloc((size_t)T * H, sizeof(double));

    oracle_router_logits(s, T, x, w_router, bias, logits);
    oracle_topk_softmax(T, E, k, logits, idx, w);
    const int invalid = oracle_slot_map(s, T, idx, replica_of, so);
    oracle_histogram(s, (int)n, so, cnt, NULL);
    oracle_dispatch(s, T, so, cnt, NULL, off, perm, inv, NULL);
    oracle_quantize_rows_e4m3(T, H, x, qx, sx);
    for (int slot = 0; slot < S; ++slot) {
        for (int row = off[slot]; row < off[slot + 1]; ++row) {
            const int t = perm[row] / k;
            oracle_swiglu_row_fp8(H, I, qx + (size_t)t * H, sx[t], qg + (size_t)slot * I * H, sg + (size_t)slot * I,
                                  qu + (size_t)slot * I * H, su + (size_t)slot * I, qd + (size_t)slot * H * I,
                                  sd + (size_t)slot * H, yd + (size_t)row * H);
        }
    }
    oracle_payload_e4m3((int)n, H, yd, yd, y_codes, y_scale);  /* in place: each row read before it is written */
    for (int t = 0; t < T; ++t)
        oracle_shared_row_fp8(s, qx + (size_t)t * H, sx[t], qsg, ssg, qsu, ssu, qsd, ssd, ysh + (size_t)t * H);
    oracle_combine(s, T, yd, inv, w, ysh, out);
    if (weight) memcpy(weight, w, n * sizeof(double));
    if (inv_perm) memcpy(inv_perm, inv, n * sizeof(int32_t));
    free(logits); free(w); free(so); free(cnt); free(off); free(perm); free(inv);
    free(qx); free(sx); free(yd); free(ysh);
    return invalid;
}
