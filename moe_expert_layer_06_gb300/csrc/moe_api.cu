// C ABI of libmoe (declared in include/moe.h): argument validation, TMA
// tensor maps, workspace carving and kernel launches.  No allocation, no
// host synchronisation except in moe_check_status().
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include "moe.h"
#include "kernels.h"

namespace moe {

// ------------------------------------------------------------------ errors
static thread_local char g_err[512] = "";

static int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

static int cuda_fail(cudaError_t e, const char* what) {
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MOE_CUDA(call, what)                          \
    do {                                              \
        cudaError_t e_ = (call);                      \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

// ------------------------------------------------------------------ device status
__device__ unsigned int g_status_word;
// Shared by every host thread: the wait bound (set by moe_set_wait_limit_ns) and
// per-device caches filled on first use (a racing first use fills the same value).
static std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};
static constexpr int kMaxDevices = 64;
static std::atomic<unsigned int*> g_status_ptr[kMaxDevices];
static std::atomic<int> g_num_sms[kMaxDevices];

static int current_device(int* dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (*dev < 0 || *dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device ordinal %d too large", *dev);
    return MOE_OK;
}

static int device_status(DevStatus* st) {
    int dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    unsigned int* word = g_status_ptr[dev].load(std::memory_order_acquire);
    if (!word) {
        void* p = nullptr;
        MOE_CUDA(cudaGetSymbolAddress(&p, g_status_word), "cudaGetSymbolAddress(status)");
        word = static_cast<unsigned int*>(p);
        g_status_ptr[dev].store(word, std::memory_order_release);
    }
    st->word = word;
    st->limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    return MOE_OK;
}

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int n = g_num_sms[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_num_sms[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// ------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once (thread-safe static initialisation); null without a driver.
static EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

int make_tmap_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1,
                 uint64_t stride2, uint32_t box0, uint32_t box1, uint32_t box2, bool fp8) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1, stride2};
    const cuuint32_t box[3] = {box0, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return MOE_OK;
}

// weight stack [n][rows][K] -> dims {K, rows, n}, box {64, 128, 1}
static int tmap_weights(CUtensorMap* m, const void* p, int n, int rows, int K) {
    return make_tmap_3d(m, p, (uint64_t)K, (uint64_t)rows, (uint64_t)n, (uint64_t)K * 2, (uint64_t)K * rows * 2,
                        64, 128, 1);
}

// activations [rows][K] -> dims {K, 1, rows}; four maps with boxes {64, 1, 16 << j}
static int tmap_rows(CUtensorMap* m, const void* p, int rows, int K) {
    for (int j = 0; j < 4; ++j) {
        const int rc = make_tmap_3d(m + j, p, (uint64_t)K, 1, (uint64_t)rows, (uint64_t)K * 2, (uint64_t)K * 2,
                                    64, 1, 16u << j);
        if (rc) return rc;
    }
    return MOE_OK;
}

// shared intermediate [T][n_sh][I_sh] -> dims {I_sh, n_sh, T}; boxes {64, 1, 16 << j}
static int tmap_hsh(CUtensorMap* m, const void* p, int T, int n_sh, int I_sh) {
    for (int j = 0; j < 4; ++j) {
        const int rc = make_tmap_3d(m + j, p, (uint64_t)I_sh, (uint64_t)n_sh, (uint64_t)T, (uint64_t)I_sh * 2,
                                    (uint64_t)I_sh * n_sh * 2, 64, 1, 16u << j);
        if (rc) return rc;
    }
    return MOE_OK;
}

// FP8 (one byte per element, 128-element rows per chunk)
static int tmap_weights_f8(CUtensorMap* m, const void* p, int n, int rows, int K) {
    return make_tmap_3d(m, p, (uint64_t)K, (uint64_t)rows, (uint64_t)n, (uint64_t)K, (uint64_t)K * rows, 128, 128, 1,
                        true);
}

static int tmap_rows_f8(CUtensorMap* m, const void* p, int rows, int K) {
    for (int j = 0; j < 4; ++j) {
        const int rc = make_tmap_3d(m + j, p, (uint64_t)K, 1, (uint64_t)rows, (uint64_t)K, (uint64_t)K, 128, 1,
                                    16u << j, true);
        if (rc) return rc;
    }
    return MOE_OK;
}

// ------------------------------------------------------------------ validation
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_shape(const moe_shape_t* s, int T) {
    if (!s) return fail(MOE_ERR_INVALID_ARG, "shape is NULL");
    if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d < 0", T);
    if (s->hidden <= 0 || s->inter <= 0 || s->n_experts <= 0 || s->top_k <= 0 || s->n_slots <= 0 ||
        s->n_blocks <= 0 || s->n_shared < 0)
        return fail(MOE_ERR_INVALID_ARG, "non-positive shape field");
    if (s->n_shared > 0 && s->inter_shared <= 0) return fail(MOE_ERR_INVALID_ARG, "inter_shared <= 0");
    if (s->top_k > s->n_experts) return fail(MOE_ERR_INVALID_ARG, "top_k %d > n_experts %d", s->top_k, s->n_experts);
    if (s->top_k > 32) return fail(MOE_ERR_INVALID_ARG, "top_k %d > 32", s->top_k);
    if (s->hidden % 8 || s->inter % 8 || (s->n_shared > 0 && s->inter_shared % 8))
        return fail(MOE_ERR_INVALID_ARG, "hidden, inter and inter_shared must be multiples of 8");
    if (s->n_experts % s->n_blocks || s->n_slots % s->n_blocks || s->n_slots < s->n_experts)
        return fail(MOE_ERR_INVALID_ARG, "n_experts and n_slots must divide into n_blocks, n_slots >= n_experts");
    const int max_slots = std::min(gemm_max_slots(), dispatch_max_slots());
    if (s->n_experts > max_slots) return fail(MOE_ERR_UNSUPPORTED, "n_experts %d > %d", s->n_experts, max_slots);
    if (s->n_slots > max_slots) return fail(MOE_ERR_UNSUPPORTED, "n_slots %d > %d", s->n_slots, max_slots);
    if ((int64_t)T * s->top_k > INT32_MAX / 2) return fail(MOE_ERR_UNSUPPORTED, "T*k too large");
    return MOE_OK;
}

#define NEED(ptr, name)                                                                    \
    do {                                                                                   \
        if (!(ptr)) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", name);                  \
        if (!aligned16(ptr)) return fail(MOE_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
    } while (0)

#define NEED4(ptr, name)                                                                  \
    do {                                                                                  \
        if (!(ptr)) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", name);                 \
        if (reinterpret_cast<uintptr_t>(ptr) & 3u)                                        \
            return fail(MOE_ERR_INVALID_ARG, "%s is not 4-byte aligned", name);           \
    } while (0)

static inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// mid: the E4M3 down GEMM, which takes kMidBN rows when slots average few rows
static int ffn_bn(const moe_shape_t* s, int T, int mode, bool mid) {
    if (mode == MOE_FFN_DECODE) return 32;
    if (mode == MOE_FFN_PREFILL) return kPrefillBN;
    if (T <= 32) return 32;
    const bool few_rows = (long)T * s->top_k <= (long)kMidMaxRowsPerSlot * s->n_slots;
    return (mid && few_rows) ? kMidBN : kPrefillBN;
}

static inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

namespace {
thread_local bool t_pdl = true;
}
bool pdl_enabled() { return t_pdl; }
PdlScope::PdlScope(long assignments) : saved(t_pdl) { t_pdl = assignments <= kPdlMaxAssignments; }
PdlScope::~PdlScope() { t_pdl = saved; }

// ------------------------------------------------------------------ routing
struct RoutePlan {
    int bn, ksplit, kc_split, tiles;
};

static RoutePlan route_plan(const moe_shape_t* s, int T, int sms) {
    RoutePlan p;
    p.bn = T <= 32 ? 32 : kPrefillBN;
    const int kc = (s->hidden + 63) / 64;
    p.tiles = ((s->n_experts + 127) / 128) * ((T + p.bn - 1) / p.bn);
    const int want = std::max(1, (sms + p.tiles - 1) / std::max(1, p.tiles));
    p.kc_split = std::max(1, (kc + want - 1) / want);
    p.ksplit = (kc + p.kc_split - 1) / p.kc_split;
    return p;
}

static RoutePlan route_plan(const moe_shape_t* s, int T) { return route_plan(s, T, num_sms()); }

static size_t route_partials_bytes(const moe_shape_t* s, int T, int sms) {
    const RoutePlan p = route_plan(s, T, sms);
    return (size_t)p.ksplit * T * s->n_experts * sizeof(float);
}

// The K-split partials of the largest need among batches of 1..T tokens, so a
// workspace sized for the largest batch serves every smaller one.  The need
// grows with T between token-chunk boundaries and drops after one (more tiles,
// fewer K splits), so the maximum is at T or at a boundary below it; a boundary
// whose tiles fill the SMs has one K split and cannot exceed the need at T.
static size_t route_ws(const moe_shape_t* s, int T) {
    if (T == 0) return 0;
    const int sms = num_sms();
    const long row_tiles = (s->n_experts + 127) / 128;
    size_t need = route_partials_bytes(s, T, sms);
    for (long j = 1; j * kPrefillBN < T && j * row_tiles < sms; ++j)
        need = std::max(need, route_partials_bytes(s, (int)(j * kPrefillBN), sms));
    return align256(need);
}

static int route_impl(const moe_shape_t* s, int T, int n_groups, int topk_groups, const void* x,
                      const void* w_router, const float* bias, const float* logits_in, float* logits_out,
                      int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, cudaStream_t stream) {
    NEED4(topk_idx, "topk_idx");
    NEED4(topk_w, "topk_w");
    if (logits_out) NEED4(logits_out, "logits_out");
    if (logits_in) {
        if (bias) return fail(MOE_ERR_INVALID_ARG, "bias must be NULL when logits_in is given");
        NEED4(logits_in, "logits_in");
    } else {
        NEED(x, "x");
        NEED(w_router, "w_router");
        if (bias) NEED4(bias, "bias");
        const size_t need = route_ws(s, T);
        if (!ws || ws_bytes < need) return fail(MOE_ERR_WORKSPACE, "route workspace %zu < %zu bytes", ws_bytes, need);
        if (!aligned16(ws)) return fail(MOE_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
    }
    DevStatus st;
    int rc = device_status(&st);
    if (rc) return rc;
    if (logits_in) {
        MOE_CUDA(launch_topk(logits_in, 1, nullptr, T, s->n_experts, s->top_k, logits_out, topk_idx, topk_w,
                             n_groups, topk_groups, st, stream),
                 "topk launch");
        return MOE_OK;
    }
    const RoutePlan p = route_plan(s, T);
    GemmArgs g;
    memset(&g, 0, sizeof g);
    if ((rc = tmap_weights(&g.a0, w_router, 1, s->n_experts, s->hidden))) return rc;
    if ((rc = tmap_rows(g.b, x, T, s->hidden))) return rc;
    g.a1 = g.a0;
    g.sa0 = g.sa1 = g.a0;
    for (int j = 0; j < 4; ++j) g.sb[j] = g.b[j];
    g.T = T;
    g.m_routed = s->n_experts;
    g.kc_routed = (s->hidden + 63) / 64;
    g.ksplit = p.ksplit;
    g.kc_split = p.kc_split;
    g.out = ws;
    g.out_ld = s->n_experts;
    g.st = st;
    const int items = p.tiles * p.ksplit;
    MOE_CUDA(launch_gemm(kRouter, p.bn, g, std::min(items, num_sms()), stream), "router gemm launch");
    MOE_CUDA(launch_topk(static_cast<const float*>(ws), p.ksplit, bias, T, s->n_experts, s->top_k, logits_out,
                         topk_idx, topk_w, n_groups, topk_groups, st, stream),
             "topk launch");
    return MOE_OK;
}

// ------------------------------------------------------------------ dispatch
static size_t dispatch_ws(const moe_shape_t* s, int T) {
    return align256(index_workspace_bytes(T * s->top_k, s->n_slots));
}

// The index pass: one CTA, or in chunks for a large batch with a full
// permutation (perm given), the per-chunk histograms in the workspace.
static int index_impl(const moe_shape_t* s, int T, const int32_t* topk_idx, const int32_t* replica_of,
                      int32_t* slot_of, int32_t* counts, int32_t* block_counts, int32_t* offsets, int32_t* perm,
                      int32_t* inv_perm, void* ws, size_t ws_bytes, cudaStream_t stream) {
    const bool chunked = perm && index_chunks(T * s->top_k) > 0;
    if (chunked) {
        const size_t need = dispatch_ws(s, T);
        if (!ws || ws_bytes < need) return fail(MOE_ERR_WORKSPACE, "dispatch workspace %zu < %zu bytes", ws_bytes, need);
        if (!aligned16(ws)) return fail(MOE_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
    }
    DevStatus st;
    int rc = device_status(&st);
    if (rc) return rc;
    DispatchArgs d;
    d.T = T;
    d.k = s->top_k;
    d.E = s->n_experts;
    d.S = s->n_slots;
    d.n_blocks = s->n_blocks;
    d.hidden = s->hidden;
    d.topk_idx = topk_idx;
    d.replica_of = replica_of;
    d.slot_of = slot_of;
    d.counts = counts;
    d.block_counts = block_counts;
    d.offsets = offsets;
    d.perm = perm;
    d.inv_perm = inv_perm;
    d.st = st;
    if (chunked)
        MOE_CUDA(launch_index_chunked(d, static_cast<int32_t*>(ws), stream), "chunked index pass launch");
    else
        MOE_CUDA(launch_index_pass(d, stream), "index pass launch");
    return MOE_OK;
}

// ------------------------------------------------------------------ expert FFN
static int gate_up_impl(const moe_shape_t* s, int T, const void* x, const void* x_disp, const int32_t* offsets,
                        const void* w_gate, const void* w_up, const void* ws_gate, const void* ws_up, void* h_disp,
                        void* h_shared, int mode, cudaStream_t stream) {
    NEED(x_disp, "x_disp");
    NEED4(offsets, "offsets");
    NEED(w_gate, "w_gate");
    NEED(w_up, "w_up");
    NEED(h_disp, "h_disp");
    const int n_sh = s->n_shared;
    if (n_sh > 0) {
        NEED(x, "x");
        NEED(ws_gate, "ws_gate");
        NEED(ws_up, "ws_up");
        NEED(h_shared, "h_shared");
    }
    DevStatus st;
    int rc = device_status(&st);
    if (rc) return rc;
    const int n = T * s->top_k;
    const int bn = ffn_bn(s, T, mode, false);
    GemmArgs g;
    memset(&g, 0, sizeof g);
    if ((rc = tmap_weights(&g.a0, w_gate, s->n_slots, s->inter, s->hidden))) return rc;
    if ((rc = tmap_weights(&g.a1, w_up, s->n_slots, s->inter, s->hidden))) return rc;
    if ((rc = tmap_rows(g.b, x_disp, n, s->hidden))) return rc;
    if (n_sh > 0) {
        if ((rc = tmap_weights(&g.sa0, ws_gate, n_sh, s->inter_shared, s->hidden))) return rc;
        if ((rc = tmap_weights(&g.sa1, ws_up, n_sh, s->inter_shared, s->hidden))) return rc;
        if ((rc = tmap_rows(g.sb, x, T, s->hidden))) return rc;
    } else {
        g.sa0 = g.a0;
        g.sa1 = g.a1;
        for (int j = 0; j < 4; ++j) g.sb[j] = g.b[j];
    }
    g.offsets = offsets;
    g.n_slots = s->n_slots;
    g.T = T;
    g.m_routed = s->inter;
    g.kc_routed = (s->hidden + 63) / 64;
    g.n_shared = n_sh;
    g.m_shared = s->inter_shared;
    g.kc_shared = (s->hidden + 63) / 64;
    g.kc_per_sh = 1;
    g.out = h_disp;
    g.out_ld = s->inter;
    g.out_sh = h_shared;
    g.out_sh_ld = n_sh * s->inter_shared;
    g.sh_col_stride = s->inter_shared;
    g.st = st;
    MOE_CUDA(launch_gemm(kGateUp, bn, g, num_sms(), stream), "gate/up gemm launch");
    return MOE_OK;
}

static int gate_up_fp8_impl(const moe_shape_t* s, int T, const void* x8, const float* x_scale, const void* x_disp8,
                            const float* x_disp_scale, const int32_t* offsets, const void* qg, const float* sg,
                            const void* qu, const float* su, const void* qsg, const float* ssg, const void* qsu,
                            const float* ssu, void* h_disp, void* h_shared, int mode, cudaStream_t stream) {
    if (s->hidden % 16) return fail(MOE_ERR_INVALID_ARG, "FP8 rows need hidden %% 16 == 0");
    NEED(x_disp8, "x_disp8");
    NEED4(x_disp_scale, "x_disp_scale");
    NEED4(offsets, "offsets");
    NEED(qg, "qg");
    NEED(qu, "qu");
    NEED4(sg, "sg");
    NEED4(su, "su");
    NEED(h_disp, "h_disp");
    const int n_sh = s->n_shared;
    if (n_sh > 0) {
        NEED(x8, "x8");
        NEED4(x_scale, "x_scale");
        NEED(qsg, "qsg");
        NEED(qsu, "qsu");
        NEED4(ssg, "ssg");
        NEED4(ssu, "ssu");
        NEED(h_shared, "h_shared");
    }
    DevStatus st;
    int rc = device_status(&st);
    if (rc) return rc;
    const int n = T * s->top_k;
    const int bn = ffn_bn(s, T, mode, false);
    GemmArgs g;
    memset(&g, 0, sizeof g);
    if ((rc = tmap_weights_f8(&g.a0, qg, s->n_slots, s->inter, s->hidden))) return rc;
    if ((rc = tmap_weights_f8(&g.a1, qu, s->n_slots, s->inter, s->hidden))) return rc;
    if ((rc = tmap_rows_f8(g.b, x_disp8, n, s->hidden))) return rc;
    if (n_sh > 0) {
        if ((rc = tmap_weights_f8(&g.sa0, qsg, n_sh, s->inter_shared, s->hidden))) return rc;
        if ((rc = tmap_weights_f8(&g.sa1, qsu, n_sh, s->inter_shared, s->hidden))) return rc;
        if ((rc = tmap_rows_f8(g.sb, x8, T, s->hidden))) return rc;
    } else {
        g.sa0 = g.a0;
        g.sa1 = g.a1;
        for (int j = 0; j < 4; ++j) g.sb[j] = g.b[j];
    }
    g.offsets = offsets;
    g.n_slots = s->n_slots;
    g.T = T;
    g.m_routed = s->inter;
    g.kc_routed = (s->hidden + 127) / 128;
    g.n_shared = n_sh;
    g.m_shared = s->inter_shared;
    g.kc_shared = (s->hidden + 127) / 128;
    g.kc_per_sh = 1;
    g.out = h_disp;
    g.out_ld = s->inter;
    g.out_sh = h_shared;
    g.out_sh_ld = n_sh * s->inter_shared;
    g.sh_col_stride = s->inter_shared;
    g.a0_scale = sg;
    g.a1_scale = su;
    g.sa0_scale = ssg;
    g.sa1_scale = ssu;
    g.b_scale = x_disp_scale;
    g.sb_scale = x_scale;
    g.st = st;
    MOE_CUDA(launch_gemm(kGateUpF8, bn, g, num_sms(), stream), "FP8 gate/up gemm launch");
    return MOE_OK;
}

static int down_impl(const moe_shape_t* s, int T, const void* h_disp, const void* h_shared, const int32_t* offsets,
                     const void* w_down, const void* ws_down, void* y_disp, float* y_shared, int mode,
                     cudaStream_t stream) {
    NEED(h_disp, "h_disp");
    NEED4(offsets, "offsets");
    NEED(w_down, "w_down");
    NEED(y_disp, "y_disp");
    const int n_sh = s->n_shared;
    if (n_sh > 0) {
        NEED(h_shared, "h_shared");
        NEED(ws_down, "ws_down");
        NEED(y_shared, "y_shared");
    }
    DevStatus st;
    int rc = device_status(&st);
    if (rc) return rc;
    const int n = T * s->top_k;
    const int bn = ffn_bn(s, T, mode, false);
    GemmArgs g;
    memset(&g, 0, sizeof g);
    if ((rc = tmap_weights(&g.a0, w_down, s->n_slots, s->hidden, s->inter))) return rc;
    if ((rc = tmap_rows(g.b, h_disp, n, s->inter))) return rc;
    g.a1 = g.a0;
    if (n_sh > 0) {
        if ((rc = tmap_weights(&g.sa0, ws_down, n_sh, s->hidden, s->inter_shared))) return rc;
        if ((rc = tmap_hsh(g.sb, h_shared, T, n_sh, s->inter_shared))) return rc;
    } else {
        g.sa0 = g.a0;
        for (int j = 0; j < 4; ++j) g.sb[j] = g.b[j];
    }
    g.sa1 = g.sa0;
    g.offsets = offsets;
    g.n_slots = s->n_slots;
    g.T = T;
    g.m_routed = s->hidden;
    g.kc_routed = (s->inter + 63) / 64;
    g.n_shared = n_sh;
    g.m_shared = s->hidden;
    g.kc_per_sh = n_sh > 0 ? (s->inter_shared + 63) / 64 : 1;
    g.kc_shared = n_sh * g.kc_per_sh;
    g.out = y_disp;
    g.out_ld = s->hidden;
    g.out_sh = y_shared;
    g.out_sh_ld = s->hidden;
    g.st = st;
    MOE_CUDA(launch_gemm(kDown, bn, g, num_sms(), stream), "down gemm launch");
    return MOE_OK;
}

// y8 != null: the routed outputs leave as the E4M3 combine payload (y8 codes,
// y8_scale block scales) instead of bf16 y_disp.
static int down_fp8_impl(const moe_shape_t* s, int T, const void* h8, const float* h_scale, const void* hs8,
                         const float* hs_scale, const int32_t* offsets, const void* qd, const float* sd,
                         const void* qsd, const float* ssd, void* y_disp, float* y_shared, int mode,
                         cudaStream_t stream, uint8_t* y8 = nullptr, float* y8_scale = nullptr) {
    const int n_sh = s->n_shared;
    const int Ks = n_sh * s->inter_shared;  // K of the concatenated shared down matrix
    if (s->inter % 16 || Ks % 16)
        return fail(MOE_ERR_INVALID_ARG, "FP8 down needs inter %% 16 == 0 and n_shared*inter_shared %% 16 == 0");
    NEED(h8, "h8");
    NEED4(h_scale, "h_scale");
    NEED4(offsets, "offsets");
    NEED(qd, "qd");
    NEED4(sd, "sd");
    if (y8) {
        NEED(y8, "y_disp8");
        NEED4(y8_scale, "y_disp_scale");
    } else {
        NEED(y_disp, "y_disp");
    }
    if (n_sh > 0) {
        NEED(hs8, "hs8");
        NEED4(hs_scale, "hs_scale");
        NEED(qsd, "qsd");
        NEED4(ssd, "ssd");
        NEED4(y_shared, "y_shared");
    }
    DevStatus st;
    int rc = device_status(&st);
    if (rc) return rc;
    const int n = T * s->top_k;
    const int bn = ffn_bn(s, T, mode, true);
    GemmArgs g;
    memset(&g, 0, sizeof g);
    if ((rc = tmap_weights_f8(&g.a0, qd, s->n_slots, s->hidden, s->inter))) return rc;
    if ((rc = tmap_rows_f8(g.b, h8, n, s->inter))) return rc;
    g.a1 = g.a0;
    if (n_sh > 0) {
        if ((rc = tmap_weights_f8(&g.sa0, qsd, 1, s->hidden, Ks))) return rc;
        if ((rc = tmap_rows_f8(g.sb, hs8, T, Ks))) return rc;
    } else {
        g.sa0 = g.a0;
        for (int j = 0; j < 4; ++j) g.sb[j] = g.b[j];
    }
    g.sa1 = g.sa0;
    g.offsets = offsets;
    g.n_slots = s->n_slots;
    g.T = T;
    g.m_routed = s->hidden;
    g.kc_routed = (s->inter + 127) / 128;
    g.n_shared = n_sh;
    g.m_shared = s->hidden;
    g.kc_shared = (Ks + 127) / 128;
    g.kc_per_sh = 1;
    g.out = y_disp;
    g.out_ld = s->hidden;
    g.out_sh = y_shared;
    g.out_sh_ld = s->hidden;
    g.a0_scale = sd;
    g.sa0_scale = ssd;
    g.b_scale = h_scale;
    g.sb_scale = hs_scale;
    g.out8 = y8;
    g.out8_scale = y8_scale;
    g.n_blk = (s->hidden + kPayloadBlock - 1) / kPayloadBlock;
    g.st = st;
    MOE_CUDA(launch_gemm(y8 ? kDownF8Q : kDownF8, bn, g, num_sms(), stream), "FP8 down gemm launch");
    return MOE_OK;
}

static size_t ffn_ws(const moe_shape_t* s, int T) {
    const size_t n = (size_t)T * s->top_k;
    return align256(n * s->inter * 2) + align256((size_t)T * s->n_shared * s->inter_shared * 2);
}

// ------------------------------------------------------------------ forward workspace carving
struct FwdLayout {
    size_t route, idx, w, slot_of, perm, inv_perm, counts, blocks, offsets, x_disp, ffn, y_disp, y_sh, dispatch, total;
};

// with_y_disp = false: no bf16 expert-output buffer (the E4M3 forward carries
// its own payload buffers instead)
static FwdLayout fwd_layout(const moe_shape_t* s, int T, bool with_y_disp = true) {
    FwdLayout L;
    const size_t n = (size_t)T * s->top_k;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += align256(bytes);
        return o;
    };
    L.route = take(route_ws(s, T));
    L.idx = take(n * 4);
    L.w = take(n * 4);
    L.slot_of = take(n * 4);
    L.perm = take(n * 4);
    L.inv_perm = take(n * 4);
    L.counts = take((size_t)(s->n_slots + 1) * 4);
    L.blocks = take((size_t)s->n_blocks * 4);
    L.offsets = take((size_t)(s->n_slots + 2) * 4);
    L.x_disp = take(n * s->hidden * 2);
    L.ffn = take(ffn_ws(s, T));
    L.y_disp = take(with_y_disp ? n * s->hidden * 2 : 0);
    L.y_sh = take((size_t)T * s->hidden * 4);
    L.dispatch = take(dispatch_ws(s, T));
    L.total = off;
    return L;
}

// FP8 forward: the bf16 layout plus the quantised tokens, their dispatched copies and the
// quantised intermediates (routed rows, shared rows)
struct FwdLayoutF8 {
    FwdLayout base;
    size_t x8, x_scale, x_disp8, x_disp_scale, h8, h_scale, hs8, hs_scale, y8, y_scale, total;
};

static FwdLayoutF8 fwd_layout_f8(const moe_shape_t* s, int T) {
    FwdLayoutF8 L;
    L.base = fwd_layout(s, T, false);
    const size_t n = (size_t)T * s->top_k;
    size_t off = L.base.total;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += align256(bytes);
        return o;
    };
    L.x8 = take((size_t)T * s->hidden);
    L.x_scale = take((size_t)T * 4);
    L.x_disp8 = take(n * s->hidden);
    L.x_disp_scale = take(n * 4);
    L.h8 = take(n * s->inter);
    L.h_scale = take(n * 4);
    L.hs8 = take((size_t)T * s->n_shared * s->inter_shared);
    L.hs_scale = take((size_t)T * 4);
    L.y8 = take(n * s->hidden);
    L.y_scale = take(n * (size_t)((s->hidden + kPayloadBlock - 1) / kPayloadBlock) * 4);
    L.total = off;
    return L;
}

// ------------------------------------------------------------------ host EPLB plan
static int plan_replicas_host(const moe_shape_t* s, const int32_t* counts, int n_rep, int32_t* replica_of) {
    const int E = s->n_experts, B = s->n_blocks;
    const int epb = E / B, spb = s->n_slots / B, free_per_block = spb - epb;
    for (int e = 0; e < E; ++e) replica_of[e] = -1;
    if (n_rep == 0) return MOE_OK;
    if (n_rep < 0 || n_rep > E || free_per_block <= 0 || n_rep > free_per_block * B)
        return fail(MOE_ERR_INVALID_ARG, "n_rep %d does not fit %d free slots per block", n_rep, free_per_block);
    std::vector<int> order(E);
    for (int e = 0; e < E; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return counts[a] > counts[b]; });
    std::vector<char> hot(E, 0);
    for (int r = 0; r < n_rep; ++r) hot[order[r]] = 1;
    // loads in half-token units so that halving stays exact
    std::vector<long long> load(B, 0);
    for (int e = 0; e < E; ++e) load[e / epb] += hot[e] ? (long long)counts[e] : 2LL * counts[e];
    std::vector<int> used(B, 0);
    for (int r = 0; r < n_rep; ++r) {
        const int e = order[r], home = e / epb;
        int best = -1;
        for (int b = 0; b < B; ++b) {
            if (b == home || used[b] >= free_per_block) continue;
            if (best < 0 || load[b] < load[best]) best = b;
        }
        if (best < 0 && used[home] < free_per_block) best = home;
        if (best < 0) return fail(MOE_ERR_INVALID_ARG, "no free replica slot for expert %d", e);
        replica_of[e] = best * spb + epb + used[best];
        used[best] += 1;
        load[best] += counts[e];
    }
    return MOE_OK;
}

// ------------------------------------------------------------------ failure-path probe
__global__ void expire_wait_kernel(DevStatus st) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
        // phase 0 never completes: nothing arrives on this barrier
        if (!mbar_wait(smem_u32(&bar), 0, st.limit_ns)) raise_status(st, kStatusWaitTimeout);
    }
}

int api_fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int api_check_shape(const moe_shape_t* shape, int T) { return check_shape(shape, T); }

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_last_error_string(void) { return g_err; }

int moe_abi_version(void) { return 1; }

int moe_set_wait_limit_ns(uint64_t ns) {
    if (ns == 0) return fail(MOE_ERR_INVALID_ARG, "wait limit must be > 0");
    g_wait_limit_ns.store(ns, std::memory_order_relaxed);
    return MOE_OK;
}

int moe_check_status(void* stream) {
    MOE_CUDA(cudaStreamSynchronize(as_stream(stream)), "cudaStreamSynchronize");
    unsigned int v = 0;
    MOE_CUDA(cudaMemcpyFromSymbol(&v, g_status_word, sizeof v), "read status");
    if (v == 0) return MOE_OK;
    const unsigned int zero = 0;
    MOE_CUDA(cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero), "clear status");
    if (v & kStatusWaitTimeout) return fail(MOE_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait expired (status 0x%x)", v);
    if (v & kStatusInvalidExpert)
        return fail(MOE_ERR_DEVICE_STATUS, "expert id outside [0, n_experts) or bad replica slot (status 0x%x)", v);
    return fail(MOE_ERR_DEVICE_STATUS, "device status 0x%x", v);
}

int moe_debug_expire_wait(void* stream) {
    DevStatus st;
    int rc = device_status(&st);
    if (rc) return rc;
    expire_wait_kernel<<<1, 32, 0, as_stream(stream)>>>(st);
    MOE_CUDA(cudaGetLastError(), "expire-wait launch");
    return MOE_OK;
}

size_t moe_route_workspace_size(const moe_shape_t* shape, int T) {
    if (check_shape(shape, T)) return 0;
    return route_ws(shape, T);
}

int moe_route(const moe_shape_t* shape, int T, const void* x, const void* w_router, const float* bias,
              const float* logits_in, float* logits_out, int32_t* topk_idx, float* topk_w, void* ws,
              size_t ws_bytes, void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (T == 0) return MOE_OK;
    return route_impl(shape, T, 0, 0, x, w_router, bias, logits_in, logits_out, topk_idx, topk_w, ws, ws_bytes,
                      as_stream(stream));
}

int moe_route_grouped(const moe_shape_t* shape, int T, int n_groups, int topk_groups, const void* x,
                      const void* w_router, const float* bias, const float* logits_in, float* logits_out,
                      int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (n_groups < 1 || n_groups > 32 || shape->n_experts % n_groups)
        return fail(MOE_ERR_INVALID_ARG, "n_groups %d must divide n_experts and be in [1, 32]", n_groups);
    if (topk_groups < 1 || topk_groups > n_groups)
        return fail(MOE_ERR_INVALID_ARG, "topk_groups %d not in [1, n_groups]", topk_groups);
    if ((int64_t)topk_groups * (shape->n_experts / n_groups) < shape->top_k)
        return fail(MOE_ERR_INVALID_ARG, "top_k %d exceeds the experts of %d groups", shape->top_k, topk_groups);
    if (T == 0) return MOE_OK;
    return route_impl(shape, T, n_groups, topk_groups, x, w_router, bias, logits_in, logits_out, topk_idx, topk_w,
                      ws, ws_bytes, as_stream(stream));
}

int moe_expert_histogram(const moe_shape_t* shape, int T, const int32_t* topk_idx, const int32_t* replica_of,
                         int32_t* counts, int32_t* block_counts, void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    NEED4(counts, "counts");
    if (T > 0) NEED4(topk_idx, "topk_idx");
    if (T == 0) {
        MOE_CUDA(cudaMemsetAsync(counts, 0, (size_t)(shape->n_slots + 1) * 4, as_stream(stream)), "memset counts");
        if (block_counts)
            MOE_CUDA(cudaMemsetAsync(block_counts, 0, (size_t)shape->n_blocks * 4, as_stream(stream)),
                     "memset block_counts");
        return MOE_OK;
    }
    if (replica_of) NEED4(replica_of, "replica_of");
    if (block_counts) NEED4(block_counts, "block_counts");
    return index_impl(shape, T, topk_idx, replica_of, nullptr, counts, block_counts, nullptr, nullptr, nullptr,
                      nullptr, 0, as_stream(stream));
}

double moe_eplb_imbalance(const int32_t* host_block_counts, int n_blocks) {
    if (!host_block_counts || n_blocks <= 0) return 0.0;
    long long sum = 0;
    int mx = 0;
    for (int b = 0; b < n_blocks; ++b) {
        sum += host_block_counts[b];
        mx = std::max(mx, (int)host_block_counts[b]);
    }
    if (sum == 0) return 0.0;
    return (double)mx * n_blocks / (double)sum;
}

int moe_eplb_plan_replicas(const moe_shape_t* shape, const int32_t* host_expert_counts, int n_rep,
                           int32_t* host_replica_of) {
    int rc = check_shape(shape, 0);
    if (rc) return rc;
    if (!host_expert_counts || !host_replica_of) return fail(MOE_ERR_INVALID_ARG, "NULL host array");
    return plan_replicas_host(shape, host_expert_counts, n_rep, host_replica_of);
}

size_t moe_dispatch_workspace_size(const moe_shape_t* shape, int T) {
    if (check_shape(shape, T)) return 0;
    return dispatch_ws(shape, T);
}

int moe_dispatch(const moe_shape_t* shape, int T, const void* x, const int32_t* topk_idx, const int32_t* replica_of,
                 int32_t* slot_of, int32_t* counts, int32_t* block_counts, int32_t* offsets, int32_t* perm,
                 int32_t* inv_perm, void* x_disp, void* ws, size_t ws_bytes, void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    NEED4(counts, "counts");
    NEED4(offsets, "offsets");
    if (T == 0) {
        cudaStream_t st = as_stream(stream);
        MOE_CUDA(cudaMemsetAsync(counts, 0, (size_t)(shape->n_slots + 1) * 4, st), "memset counts");
        MOE_CUDA(cudaMemsetAsync(offsets, 0, (size_t)(shape->n_slots + 2) * 4, st), "memset offsets");
        if (block_counts) MOE_CUDA(cudaMemsetAsync(block_counts, 0, (size_t)shape->n_blocks * 4, st), "memset blocks");
        return MOE_OK;
    }
    NEED(x, "x");
    NEED4(topk_idx, "topk_idx");
    NEED4(slot_of, "slot_of");
    NEED4(perm, "perm");
    NEED4(inv_perm, "inv_perm");
    NEED(x_disp, "x_disp");
    if (replica_of) NEED4(replica_of, "replica_of");
    if ((rc = index_impl(shape, T, topk_idx, replica_of, slot_of, counts, block_counts, offsets, perm, inv_perm, ws,
                         ws_bytes, as_stream(stream))))
        return rc;
    MOE_CUDA(launch_scatter_rows(static_cast<const uint16_t*>(x), perm, T * shape->top_k, shape->top_k,
                                 shape->hidden, static_cast<uint16_t*>(x_disp), as_stream(stream)),
             "scatter launch");
    return MOE_OK;
}

int moe_expert_gate_up(const moe_shape_t* shape, int T, const void* x, const void* x_disp, const int32_t* offsets,
                       const void* w_gate, const void* w_up, const void* ws_gate, const void* ws_up, void* h_disp,
                       void* h_shared, int mode, void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (mode < MOE_FFN_AUTO || mode > MOE_FFN_PREFILL) return fail(MOE_ERR_INVALID_ARG, "bad mode %d", mode);
    if (T == 0) return MOE_OK;
    return gate_up_impl(shape, T, x, x_disp, offsets, w_gate, w_up, ws_gate, ws_up, h_disp, h_shared, mode,
                        as_stream(stream));
}

int moe_expert_down(const moe_shape_t* shape, int T, const void* h_disp, const void* h_shared,
                    const int32_t* offsets, const void* w_down, const void* ws_down, void* y_disp, float* y_shared,
                    int mode, void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (mode < MOE_FFN_AUTO || mode > MOE_FFN_PREFILL) return fail(MOE_ERR_INVALID_ARG, "bad mode %d", mode);
    if (T == 0) return MOE_OK;
    return down_impl(shape, T, h_disp, h_shared, offsets, w_down, ws_down, y_disp, y_shared, mode,
                     as_stream(stream));
}

size_t moe_ffn_workspace_size(const moe_shape_t* shape, int T) {
    if (check_shape(shape, T)) return 0;
    return ffn_ws(shape, T);
}

int moe_expert_ffn(const moe_shape_t* shape, int T, const void* x, const void* x_disp, const int32_t* offsets,
                   const void* w_gate, const void* w_up, const void* w_down, const void* ws_gate, const void* ws_up,
                   const void* ws_down, void* y_disp, float* y_shared, int mode, void* ws, size_t ws_bytes,
                   void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (mode < MOE_FFN_AUTO || mode > MOE_FFN_PREFILL) return fail(MOE_ERR_INVALID_ARG, "bad mode %d", mode);
    if (T == 0) return MOE_OK;
    const size_t need = ffn_ws(shape, T);
    if (!ws || ws_bytes < need) return fail(MOE_ERR_WORKSPACE, "ffn workspace %zu < %zu bytes", ws_bytes, need);
    if (!aligned16(ws)) return fail(MOE_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
    uint8_t* base = static_cast<uint8_t*>(ws);
    void* h_disp = base;
    void* h_sh = shape->n_shared > 0 ? base + align256((size_t)T * shape->top_k * shape->inter * 2) : nullptr;
    if ((rc = gate_up_impl(shape, T, x, x_disp, offsets, w_gate, w_up, ws_gate, ws_up, h_disp, h_sh, mode,
                           as_stream(stream))))
        return rc;
    return down_impl(shape, T, h_disp, h_sh, offsets, w_down, ws_down, y_disp, y_shared, mode, as_stream(stream));
}

int moe_combine(const moe_shape_t* shape, int T, const void* y_disp, const int32_t* inv_perm, const float* topk_w,
                const float* y_shared, void* out, void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (T == 0) return MOE_OK;
    NEED(y_disp, "y_disp");
    NEED4(inv_perm, "inv_perm");
    NEED4(topk_w, "topk_w");
    NEED(out, "out");
    if (y_shared) NEED(y_shared, "y_shared");
    MOE_CUDA(launch_combine(static_cast<const uint16_t*>(y_disp), inv_perm, topk_w, y_shared, T, shape->top_k,
                            shape->hidden, static_cast<uint16_t*>(out), as_stream(stream)),
             "combine launch");
    return MOE_OK;
}

size_t moe_workspace_size(const moe_shape_t* shape, int T) {
    if (check_shape(shape, T)) return 0;
    return fwd_layout(shape, T).total;
}

int moe_forward(const moe_shape_t* shape, int T, const void* x, const void* w_router, const float* bias,
                const int32_t* replica_of, const void* w_gate, const void* w_up, const void* w_down,
                const void* ws_gate, const void* ws_up, const void* ws_down, void* out, int32_t* topk_idx_out,
                float* topk_w_out, int32_t* counts_out, int32_t* block_counts_out, int mode, void* ws,
                size_t ws_bytes, void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (mode < MOE_FFN_AUTO || mode > MOE_FFN_PREFILL) return fail(MOE_ERR_INVALID_ARG, "bad mode %d", mode);
    if (T == 0) return MOE_OK;
    NEED(out, "out");
    const FwdLayout L = fwd_layout(shape, T);
    if (!ws || ws_bytes < L.total) return fail(MOE_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, L.total);
    if (!aligned16(ws)) return fail(MOE_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
    if (topk_idx_out) NEED4(topk_idx_out, "topk_idx_out");
    if (topk_w_out) NEED4(topk_w_out, "topk_w_out");
    if (counts_out) NEED4(counts_out, "counts_out");
    if (block_counts_out) NEED4(block_counts_out, "block_counts_out");
    uint8_t* b = static_cast<uint8_t*>(ws);
    int32_t* idx = topk_idx_out ? topk_idx_out : reinterpret_cast<int32_t*>(b + L.idx);
    float* tw = topk_w_out ? topk_w_out : reinterpret_cast<float*>(b + L.w);
    int32_t* counts = counts_out ? counts_out : reinterpret_cast<int32_t*>(b + L.counts);
    int32_t* blocks = block_counts_out ? block_counts_out : reinterpret_cast<int32_t*>(b + L.blocks);
    int32_t* offsets = reinterpret_cast<int32_t*>(b + L.offsets);
    int32_t* perm = reinterpret_cast<int32_t*>(b + L.perm);
    int32_t* inv = reinterpret_cast<int32_t*>(b + L.inv_perm);
    float* y_sh = shape->n_shared > 0 ? reinterpret_cast<float*>(b + L.y_sh) : nullptr;

    if ((rc = moe_route(shape, T, x, w_router, bias, nullptr, nullptr, idx, tw, b + L.route, route_ws(shape, T),
                        stream)))
        return rc;
    if ((rc = moe_dispatch(shape, T, x, idx, replica_of, reinterpret_cast<int32_t*>(b + L.slot_of), counts, blocks,
                           offsets, perm, inv, b + L.x_disp, b + L.dispatch, dispatch_ws(shape, T), stream)))
        return rc;
    if ((rc = moe_expert_ffn(shape, T, x, b + L.x_disp, offsets, w_gate, w_up, w_down, ws_gate, ws_up, ws_down,
                             b + L.y_disp, y_sh, mode, b + L.ffn, ffn_ws(shape, T), stream)))
        return rc;
    return moe_combine(shape, T, b + L.y_disp, inv, tw, y_sh, out, stream);
}

int moe_quantize_rows_fp8(int rows, int cols, const void* x, uint8_t* codes, float* scale, void* stream) {
    PdlScope pdl((long)rows);
    if (rows < 0 || cols <= 0 || cols % 16) return fail(MOE_ERR_INVALID_ARG, "rows >= 0 and cols %% 16 == 0 required");
    if (rows == 0) return MOE_OK;
    NEED(x, "x");
    NEED(codes, "codes");
    NEED4(scale, "scale");
    MOE_CUDA(launch_quantize_rows(static_cast<const uint16_t*>(x), rows, cols, codes, scale, as_stream(stream)),
             "quantize launch");
    return MOE_OK;
}

int moe_dispatch_fp8(const moe_shape_t* shape, int T, const void* x, const int32_t* topk_idx,
                     const int32_t* replica_of, int32_t* slot_of, int32_t* counts, int32_t* block_counts,
                     int32_t* offsets, int32_t* perm, int32_t* inv_perm, uint8_t* x8, float* x_scale,
                     uint8_t* x_disp8, float* x_disp_scale, void* ws, size_t ws_bytes, void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (shape->hidden % 16) return fail(MOE_ERR_INVALID_ARG, "FP8 rows need hidden %% 16 == 0");
    NEED4(counts, "counts");
    NEED4(offsets, "offsets");
    if (T == 0) return moe_dispatch(shape, 0, x, topk_idx, replica_of, slot_of, counts, block_counts, offsets, perm,
                                    inv_perm, nullptr, nullptr, 0, stream);
    NEED(x, "x");
    NEED4(topk_idx, "topk_idx");
    NEED4(slot_of, "slot_of");
    NEED4(perm, "perm");
    NEED4(inv_perm, "inv_perm");
    NEED(x8, "x8");
    NEED4(x_scale, "x_scale");
    NEED(x_disp8, "x_disp8");
    NEED4(x_disp_scale, "x_disp_scale");
    if (replica_of) NEED4(replica_of, "replica_of");
    cudaStream_t st = as_stream(stream);
    if ((rc = index_impl(shape, T, topk_idx, replica_of, slot_of, counts, block_counts, offsets, perm, inv_perm, ws,
                         ws_bytes, st)))
        return rc;
    MOE_CUDA(launch_quantize_rows(static_cast<const uint16_t*>(x), T, shape->hidden, x8, x_scale, st),
             "quantize launch");
    MOE_CUDA(launch_scatter_fp8(x8, x_scale, perm, T * shape->top_k, shape->top_k, shape->hidden, x_disp8,
                                x_disp_scale, st),
             "FP8 scatter launch");
    return MOE_OK;
}

int moe_expert_gate_up_fp8(const moe_shape_t* shape, int T, const uint8_t* x8, const float* x_scale,
                           const uint8_t* x_disp8, const float* x_disp_scale, const int32_t* offsets,
                           const uint8_t* qg, const float* sg, const uint8_t* qu, const float* su,
                           const uint8_t* qsg, const float* ssg, const uint8_t* qsu, const float* ssu,
                           void* h_disp, void* h_shared, int mode, void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (mode < MOE_FFN_AUTO || mode > MOE_FFN_PREFILL) return fail(MOE_ERR_INVALID_ARG, "bad mode %d", mode);
    if (T == 0) return MOE_OK;
    return gate_up_fp8_impl(shape, T, x8, x_scale, x_disp8, x_disp_scale, offsets, qg, sg, qu, su, qsg, ssg, qsu,
                            ssu, h_disp, h_shared, mode, as_stream(stream));
}

int moe_expert_down_fp8(const moe_shape_t* shape, int T, const uint8_t* h8, const float* h_scale, const uint8_t* hs8,
                        const float* hs_scale, const int32_t* offsets, const uint8_t* qd, const float* sd,
                        const uint8_t* qsd, const float* ssd, void* y_disp, float* y_shared, int mode,
                        void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (mode < MOE_FFN_AUTO || mode > MOE_FFN_PREFILL) return fail(MOE_ERR_INVALID_ARG, "bad mode %d", mode);
    if (T == 0) return MOE_OK;
    return down_fp8_impl(shape, T, h8, h_scale, hs8, hs_scale, offsets, qd, sd, qsd, ssd, y_disp, y_shared, mode,
                         as_stream(stream));
}

int moe_expert_down_fp8_payload(const moe_shape_t* shape, int T, const uint8_t* h8, const float* h_scale,
                                const uint8_t* hs8, const float* hs_scale, const int32_t* offsets, const uint8_t* qd,
                                const float* sd, const uint8_t* qsd, const float* ssd, uint8_t* y_disp8,
                                float* y_disp_scale, float* y_shared, int mode, void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (mode < MOE_FFN_AUTO || mode > MOE_FFN_PREFILL) return fail(MOE_ERR_INVALID_ARG, "bad mode %d", mode);
    if (shape->hidden % 16) return fail(MOE_ERR_INVALID_ARG, "FP8 rows need hidden %% 16 == 0");
    if (T == 0) return MOE_OK;
    return down_fp8_impl(shape, T, h8, h_scale, hs8, hs_scale, offsets, qd, sd, qsd, ssd, nullptr, y_shared, mode,
                         as_stream(stream), y_disp8, y_disp_scale);
}

int moe_combine_fp8(const moe_shape_t* shape, int T, const uint8_t* y_disp8, const float* y_disp_scale,
                    const int32_t* inv_perm, const float* topk_w, const float* y_shared, void* out, void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (shape->hidden % 16) return fail(MOE_ERR_INVALID_ARG, "FP8 rows need hidden %% 16 == 0");
    if (T == 0) return MOE_OK;
    NEED(y_disp8, "y_disp8");
    NEED4(y_disp_scale, "y_disp_scale");
    NEED4(inv_perm, "inv_perm");
    NEED4(topk_w, "topk_w");
    NEED(out, "out");
    if (y_shared) NEED(y_shared, "y_shared");
    MOE_CUDA(launch_combine_fp8(y_disp8, y_disp_scale, inv_perm, topk_w, y_shared, T, shape->top_k, shape->hidden,
                                static_cast<uint16_t*>(out), as_stream(stream)),
             "E4M3 combine launch");
    return MOE_OK;
}

size_t moe_workspace_size_fp8(const moe_shape_t* shape, int T) {
    if (check_shape(shape, T)) return 0;
    return fwd_layout_f8(shape, T).total;
}

int moe_forward_fp8(const moe_shape_t* shape, int T, const void* x, const void* w_router, const float* bias,
                    const int32_t* replica_of, const uint8_t* qg, const float* sg, const uint8_t* qu,
                    const float* su, const uint8_t* qd, const float* sd, const uint8_t* qsg, const float* ssg,
                    const uint8_t* qsu, const float* ssu, const uint8_t* qsd, const float* ssd, void* out,
                    int32_t* topk_idx_out, float* topk_w_out,
                    int32_t* counts_out, int32_t* block_counts_out, int mode, void* ws, size_t ws_bytes,
                    void* stream) {
    PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    int rc = check_shape(shape, T);
    if (rc) return rc;
    if (mode < MOE_FFN_AUTO || mode > MOE_FFN_PREFILL) return fail(MOE_ERR_INVALID_ARG, "bad mode %d", mode);
    if (shape->hidden % 16 || shape->inter % 16 || (shape->n_shared * shape->inter_shared) % 16)
        return fail(MOE_ERR_INVALID_ARG,
                    "FP8 rows need hidden, inter and n_shared*inter_shared to be multiples of 16");
    if (T == 0) return MOE_OK;
    NEED(out, "out");
    const FwdLayoutF8 L = fwd_layout_f8(shape, T);
    if (!ws || ws_bytes < L.total) return fail(MOE_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, L.total);
    if (!aligned16(ws)) return fail(MOE_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
    uint8_t* b = static_cast<uint8_t*>(ws);
    const FwdLayout& B = L.base;
    int32_t* idx = topk_idx_out ? topk_idx_out : reinterpret_cast<int32_t*>(b + B.idx);
    float* tw = topk_w_out ? topk_w_out : reinterpret_cast<float*>(b + B.w);
    int32_t* counts = counts_out ? counts_out : reinterpret_cast<int32_t*>(b + B.counts);
    int32_t* blocks = block_counts_out ? block_counts_out : reinterpret_cast<int32_t*>(b + B.blocks);
    int32_t* offsets = reinterpret_cast<int32_t*>(b + B.offsets);
    int32_t* perm = reinterpret_cast<int32_t*>(b + B.perm);
    int32_t* inv = reinterpret_cast<int32_t*>(b + B.inv_perm);
    float* y_sh = shape->n_shared > 0 ? reinterpret_cast<float*>(b + B.y_sh) : nullptr;
    uint8_t* h = b + B.ffn;
    uint8_t* hs = shape->n_shared > 0 ? h + align256((size_t)T * shape->top_k * shape->inter * 2) : nullptr;
    if ((rc = moe_route(shape, T, x, w_router, bias, nullptr, nullptr, idx, tw, b + B.route, route_ws(shape, T),
                        stream)))
        return rc;
    if ((rc = moe_dispatch_fp8(shape, T, x, idx, replica_of, reinterpret_cast<int32_t*>(b + B.slot_of), counts,
                               blocks, offsets, perm, inv, b + L.x8, reinterpret_cast<float*>(b + L.x_scale),
                               b + L.x_disp8, reinterpret_cast<float*>(b + L.x_disp_scale), b + B.dispatch,
                               dispatch_ws(shape, T), stream)))
        return rc;
    if ((rc = moe_expert_gate_up_fp8(shape, T, b + L.x8, reinterpret_cast<float*>(b + L.x_scale), b + L.x_disp8,
                                     reinterpret_cast<float*>(b + L.x_disp_scale), offsets, qg, sg, qu, su, qsg, ssg,
                                     qsu, ssu, h, hs, mode, stream)))
        return rc;
    // the bf16 intermediates as E4M3 rows: one per (token, routed expert), one per token for the shared experts
    const int n = T * shape->top_k;
    const int Ks = shape->n_shared * shape->inter_shared;
    cudaStream_t st = as_stream(stream);
    float* h_scale = reinterpret_cast<float*>(b + L.h_scale);
    float* hs_scale = Ks > 0 ? reinterpret_cast<float*>(b + L.hs_scale) : nullptr;
    MOE_CUDA(launch_quantize_rows(reinterpret_cast<const uint16_t*>(h), n, shape->inter, b + L.h8, h_scale, st),
             "intermediate quantize launch");
    if (Ks > 0)
        MOE_CUDA(launch_quantize_rows(reinterpret_cast<const uint16_t*>(hs), T, Ks, b + L.hs8, hs_scale, st),
                 "shared intermediate quantize launch");
    // expert outputs leave as the E4M3 combine payload (codes + one scale per 128-column block)
    uint8_t* y8 = b + L.y8;
    float* y_scale = reinterpret_cast<float*>(b + L.y_scale);
    if ((rc = moe_expert_down_fp8_payload(shape, T, b + L.h8, h_scale, Ks > 0 ? b + L.hs8 : nullptr, hs_scale,
                                          offsets, qd, sd, qsd, ssd, y8, y_scale, y_sh, mode, stream)))
        return rc;
    return moe_combine_fp8(shape, T, y8, y_scale, inv, tw, y_sh, out, stream);
}

}  // extern "C"
