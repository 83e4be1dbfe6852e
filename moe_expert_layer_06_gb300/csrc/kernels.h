// Host-side declarations shared by the library's translation units (not part
// of the public C ABI, which is include/moe.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "moe.h"
#include "common.cuh"

namespace moe {

// Programmatic dependent launch pays for small and mid-size batches (launch
// gaps are a visible part of the step) and costs a little for large ones
// (measured on the same GPU: E4M3 decode T=32 0.9% and T=1024 0.8% faster,
// prefill T=4096 0.7% slower).  Each entry point of the C ABI turns it on for
// at most kPdlMaxAssignments token-expert assignments (PdlScope); launch_pdl
// reads the calling thread's setting.
constexpr long kPdlMaxAssignments = 8192;
bool pdl_enabled();

struct PdlScope {
    bool saved;
    explicit PdlScope(long assignments);
    ~PdlScope();
};

// Launch `kern`, with programmatic stream serialisation when enabled (the
// kernels' pdl_begin is then their wait for the predecessor; otherwise it
// returns at once).
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Run `configure` (a kernel attribute such as its dynamic shared memory) the
// first time the calling thread's device needs it, from any number of host
// threads: `done` holds one bit per configured device (ordinals 0..63; others
// configure on every call).  Concurrent first calls may both configure, which
// is idempotent.
template <typename F>
inline cudaError_t configure_once(std::atomic<uint64_t>& done, F&& configure) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return configure();
    const uint64_t bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = configure();
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// ---------------------------------------------------------------- grouped swap-AB GEMM (tcgen05)
// kGateUpF8 / kDownF8: gate/up and down with E4M3 operands (128-element K
// chunks, tcgen05 kind::f8f6f4), per-row weight scales and per-row token
// (or intermediate) scales applied in the epilogue (they factor out of the K
// sum).  The FP8 shared down is one matrix [H, n_sh*I_sh] on the concatenated
// shared intermediate.
// kDownF8Q: kDownF8 whose routed outputs leave as the E4M3 combine payload:
// each output row's bf16 value quantised in blocks of kPayloadBlock columns
// (one fp32 scale per block, codes as the row quantiser's); a down item owns
// 256 consecutive output columns, so every block is reduced inside one CTA.
enum GemmMode : int { kGateUp = 0, kDown = 1, kRouter = 2, kGateUpF8 = 3, kDownF8 = 4, kDownF8Q = 5 };
constexpr int kPayloadBlock = MOE_PAYLOAD_BLOCK;

// One launch computes D = A * B^T for a list of work items.  A is a weight
// tile of 128 output rows (the UMMA M operand), B is a chunk of up to BN
// token rows (the UMMA N operand), K runs over 128-byte chunks (64 bf16 or
// 128 E4M3 elements).  Every operand is read by TMA through the tensor maps
// below (3-D, 128-byte swizzle; weights box {128 B, 128, 1}; tokens box
// {128 B, 1, 16 << j}, so a chunk of n 16-row groups is loaded exactly with one
// box per set bit of n).
struct GemmArgs {
    CUtensorMap a0;   // routed weights: gate [S,I,H] | down [S,H,I] | router [1,E,H]
    CUtensorMap a1;   // routed up weights [S,I,H] (gate/up only)
    CUtensorMap b[4]; // routed activations: x_disp [T*k,H] | h_disp [T*k,I] | x [T,H]; boxes of 16,32,64,128 rows
    CUtensorMap sa0;  // shared gate [n_sh,I_sh,H] | shared down [n_sh,H,I_sh]
    CUtensorMap sa1;  // shared up [n_sh,I_sh,H]
    CUtensorMap sb[4];// shared activations: x [T,H] | h_sh [T,n_sh,I_sh]; same four box heights
    const int32_t* offsets;  // [S+2] dispatch row offsets (gate/up, down)
    int n_slots;
    int T;
    int m_routed;     // output rows per routed matrix: I | H | E
    int kc_routed;    // K chunks (128 bytes each) of a routed item
    int n_shared;     // shared experts (0: none)
    int m_shared;     // output rows per shared matrix: I_sh | H
    int kc_shared;    // K chunks of a shared item: ceil(H/64) | n_sh*ceil(I_sh/64) (E4M3: /128, one
                      // concatenated shared down matrix)
    int kc_per_sh;    // bf16 down: K chunks per shared expert, ceil(I_sh/64)
    int ksplit;       // router: number of K splits
    int kc_split;     // router: K chunks per split
    void* out;        // h_disp bf16 | y_disp bf16 | logit partials f32 [ksplit,T,E]
    int out_ld;
    void* out_sh;     // h_sh bf16 [T, n_sh*I_sh] | y_sh f32 [T,H]
    int out_sh_ld;
    int sh_col_stride;  // gate/up: I_sh (column offset of shared expert j in h_sh)
    // FP8 modes only: dequantisation scales
    const float* a0_scale;  // routed gate rows [S*I] | routed down rows [S*H]
    const float* a1_scale;  // routed up rows [S*I]
    const float* sa0_scale; // shared gate rows [n_sh*I_sh] | shared down rows [H]
    const float* sa1_scale; // shared up rows [n_sh*I_sh]
    const float* b_scale;   // dispatched token rows [T*k] | intermediate rows [T*k]
    const float* sb_scale;  // tokens [T] | shared intermediate rows [T]
    // kDownF8Q only: the E4M3 combine payload of the routed rows
    uint8_t* out8;          // codes [T*k, m_routed]
    float* out8_scale;      // block scales [T*k, n_blk]
    int n_blk;              // ceil(m_routed / kPayloadBlock)
    DevStatus st;
};

// Token chunk of the prefill variant: 160 rows covers every expert of a 4096-token
// batch with uniform routing (128 +- 11 rows) in one chunk while leaving room
// for 4 pipeline stages (128 KB of weights in flight per SM).
constexpr int kPrefillBN = 160;

// Token chunk of the E4M3 down GEMM when T > 32 and the batch averages at most
// kMidMaxRowsPerSlot rows per slot (T*k <= kMidMaxRowsPerSlot*S; T <= 1024 at
// 256 experts, top-8).  An E4M3 down item runs only ceil(I/128) K chunks (16 at
// I = 2048), so handing its accumulator to the epilogue is a large share of it;
// 128 rows leave TMEM room for two accumulators (2 x 2 x 128 columns), and the
// next item's MMAs start while the epilogue drains the last one (measured on
// one GB300: redundant T=1024 -1.9%, skewed T=256 -2.1%).  With ~128 rows per
// expert, 128-row chunks split half the experts in two and 160 is faster; so
// are the E4M3 gate/up (56 K chunks an item) and the bf16 GEMMs.
constexpr int kMidBN = 128;
constexpr int kMidMaxRowsPerSlot = 32;

// Launch the grouped GEMM for `mode` with token chunk bn (32, kPrefillBN, or
// kMidBN for the E4M3 down).
cudaError_t launch_gemm(GemmMode mode, int bn, const GemmArgs& args, int grid, cudaStream_t stream);
int gemm_max_slots();  // slots the GEMM's shared-memory item table holds

// ---------------------------------------------------------------- TMA tensor maps
// 3-D bf16 tensor map, dims innermost first (elements), strides of dims 1,2 in bytes.
int make_tmap_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                 uint32_t box2, bool fp8 = false);

// ---------------------------------------------------------------- FP8 (E4M3) quantisation
// codes[r][c] = e4m3(x[r][c] / scale[r]), scale[r] = amax(|x[r]|) / 448 (1 for a zero row),
// round to nearest even with saturation; cols % 8 == 0.
cudaError_t launch_quantize_rows(const uint16_t* x, int rows, int cols, uint8_t* codes, float* scale,
                                 cudaStream_t stream);
// x_disp8[row] = x8[perm[row] / k] (row_bytes per row, 16-byte vectors), x_disp_scale[row] likewise.
cudaError_t launch_scatter_fp8(const uint8_t* x8, const float* x_scale, const int32_t* perm, int n_rows, int k,
                               int row_bytes, uint8_t* x_disp8, float* x_disp_scale, cudaStream_t stream);

// ---------------------------------------------------------------- routing
// Top-k over the (K-split) router logits; n_groups > topk_groups restricts the
// selection to the topk_groups groups of E/n_groups experts with the best
// maximum logit (n_groups <= 32); n_groups = 0 means no grouping.
cudaError_t launch_topk(const float* partials, int ksplit, const float* bias, int T, int E, int k,
                        float* logits_out, int32_t* topk_idx, float* topk_w, int n_groups, int topk_groups,
                        const DevStatus& st, cudaStream_t stream);

// ---------------------------------------------------------------- dispatch / histogram
struct DispatchArgs {
    int T, k, E, S, n_blocks, hidden;
    const int32_t* topk_idx;
    const int32_t* replica_of;
    int32_t* slot_of;
    int32_t* counts;        // [S+1]
    int32_t* block_counts;  // [n_blocks] or null
    int32_t* offsets;       // [S+2] or null (histogram only)
    int32_t* perm;          // [T*k] or null
    int32_t* inv_perm;      // [T*k] or null
    DevStatus st;
};
cudaError_t launch_index_pass(const DispatchArgs& a, cudaStream_t stream);
// The index pass in chunks (three launches) for large batches: index_chunks(n)
// chunks (0: use launch_index_pass), with index_workspace_bytes(n, S) of
// caller workspace for the per-chunk histograms.
int index_chunks(int n);
size_t index_workspace_bytes(int n, int n_slots);
cudaError_t launch_index_chunked(const DispatchArgs& a, int32_t* hist, cudaStream_t stream);
cudaError_t launch_scatter_rows(const uint16_t* x, const int32_t* perm, int n_rows, int k, int hidden,
                                uint16_t* x_disp, cudaStream_t stream);
int dispatch_max_slots();  // slots the index pass's shared-memory histograms hold

// ---------------------------------------------------------------- combine
cudaError_t launch_combine(const uint16_t* y_disp, const int32_t* inv_perm, const float* topk_w,
                           const float* y_shared, int T, int k, int hidden, uint16_t* out,
                           cudaStream_t stream);

// E4M3 combine payload: y8 [T*k, hidden] codes, y_scale [T*k, ceil(hidden/kPayloadBlock)].
cudaError_t launch_combine_fp8(const uint8_t* y8, const float* y_scale, const int32_t* inv_perm, const float* topk_w,
                               const float* y_shared, int T, int k, int hidden, uint16_t* out, cudaStream_t stream);

int num_sms();

// Error reporting and shape validation of the C ABI, for entry points defined
// outside moe_api.cu.
int api_fail(int code, const char* fmt, ...);
int api_check_shape(const moe_shape_t* shape, int T);

}  // namespace moe
