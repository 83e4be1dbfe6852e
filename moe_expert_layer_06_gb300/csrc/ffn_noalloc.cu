// moe_expert_ffn_noalloc: the expert FFN (gate/up + SwiGLU, then down) for
// callers that cannot allocate device memory.
//
// moe_expert_ffn needs a caller-provided workspace for the SwiGLU
// intermediate h.  Some callers have no way to provide one: a plugin inside
// a host program that owns every device allocation and hands the plugin only
// its inputs and outputs, or code on a latency-critical path where
// cudaMalloc's implicit device synchronisation is not acceptable.  This
// entry point keeps h in a fixed array in the library's own device memory
// instead, so it allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (MOE_FFN_NOALLOC_SCRATCH_BYTES) until the process exits.
// Host code may not use the array's name as a device address (on the host it
// is only a stand-in symbol), so the device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, on the first
// call made on that device.  Every call shares the array: calls whose work
// overlaps on the GPU (two streams, or two host threads on one device) race
// on it, and each call overwrites what the previous one left there.  The
// kernels write every element of h they later read, so nothing needs to be
// cleared between calls.
#include <mutex>

#include "moe.h"
#include "kernels.h"

namespace moe {
namespace {

static __device__ __align__(256) unsigned char g_ffn_scratch[MOE_FFN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
static void* g_scratch_ptr[kMaxDevices];
static std::mutex g_scratch_mu;

// Device address of g_ffn_scratch on the current device (looked up once per device).
static cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_ffn_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

inline size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace
}  // namespace moe

extern "C" int moe_expert_ffn_noalloc(const moe_shape_t* shape, int T, const void* x, const void* x_disp,
                                      const int32_t* offsets, const void* w_gate, const void* w_up,
                                      const void* w_down, const void* ws_gate, const void* ws_up,
                                      const void* ws_down, void* y_disp, float* y_shared, int mode,
                                      void* stream) {
    moe::PdlScope pdl((long)T * (shape ? shape->top_k : 0));
    using namespace moe;
    int rc = api_check_shape(shape, T);
    if (rc != MOE_OK) return rc;
    if (mode < MOE_FFN_AUTO || mode > MOE_FFN_PREFILL) return api_fail(MOE_ERR_INVALID_ARG, "bad mode %d", mode);
    if (T == 0) return MOE_OK;
    const size_t h_bytes = round256((size_t)T * shape->top_k * shape->inter * 2);
    const size_t hs_bytes = shape->n_shared > 0 ? (size_t)T * shape->n_shared * shape->inter_shared * 2 : 0;
    if (h_bytes + hs_bytes > (size_t)MOE_FFN_NOALLOC_SCRATCH_BYTES)
        return api_fail(MOE_ERR_UNSUPPORTED,
                        "moe_expert_ffn_noalloc: T=%d needs %zu bytes of intermediate, the library's fixed "
                        "scratch holds %zu; use moe_expert_ffn with a workspace",
                        T, h_bytes + hs_bytes, (size_t)MOE_FFN_NOALLOC_SCRATCH_BYTES);
    void* base = nullptr;
    const cudaError_t e = scratch_address(&base);
    if (e != cudaSuccess)
        return api_fail(MOE_ERR_CUDA, "moe_expert_ffn_noalloc: scratch address: %s", cudaGetErrorString(e));
    unsigned char* h = static_cast<unsigned char*>(base);
    void* hs = shape->n_shared > 0 ? h + h_bytes : nullptr;
    rc = moe_expert_gate_up(shape, T, x, x_disp, offsets, w_gate, w_up, ws_gate, ws_up, h, hs, mode, stream);
    if (rc != MOE_OK) return rc;
    return moe_expert_down(shape, T, h, hs, offsets, w_down, ws_down, y_disp, y_shared, mode, stream);
}
