// FP8 (E4M3) quantisation of rows and the FP8 dispatch scatter.
//
// Blog post "专家并行(EP)", section 2.3: with FP8 communication the dispatch
// and combine volume per token halves (229 KB -> 115 KB at top-8, hidden
// 7168).  A row (a token's hidden state, or one output row of a weight
// matrix) is stored as E4M3 codes with one fp32 scale: scale = amax / 448
// (1 for an all-zero row), code = e4m3(x / scale) rounded to nearest even
// with saturation; the value is code * scale.
#include <cuda_fp8.h>

#include "kernels.h"

namespace moe {
namespace {

// One warp per row, 8 bf16 (16 bytes) per lane per step.
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint4* __restrict__ x, int rows, int vec_per_row,
                                                            uint2* __restrict__ codes, float* __restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < rows; r += gridDim.x * wpb) {
        const uint4* src = x + (size_t)r * vec_per_row;
        float amax = 0.0f;
        for (int v = lane; v < vec_per_row; v += 32) {
            const uint4 q = __ldg(src + v);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
                amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xffff0000u)));
            }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        if (lane == 0) scale[r] = s;
        uint2* dst = codes + (size_t)r * vec_per_row;
        for (int v = lane; v < vec_per_row; v += 32) {
            const uint4 q = __ldg(src + v);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
            uint32_t packed[2] = {0, 0};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float lo = __fdiv_rn(__uint_as_float(w[i] << 16), s);
                const float hi = __fdiv_rn(__uint_as_float(w[i] & 0xffff0000u), s);
                const uint32_t c0 = __nv_cvt_float_to_fp8(lo, __NV_SATFINITE, __NV_E4M3);
                const uint32_t c1 = __nv_cvt_float_to_fp8(hi, __NV_SATFINITE, __NV_E4M3);
                packed[i >> 1] |= (c0 | (c1 << 8)) << ((i & 1) * 16);
            }
            dst[v] = make_uint2(packed[0], packed[1]);
        }
    }
}

// x_disp8[row] = x8[perm[row] / k], one warp per row, 16-byte vectors; lane 0 copies the scale.
__global__ void __launch_bounds__(256) scatter_fp8_kernel(const uint4* __restrict__ x8, const float* __restrict__ xs,
                                                          const int32_t* __restrict__ perm, int n_rows, int k,
                                                          int vec_per_row, uint4* __restrict__ out,
                                                          float* __restrict__ out_scale) {
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    for (int row = blockIdx.x * wpb + (threadIdx.x >> 5); row < n_rows; row += gridDim.x * wpb) {
        const int t = perm[row] / k;
        const uint4* src = x8 + (size_t)t * vec_per_row;
        uint4* dst = out + (size_t)row * vec_per_row;
#pragma unroll 4
        for (int v = lane; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
        if (lane == 0) out_scale[row] = __ldg(xs + t);
    }
}

}  // namespace

cudaError_t launch_quantize_rows(const uint16_t* x, int rows, int cols, uint8_t* codes, float* scale,
                                 cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const int wpb = 8;
    int blocks = (rows + wpb - 1) / wpb;
    const int cap = num_sms() * 16;
    if (blocks > cap) blocks = cap;
    quantize_rows_kernel<<<blocks, wpb * 32, 0, stream>>>(reinterpret_cast<const uint4*>(x), rows, cols / 8,
                                                          reinterpret_cast<uint2*>(codes), scale);
    return cudaGetLastError();
}

cudaError_t launch_scatter_fp8(const uint8_t* x8, const float* x_scale, const int32_t* perm, int n_rows, int k,
                               int row_bytes, uint8_t* x_disp8, float* x_disp_scale, cudaStream_t stream) {
    if (n_rows <= 0) return cudaSuccess;
    const int wpb = 8;
    int blocks = (n_rows + wpb - 1) / wpb;
    const int cap = num_sms() * 16;
    if (blocks > cap) blocks = cap;
    scatter_fp8_kernel<<<blocks, wpb * 32, 0, stream>>>(reinterpret_cast<const uint4*>(x8), x_scale, perm, n_rows, k,
                                                        row_bytes / 16, reinterpret_cast<uint4*>(x_disp8),
                                                        x_disp_scale);
    return cudaGetLastError();
}

}  // namespace moe
