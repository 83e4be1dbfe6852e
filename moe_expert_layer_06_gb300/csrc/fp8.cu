// FP8 (E4M3) quantisation of rows and the FP8 dispatch scatter.
//
// Blog post "专家并行(EP)", section 2.3: with FP8 communication the dispatch
// and combine volume per token halves (229 KB -> 115 KB at top-8, hidden
// 7168).  A row (a token's hidden state, or one output row of a weight
// matrix) is stored as E4M3 codes with one fp32 scale: scale = amax / 448
// (1 for an all-zero row), code = e4m3(x / scale) rounded to nearest even
// with saturation; the value is code * scale.
#include <cuda_fp8.h>

#include "e4m3.cuh"
#include "kernels.h"

namespace moe {
namespace {

// E4M3 codes of 8 bf16 values (one 16-byte vector) at a row's scale, packed
// into 8 bytes in element order (two values per conversion).
template <bool FAST>
__device__ __forceinline__ uint2 encode8(const uint4 q, const RowDiv& div) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint32_t packed[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = div_rn<FAST>(div, __uint_as_float(w[i] << 16));
        const float hi = div_rn<FAST>(div, __uint_as_float(w[i] & 0xffff0000u));
        const uint32_t c = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
        packed[i >> 1] |= c << ((i & 1) * 16);
    }
    return make_uint2(packed[0], packed[1]);
}

__device__ __forceinline__ float amax8(const uint4 q, float m) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
        m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xffff0000u)));
    }
    return m;
}

// Single pass: a row is spread over tpr threads (a multiple of 32), each
// holding up to kVpt 16-byte vectors in registers: load, amax over the row
// (warp shuffles, then shared memory across the row's warps), encode from the
// registers, store.  blockDim.x / tpr rows per CTA, grid-stride over rows.
constexpr int kVpt = 8;
constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads, 3) quantize_rows_kernel(const uint4* __restrict__ x, int rows,
                                                                      int vec_per_row, int tpr,
                                                                      uint2* __restrict__ codes,
                                                                      float* __restrict__ scale) {
    pdl_begin();
    __shared__ float part[kQuantThreads / 32];
    const int rows_per_cta = blockDim.x / tpr;
    const int sub = threadIdx.x / tpr;  // row slot of this thread in the CTA
    const int t = threadIdx.x - sub * tpr;
    const int lane = threadIdx.x & 31;
    const int wpr = tpr >> 5;  // warps per row
    for (int r0 = blockIdx.x * rows_per_cta; r0 < rows; r0 += gridDim.x * rows_per_cta) {
        const int r = r0 + sub;
        const bool live = r < rows;
        const uint4* src = x + (size_t)r * vec_per_row;
        uint4 v[kVpt];
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < kVpt; ++j) {
            const int c = t + j * tpr;
            v[j] = make_uint4(0, 0, 0, 0);
            if (live && c < vec_per_row) v[j] = __ldg(src + c);
        }
#pragma unroll
        for (int j = 0; j < kVpt; ++j) amax = amax8(v[j], amax);
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        if (wpr > 1) {
            __syncthreads();  // part[] free from the previous round
            if (lane == 0) part[threadIdx.x >> 5] = amax;
            __syncthreads();
            const int w0 = sub * wpr;
            for (int q = 0; q < wpr; ++q) amax = fmaxf(amax, part[w0 + q]);
        }
        const float s = row_scale(amax);
        if (live) {
            if (t == 0) scale[r] = s;
            const RowDiv div = row_div(s);
            uint2* dst = codes + (size_t)r * vec_per_row;
            if (div.fast) {
#pragma unroll
                for (int j = 0; j < kVpt; ++j) {
                    const int c = t + j * tpr;
                    if (c < vec_per_row) dst[c] = encode8<true>(v[j], div);
                }
            } else {
#pragma unroll
                for (int j = 0; j < kVpt; ++j) {
                    const int c = t + j * tpr;
                    if (c < vec_per_row) dst[c] = encode8<false>(v[j], div);
                }
            }
        }
    }
}

// Rows too long for the registers of one CTA: one warp per row, two passes.
__global__ void __launch_bounds__(256) quantize_long_rows_kernel(const uint4* __restrict__ x, int rows,
                                                                 int vec_per_row, uint2* __restrict__ codes,
                                                                 float* __restrict__ scale) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < rows; r += gridDim.x * wpb) {
        const uint4* src = x + (size_t)r * vec_per_row;
        float amax = 0.0f;
        for (int c = lane; c < vec_per_row; c += 32) amax = amax8(__ldg(src + c), amax);
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        const float s = row_scale(amax);
        if (lane == 0) scale[r] = s;
        const RowDiv div = row_div(s);
        uint2* dst = codes + (size_t)r * vec_per_row;
        if (div.fast)
            for (int c = lane; c < vec_per_row; c += 32) dst[c] = encode8<true>(__ldg(src + c), div);
        else
            for (int c = lane; c < vec_per_row; c += 32) dst[c] = encode8<false>(__ldg(src + c), div);
    }
}

// x_disp8[row] = x8[perm[row] / k] (16-byte vectors, a row over tpr threads that
// issue all of their loads before storing), x_disp_scale[row] likewise.
__global__ void __launch_bounds__(kQuantThreads) scatter_fp8_kernel(const uint4* __restrict__ x8,
                                                                    const float* __restrict__ xs,
                                                                    const int32_t* __restrict__ perm, int n_rows,
                                                                    int k, int vec_per_row, int tpr,
                                                                    uint4* __restrict__ out,
                                                                    float* __restrict__ out_scale) {
    pdl_begin();
    const int rows_per_cta = blockDim.x / tpr;
    const int sub = threadIdx.x / tpr;
    const int t0 = threadIdx.x - sub * tpr;
    for (int r0 = blockIdx.x * rows_per_cta; r0 < n_rows; r0 += gridDim.x * rows_per_cta) {
        const int row = r0 + sub;
        if (row >= n_rows) continue;
        const int t = __ldg(perm + row) / k;
        const uint4* src = x8 + (size_t)t * vec_per_row;
        uint4* dst = out + (size_t)row * vec_per_row;
        for (int c0 = 0; c0 < vec_per_row; c0 += kVpt * tpr) {
            uint4 v[kVpt];
#pragma unroll
            for (int j = 0; j < kVpt; ++j) {
                const int c = c0 + t0 + j * tpr;
                if (c < vec_per_row) v[j] = __ldg(src + c);
            }
#pragma unroll
            for (int j = 0; j < kVpt; ++j) {
                const int c = c0 + t0 + j * tpr;
                if (c < vec_per_row) dst[c] = v[j];
            }
        }
        if (t0 == 0) out_scale[row] = __ldg(xs + t);
    }
}

}  // namespace

cudaError_t launch_quantize_rows(const uint16_t* x, int rows, int cols, uint8_t* codes, float* scale,
                                 cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const int vec = cols / 8;
    const int cap = num_sms() * 8;
    if (vec > kVpt * kQuantThreads) {
        int blocks = (rows + 7) / 8;
        if (blocks > cap) blocks = cap;
        return launch_pdl(quantize_long_rows_kernel, dim3(blocks), dim3(256), 0, stream,
                          reinterpret_cast<const uint4*>(x), rows, vec, reinterpret_cast<uint2*>(codes), scale);
    }
    // threads per row: the fewest warps whose registers hold the row
    int tpr = 32;
    while (tpr * kVpt < vec) tpr <<= 1;
    const int rows_per_cta = kQuantThreads / tpr;
    int blocks = (rows + rows_per_cta - 1) / rows_per_cta;
    if (blocks > cap) blocks = cap;
    return launch_pdl(quantize_rows_kernel, dim3(blocks), dim3(kQuantThreads), 0, stream,
                      reinterpret_cast<const uint4*>(x), rows, vec, tpr, reinterpret_cast<uint2*>(codes), scale);
}

cudaError_t launch_scatter_fp8(const uint8_t* x8, const float* x_scale, const int32_t* perm, int n_rows, int k,
                               int row_bytes, uint8_t* x_disp8, float* x_disp_scale, cudaStream_t stream) {
    if (n_rows <= 0) return cudaSuccess;
    const int vec = row_bytes / 16;
    int tpr = 32;
    while (tpr * kVpt < vec && tpr < kQuantThreads) tpr <<= 1;
    const int rows_per_cta = kQuantThreads / tpr;
    int blocks = (n_rows + rows_per_cta - 1) / rows_per_cta;
    const int cap = num_sms() * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(scatter_fp8_kernel, dim3(blocks), dim3(kQuantThreads), 0, stream,
                      reinterpret_cast<const uint4*>(x8), x_scale, perm, n_rows, k, vec, tpr,
                      reinterpret_cast<uint4*>(x_disp8), x_disp_scale);
}

}  // namespace moe
