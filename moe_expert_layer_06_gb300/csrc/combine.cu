// Combine of the MoE layer on one device, fused with the shared-expert add.
//
// Blog post "专家并行(EP)", section 2.2 steps 4-5: expert outputs return to
// their token (here: a gather through inv_perm) and
//   out[t] = sum_{j<k} softmax(logits)[idx_j] * expert_out_j + shared_out[t],
// accumulated in fp32 in ascending j, then the shared expert output, rounded
// once to bf16.  8 bf16 (16 bytes) per thread per step.  With the E4M3
// combine payload (section 2.3: FP8 communication) each expert output element
// is its code times the fp32 scale of its 128-column block.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "kernels.h"

namespace moe {
namespace {

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&p);
}

__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ y_disp,
                                                      const int32_t* __restrict__ inv_perm,
                                                      const float* __restrict__ topk_w,
                                                      const float4* __restrict__ y_shared, int T, int k,
                                                      int vec_per_row, uint4* __restrict__ out) {
    pdl_begin();
    const size_t total = (size_t)T * vec_per_row;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(idx / vec_per_row);
        const int c = (int)(idx - (size_t)t * vec_per_row);
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
        if (y_shared) {  // independent of the gathers: issue first
            s0 = __ldg(y_shared + ((size_t)t * vec_per_row + c) * 2);
            s1 = __ldg(y_shared + ((size_t)t * vec_per_row + c) * 2 + 1);
        }
        // up to 8 assignments at a time: all row indices, then all rows, then the sum in ascending j
        for (int j0 = 0; j0 < k; j0 += 8) {
            int row[8];
            float w[8];
            uint4 yv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (j0 + u < k) {
                    row[u] = __ldg(inv_perm + (size_t)t * k + j0 + u);
                    w[u] = __ldg(topk_w + (size_t)t * k + j0 + u);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (j0 + u < k) yv[u] = __ldg(y_disp + (size_t)row[u] * vec_per_row + c);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (j0 + u < k) {
                    float y[8];
                    unpack8(yv[u], y);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = fmaf(w[u], y[i], acc[i]);
                }
            }
        }
        if (y_shared) {
            acc[0] += s0.x; acc[1] += s0.y; acc[2] += s0.z; acc[3] += s0.w;
            acc[4] += s1.x; acc[5] += s1.y; acc[6] += s1.z; acc[7] += s1.w;
        }
        uint4 o;
        o.x = pack2(acc[0], acc[1]);
        o.y = pack2(acc[2], acc[3]);
        o.z = pack2(acc[4], acc[5]);
        o.w = pack2(acc[6], acc[7]);
        out[idx] = o;
    }
}

// E4M3 payload: 16 codes (one 16-byte vector) per thread per step, dequantised
// with the scale of their 128-column block (16 | 128, so a vector never
// straddles two blocks); otherwise as combine_kernel.  A code byte carries half
// the bytes of a bf16 element, so each thread covers twice the columns to keep
// as many bytes in flight.
__global__ void __launch_bounds__(256, 2) combine_fp8_kernel(const uint4* __restrict__ y8,
                                                          const float* __restrict__ y_scale,
                                                          const int32_t* __restrict__ inv_perm,
                                                          const float* __restrict__ topk_w,
                                                          const float4* __restrict__ y_shared, int T, int k,
                                                          int vec_per_row, int n_blk, uint4* __restrict__ out) {
    pdl_begin();
    const size_t total = (size_t)T * vec_per_row;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(idx / vec_per_row);
        const int c = (int)(idx - (size_t)t * vec_per_row);
        const int blk = (c * 16) / kPayloadBlock;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
        float4 sh[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) sh[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (y_shared) {  // independent of the gathers: issue first
#pragma unroll
            for (int i = 0; i < 4; ++i) sh[i] = __ldg(y_shared + ((size_t)t * vec_per_row + c) * 4 + i);
        }
        for (int j0 = 0; j0 < k; j0 += 8) {
            int row[8];
            float w[8], sc[8];
            uint4 yv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (j0 + u < k) {
                    row[u] = __ldg(inv_perm + (size_t)t * k + j0 + u);
                    w[u] = __ldg(topk_w + (size_t)t * k + j0 + u);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (j0 + u < k) {
                    yv[u] = __ldg(y8 + (size_t)row[u] * vec_per_row + c);
                    sc[u] = __ldg(y_scale + (size_t)row[u] * n_blk + blk);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (j0 + u < k) {
                    const uint32_t wd[4] = {yv[u].x, yv[u].y, yv[u].z, yv[u].w};
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
                            (__nv_fp8x2_storage_t)((wd[h >> 1] >> ((h & 1) * 16)) & 0xffffu), __NV_E4M3);
                        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
                        acc[2 * h] = fmaf(w[u], f.x * sc[u], acc[2 * h]);
                        acc[2 * h + 1] = fmaf(w[u], f.y * sc[u], acc[2 * h + 1]);
                    }
                }
            }
        }
        if (y_shared) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[4 * i] += sh[i].x;
                acc[4 * i + 1] += sh[i].y;
                acc[4 * i + 2] += sh[i].z;
                acc[4 * i + 3] += sh[i].w;
            }
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            uint4 o;
            o.x = pack2(acc[8 * i], acc[8 * i + 1]);
            o.y = pack2(acc[8 * i + 2], acc[8 * i + 3]);
            o.z = pack2(acc[8 * i + 4], acc[8 * i + 5]);
            o.w = pack2(acc[8 * i + 6], acc[8 * i + 7]);
            out[idx * 2 + i] = o;
        }
    }
}

}  // namespace

cudaError_t launch_combine_fp8(const uint8_t* y8, const float* y_scale, const int32_t* inv_perm, const float* topk_w,
                               const float* y_shared, int T, int k, int hidden, uint16_t* out, cudaStream_t stream) {
    const int vpr = hidden / 16;
    const size_t total = (size_t)T * vpr;
    if (total == 0) return cudaSuccess;
    size_t blocks = (total + 255) / 256;
    const size_t cap = (size_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(combine_fp8_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                      reinterpret_cast<const uint4*>(y8), y_scale, inv_perm, topk_w,
                      reinterpret_cast<const float4*>(y_shared), T, k, vpr, (hidden + kPayloadBlock - 1) / kPayloadBlock,
                      reinterpret_cast<uint4*>(out));
}

cudaError_t launch_combine(const uint16_t* y_disp, const int32_t* inv_perm, const float* topk_w,
                           const float* y_shared, int T, int k, int hidden, uint16_t* out,
                           cudaStream_t stream) {
    const int vpr = hidden / 8;
    const size_t total = (size_t)T * vpr;
    if (total == 0) return cudaSuccess;
    size_t blocks = (total + 255) / 256;
    const size_t cap = (size_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(combine_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                      reinterpret_cast<const uint4*>(y_disp), inv_perm, topk_w,
                      reinterpret_cast<const float4*>(y_shared), T, k, vpr, reinterpret_cast<uint4*>(out));
}

}  // namespace moe
