// Weighted combine / unpermute.
//
// Follows the vLLM-Ascend "Kimi K3 MoE Forward Insight" page, section
// "Stage 4: Dispatch, MLP, Combine", AllGather row: the combine restores token
// order and applies the routing probabilities; the shared expert's output is
// added to the routed output ("Forward Skeleton", shared experts).
//
// out[t] = bf16( sum_{j=0..k-1} w[t,j] * y[flat_to_row[t*k+j]] + shared_y[t] )
// with y and shared_y in fp32, accumulated in fp32 with fused multiply-adds
// in the fixed order j = 0..k-1, then the shared term; one CTA per token,
// each thread owns 8 consecutive outputs (two 16-byte loads per expert row,
// one 16-byte bf16 store).  Memory bound: reads (k+1)*H*4 bytes and writes
// H*2 bytes per token.
#include "common.cuh"
#include "internal.h"

namespace gbmoe {
namespace {

constexpr int kMaxK = 32;

__device__ __forceinline__ void fma8(float (&acc)[8], float w, const float4& a, const float4& b) {
    acc[0] = __fmaf_rn(w, a.x, acc[0]);
    acc[1] = __fmaf_rn(w, a.y, acc[1]);
    acc[2] = __fmaf_rn(w, a.z, acc[2]);
    acc[3] = __fmaf_rn(w, a.w, acc[3]);
    acc[4] = __fmaf_rn(w, b.x, acc[4]);
    acc[5] = __fmaf_rn(w, b.y, acc[5]);
    acc[6] = __fmaf_rn(w, b.z, acc[6]);
    acc[7] = __fmaf_rn(w, b.w, acc[7]);
}

__global__ void __launch_bounds__(128) combine_kernel(const float4* __restrict__ y,
                                                      const int32_t* __restrict__ flat_to_row,
                                                      const float* __restrict__ weights,
                                                      const float4* __restrict__ shared_y, int k,
                                                      int H, uint4* __restrict__ out) {
    __shared__ int64_t rows[kMaxK];
    __shared__ float wts[kMaxK];
    const int t = blockIdx.x;
    if (threadIdx.x < k) {
        rows[threadIdx.x] = flat_to_row[static_cast<int64_t>(t) * k + threadIdx.x];
        wts[threadIdx.x] = weights[static_cast<int64_t>(t) * k + threadIdx.x];
    }
    __syncthreads();
    const int v4_per_row = H / 4;  // float4 per fp32 row
    for (int v = threadIdx.x; v < H / 8; v += blockDim.x) {
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const float4* src = y + rows[j] * v4_per_row + 2 * v;
            fma8(acc, wts[j], __ldg(src), __ldg(src + 1));
        }
        if (shared_y) {
            const float4* src = shared_y + static_cast<int64_t>(t) * v4_per_row + 2 * v;
            const float4 a = __ldg(src), b = __ldg(src + 1);
            acc[0] = __fadd_rn(acc[0], a.x);
            acc[1] = __fadd_rn(acc[1], a.y);
            acc[2] = __fadd_rn(acc[2], a.z);
            acc[3] = __fadd_rn(acc[3], a.w);
            acc[4] = __fadd_rn(acc[4], b.x);
            acc[5] = __fadd_rn(acc[5], b.y);
            acc[6] = __fadd_rn(acc[6], b.z);
            acc[7] = __fadd_rn(acc[7], b.w);
        }
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            o[q] = static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * q])) |
                   (static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * q + 1])) << 16);
        out[static_cast<int64_t>(t) * (H / 8) + v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_combine(const float* y, const int32_t* flat_to_row, const float* weights,
                           const float* shared_y, int T, int k, int H, uint16_t* out,
                           const DevCtx& ctx, cudaStream_t s) {
    (void)ctx;
    if (T == 0) return cudaSuccess;
    combine_kernel<<<T, 128, 0, s>>>(reinterpret_cast<const float4*>(y), flat_to_row, weights,
                                     reinterpret_cast<const float4*>(shared_y), k, H,
                                     reinterpret_cast<uint4*>(out));
    return cudaGetLastError();
}

}  // namespace gbmoe
