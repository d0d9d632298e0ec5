// Weighted combine / unpermute.
//
// Follows the vLLM-Ascend "Kimi K3 MoE Forward Insight" page, section
// "Stage 4: Dispatch, MLP, Combine", AllGather row: the combine restores token
// order and applies the routing probabilities; the shared expert's output is
// added to the routed output ("Forward Skeleton", shared experts).
//
// out[t] = bf16( sum_{j=0..k-1} w[t,j] * y[flat_to_row[t*k+j]] + shared_y[t] )
// accumulated in fp32 with fused multiply-adds in the fixed order j = 0..k-1,
// then the shared term; one CTA per token, 16-byte vector loads (gather of
// the k expert rows) and stores.  Memory bound: reads k*H*2 + H*2 bytes and
// writes H*2 bytes per token.
#include "common.cuh"
#include "internal.h"

namespace gbmoe {
namespace {

constexpr int kMaxK = 32;

__global__ void __launch_bounds__(128) combine_kernel(const uint4* __restrict__ y,
                                                      const int32_t* __restrict__ flat_to_row,
                                                      const float* __restrict__ weights,
                                                      const uint4* __restrict__ shared_y, int k,
                                                      int vec_per_row, uint4* __restrict__ out) {
    __shared__ int64_t rows[kMaxK];
    __shared__ float wts[kMaxK];
    const int t = blockIdx.x;
    if (threadIdx.x < k) {
        rows[threadIdx.x] = flat_to_row[static_cast<int64_t>(t) * k + threadIdx.x];
        wts[threadIdx.x] = weights[static_cast<int64_t>(t) * k + threadIdx.x];
    }
    __syncthreads();
    for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x) {
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const uint4 pk = __ldg(y + rows[j] * vec_per_row + v);
            const uint32_t wd[4] = {pk.x, pk.y, pk.z, pk.w};
            const float wj = wts[j];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[2 * q] = __fmaf_rn(wj, __uint_as_float(wd[q] << 16), acc[2 * q]);
                acc[2 * q + 1] = __fmaf_rn(wj, __uint_as_float(wd[q] & 0xffff0000u), acc[2 * q + 1]);
            }
        }
        if (shared_y) {
            const uint4 pk = __ldg(shared_y + static_cast<int64_t>(t) * vec_per_row + v);
            const uint32_t wd[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[2 * q] = __fadd_rn(acc[2 * q], __uint_as_float(wd[q] << 16));
                acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], __uint_as_float(wd[q] & 0xffff0000u));
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            o[q] = static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * q])) |
                   (static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * q + 1])) << 16);
        out[static_cast<int64_t>(t) * vec_per_row + v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_combine(const uint16_t* y, const int32_t* flat_to_row, const float* weights,
                           const uint16_t* shared_y, int T, int k, int H, uint16_t* out,
                           const DevCtx& ctx, cudaStream_t s) {
    (void)ctx;
    if (T == 0) return cudaSuccess;
    combine_kernel<<<T, 128, 0, s>>>(reinterpret_cast<const uint4*>(y), flat_to_row, weights,
                                     reinterpret_cast<const uint4*>(shared_y), k, H / 8,
                                     reinterpret_cast<uint4*>(out));
    return cudaGetLastError();
}

}  // namespace gbmoe
