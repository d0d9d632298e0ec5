// Weighted combine / unpermute.
//
// Follows the vLLM-Ascend "Kimi K3 MoE Forward Insight" page, section
// "Stage 4: Dispatch, MLP, Combine", AllGather row: the combine restores token
// order and applies the routing probabilities; the shared expert's output is
// added to the routed output ("Forward Skeleton", shared experts).
//
// out[t] = bf16( sum_{j=0..k-1} w[t,j] * y[flat_to_row[t*k+j]] + shared_y[t] )
// with y and shared_y in fp32, accumulated in fp32 with fused multiply-adds
// in the fixed order j = 0..k-1, then the shared term.  Block (t, c) covers
// 1024 outputs of token t: each thread owns 8 consecutive outputs, issues the
// loads of up to 8 expert rows at once (two 16-byte loads each) and only then
// folds them in order, so a token costs one memory round trip per 8 experts.
// Memory bound: reads (k+1)*H*4 bytes and writes H*2 bytes per token.
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

constexpr int kCombineThreads = 128;
constexpr int kCombineGroup = 8;  // expert rows whose loads are in flight together

__device__ __forceinline__ float4 ld_stream(const float4* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// A row outside [0, n_rows) (the permutation marks a skipped id with -1)
// contributes nothing: its slot is neither read nor added, and the device
// status records the bad entry.
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    const float4* __restrict__ y, const int32_t* __restrict__ flat_to_row,
    const float* __restrict__ weights, const float4* __restrict__ shared_y, int k, int H,
    int64_t n_rows, uint4* __restrict__ out, int* status) {
    __shared__ int64_t rows[kMaxK];
    __shared__ float wts[kMaxK];
    const int t = blockIdx.x;
    if (threadIdx.x < k) {
        const int64_t r = flat_to_row[static_cast<int64_t>(t) * k + threadIdx.x];
        const bool ok = r >= 0 && r < n_rows;
        if (!ok && blockIdx.y == 0) record_error(status, GBMOE_ERR_DEVICE);
        rows[threadIdx.x] = ok ? r : -1;
        wts[threadIdx.x] = ok ? weights[static_cast<int64_t>(t) * k + threadIdx.x] : 0.0f;
    }
    __syncthreads();
    const int v = blockIdx.y * kCombineThreads + threadIdx.x;  // group of 8 outputs
    if (v >= H / 8) return;
    const int v4_per_row = H / 4;  // float4 per fp32 row
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += kCombineGroup) {
        float4 a[kCombineGroup], b[kCombineGroup];
#pragma unroll
        for (int g = 0; g < kCombineGroup; ++g) {
            if (j0 + g < k && rows[j0 + g] >= 0) {
                const float4* src = y + rows[j0 + g] * v4_per_row + 2 * v;
                a[g] = ld_stream(src);
                b[g] = ld_stream(src + 1);
            }
        }
#pragma unroll
        for (int g = 0; g < kCombineGroup; ++g)
            if (j0 + g < k && rows[j0 + g] >= 0) fma8(acc, wts[j0 + g], a[g], b[g]);
    }
    if (shared_y) {
        const float4* src = shared_y + static_cast<int64_t>(t) * v4_per_row + 2 * v;
        const float4 a = ld_stream(src), b = ld_stream(src + 1);
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

}  // namespace

cudaError_t launch_combine(const float* y, const int32_t* flat_to_row, const float* weights,
                           const float* shared_y, int T, int k, int H, uint16_t* out,
                           const DevCtx& ctx, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const dim3 grid(T, (H / 8 + kCombineThreads - 1) / kCombineThreads);
    combine_kernel<<<grid, kCombineThreads, 0, s>>>(
        reinterpret_cast<const float4*>(y), flat_to_row, weights,
        reinterpret_cast<const float4*>(shared_y), k, H, static_cast<int64_t>(T) * k,
        reinterpret_cast<uint4*>(out), ctx.status);
    return cudaGetLastError();
}

}  // namespace gbmoe
