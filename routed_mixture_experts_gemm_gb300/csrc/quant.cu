// FP8 (OCP E4M3) row quantization for the FP8 expert path.
//
// Follows the vLLM-Ascend "Kimi K3 MoE Forward Insight" page, section
// "Stage 4: Dispatch, MLP, Combine" (quantized paths: W8A8FP).  Each row gets
// one fp32 scale s = amax / 448 (1 for an all-zero row) and the codes
// q = e4m3(x / s): IEEE division, then the hardware conversion with round to
// nearest even and saturation to +-448 (cvt.rn.satfinite.e4m3x2.f32).  One
// warp per row: a max-reduction (exact in any order), then 16-byte loads of 8
// bf16 values turned into 8 codes per lane and step.
#include "common.cuh"
#include "internal.h"

namespace gbmoe {
namespace {

constexpr int kQuantWarps = 8;

// two fp32 values -> two E4M3 codes, the first in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

__global__ void __launch_bounds__(32 * kQuantWarps) quantize_rows_kernel(
    const uint4* __restrict__ x, int64_t n, int K, uint2* __restrict__ q, float* __restrict__ s) {
    const int lane = threadIdx.x & 31;
    const int v8 = K / 8;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kQuantWarps + (threadIdx.x >> 5); r < n;
         r += static_cast<int64_t>(gridDim.x) * kQuantWarps) {
        const uint4* row = x + r * v8;
        float amax = 0.0f;
        for (int i = lane; i < v8; i += 32) {
            const uint4 v = row[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
                amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xffff0000u)));
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        if (lane == 0) s[r] = sc;
        uint2* qrow = q + r * v8;
        for (int i = lane; i < v8; i += 32) {
            const uint4 v = row[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t c[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                c[j] = e4m3x2(__fdiv_rn(__uint_as_float(w[j] << 16), sc),
                              __fdiv_rn(__uint_as_float(w[j] & 0xffff0000u), sc));
            qrow[i] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
        }
    }
}

}  // namespace

cudaError_t launch_quantize_rows(const uint16_t* x, int64_t n, int K, uint8_t* q, float* s,
                                 const DevCtx& ctx, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int64_t want = (n + kQuantWarps - 1) / kQuantWarps;
    const int grid = static_cast<int>(want < 16L * ctx.num_sms ? want : 16L * ctx.num_sms);
    quantize_rows_kernel<<<grid, 32 * kQuantWarps, 0, st>>>(
        reinterpret_cast<const uint4*>(x), n, K, reinterpret_cast<uint2*>(q), s);
    return cudaGetLastError();
}

}  // namespace gbmoe
