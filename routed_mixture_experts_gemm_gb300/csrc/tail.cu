// Post-MoE tail of a latent MoE on one GPU.
//
// Follows the NVIDIA vLLM LatentMoERunner page, tier 1 of the latent tail
// ("_overlap_allreduce_tail"): the routed output lives in a latent space; the
// tail normalises it (standard RMSNorm), up-projects it to the hidden size
// with a replicated weight and adds the shared-expert output.  With one rank
// the page's all-reduces are identities, so what remains is
//   out = bf16(rmsnorm(latent) . up_proj^T + shared).
//
// rmsnorm_kernel: one warp per token; lane j accumulates v_l^2 for
// l = j, j+32, ... with fused multiply-adds, the warp xor-butterfly is the
// pairwise tree over the 32 partials, r = 1 / sqrt(s / L + eps) with IEEE
// division and square root, z_l = bf16((v_l * r) * w_l): bit-for-bit the
// pinned definition.  The up-projection is the grouped GEMM (one group, the
// weight rows as M, fp32 out), and add_round_kernel adds the shared output
// and rounds to bf16.
#include "common.cuh"
#include "internal.h"

namespace gbmoe {
namespace {

__device__ __forceinline__ float warp_sum_tree_f(float v) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, s));
    return v;
}

constexpr int kNormWarps = 8;

__global__ void __launch_bounds__(32 * kNormWarps) rmsnorm_kernel(
    const uint16_t* __restrict__ v, int T, int L, const uint16_t* __restrict__ w, float eps,
    uint16_t* __restrict__ z) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kNormWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const uint16_t* row = v + static_cast<size_t>(t) * L;
    float p = 0.0f;
    for (int l = lane; l < L; l += 32) {
        const float x = bf16_bits_to_f32(row[l]);
        p = __fmaf_rn(x, x, p);
    }
    const float s = warp_sum_tree_f(p);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(s, static_cast<float>(L)), eps)));
    uint16_t* out = z + static_cast<size_t>(t) * L;
    for (int l = lane; l < L; l += 32)
        out[l] = f32_to_bf16_bits(
            __fmul_rn(__fmul_rn(bf16_bits_to_f32(row[l]), r), bf16_bits_to_f32(w[l])));
}

// out = bf16(y + shared), 8 outputs per thread (shared may be null).
__global__ void __launch_bounds__(256) add_round_kernel(const float4* __restrict__ y,
                                                        const uint4* __restrict__ shared,
                                                        int64_t n8, uint4* __restrict__ out) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 a = y[2 * i], b = y[2 * i + 1];
        float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        if (shared) {
            const uint4 sh = shared[i];
            const uint32_t s4[4] = {sh.x, sh.y, sh.z, sh.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                v[2 * q] = __fadd_rn(v[2 * q], __uint_as_float(s4[q] << 16));
                v[2 * q + 1] = __fadd_rn(v[2 * q + 1], __uint_as_float(s4[q] & 0xffff0000u));
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            o[q] = static_cast<uint32_t>(f32_to_bf16_bits(v[2 * q])) |
                   (static_cast<uint32_t>(f32_to_bf16_bits(v[2 * q + 1])) << 16);
        out[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

size_t latent_tail_ws_bytes(int T, int L, int Hm) {
    const size_t zb = ((static_cast<size_t>(T) * L * 2 + 255) / 256) * 256;
    return zb + static_cast<size_t>(T) * Hm * 4;
}

int launch_latent_tail(const uint16_t* latent, int T, int L, const uint16_t* norm_w, float eps,
                       const uint16_t* up_proj, int Hm, const uint16_t* shared, uint16_t* out,
                       void* ws, const DevCtx& ctx, cudaStream_t s) {
    if (T == 0) return GBMOE_OK;
    const size_t zb = ((static_cast<size_t>(T) * L * 2 + 255) / 256) * 256;
    uint16_t* z = static_cast<uint16_t*>(ws);
    float* y = reinterpret_cast<float*>(static_cast<char*>(ws) + zb);
    const uint16_t* rows = latent;
    if (norm_w) {
        rmsnorm_kernel<<<(T + kNormWarps - 1) / kNormWarps, 32 * kNormWarps, 0, s>>>(
            latent, T, L, norm_w, eps, z);
        if (cudaGetLastError() != cudaSuccess) return GBMOE_ERR_CUDA;
        rows = z;
    }
    // y[t, h] = sum_l rows[t, l] up_proj[h, l]: the grouped GEMM's down mode
    // with one group of T rows
    const int st = launch_gemm_down(rows, nullptr, 1, T, Hm, L, up_proj, y, ctx, s);
    if (st) return st;
    const int64_t n8 = static_cast<int64_t>(T) * Hm / 8;
    const int64_t want = (n8 + 255) / 256;
    const int grid = static_cast<int>(want < 8L * ctx.num_sms ? want : 8L * ctx.num_sms);
    add_round_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(y),
                                          reinterpret_cast<const uint4*>(shared), n8,
                                          reinterpret_cast<uint4*>(out));
    return cudaGetLastError() == cudaSuccess ? GBMOE_OK : GBMOE_ERR_CUDA;
}

}  // namespace gbmoe
