// FP8 (OCP E4M3) row quantization for the FP8 expert path, and MX block
// quantization (E4M3 or E2M1 elements, UE8M0 block scales) for the MX path.
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
                c[j] = cvt_e4m3x2(__fdiv_rn(__uint_as_float(w[j] << 16), sc),
                              __fdiv_rn(__uint_as_float(w[j] & 0xffff0000u), sc));
            qrow[i] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
        }
    }
}

// ---- MX block scales: blocks of 32 consecutive elements of a row share one
// power-of-two scale 2^e (UE8M0 byte e + 127), e = floor(log2(amax)) - emax
// (emax 8 for E4M3, 2 for E2M1), clamped to [-127, 127], byte 127 for an
// all-zero block; elements v * 2^-e (exact) rounded to nearest even with
// saturation by the hardware conversions.  One thread per block.

// two fp32 values -> two E2M1 codes, the first in the low nibble
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint32_t d;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(d)
        : "f"(hi), "f"(lo));
    return d;
}

template <int FMT>
__global__ void __launch_bounds__(256) mx_quantize_kernel(const uint4* __restrict__ x,
                                                          int64_t blocks, uint4* __restrict__ q,
                                                          uint8_t* __restrict__ sc) {
    for (int64_t b = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; b < blocks;
         b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = x[b * 4 + i];
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
        float f[32];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            amax = fmaxf(amax, fmaxf(fabsf(f[2 * i]), fabsf(f[2 * i + 1])));
        }
        const int e = mx_block_exp(amax, FMT == kMxE2M1 ? 2 : 8);
        sc[b] = static_cast<uint8_t>(e + 127);
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
        if (FMT == kMxE2M1) {
            uint32_t c[4] = {0, 0, 0, 0};
#pragma unroll
            for (int i = 0; i < 16; ++i)
                c[i >> 2] |= e2m1x2(__fmul_rn(f[2 * i], inv), __fmul_rn(f[2 * i + 1], inv))
                             << (8 * (i & 3));
            q[b] = make_uint4(c[0], c[1], c[2], c[3]);
        } else {
            uint32_t c[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                c[i] = cvt_e4m3x2(__fmul_rn(f[4 * i], inv), __fmul_rn(f[4 * i + 1], inv)) |
                       (cvt_e4m3x2(__fmul_rn(f[4 * i + 2], inv), __fmul_rn(f[4 * i + 3], inv)) << 16);
            q[2 * b] = make_uint4(c[0], c[1], c[2], c[3]);
            q[2 * b + 1] = make_uint4(c[4], c[5], c[6], c[7]);
        }
    }
}

// MX weight scale bytes, row-major [rows, K/32] (as 32-bit words: the four
// K blocks of one 128-element K stage of a row) -> the tiled layout of the
// grouped GEMMs: for row block rb (128 rows) and K stage ks, 512 bytes at
// chunk rb * KS + ks whose 16-byte row r holds, in word j, the four scale
// bytes of row rb*128 + 32j + r -- the tensor-memory column order of the
// block-scaled MMA (lane r, column j).  One thread per 16-byte row.
__global__ void __launch_bounds__(256) mx_tile_scales_kernel(const uint32_t* __restrict__ rows_w,
                                                            int64_t n16, int ks_n,
                                                            uint4* __restrict__ tiled) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(i & 31);
        const int64_t chunk = i >> 5;
        const int ks = static_cast<int>(chunk % ks_n);
        const int64_t row0 = (chunk / ks_n) * 128 + r;
        uint4 o;
        o.x = rows_w[(row0 + 0) * ks_n + ks];
        o.y = rows_w[(row0 + 32) * ks_n + ks];
        o.z = rows_w[(row0 + 64) * ks_n + ks];
        o.w = rows_w[(row0 + 96) * ks_n + ks];
        tiled[i] = o;
    }
}

}  // namespace

cudaError_t launch_mx_tile_scales(const uint8_t* sf_rows, int64_t rows, int K, uint8_t* tiled,
                                  const DevCtx& ctx, cudaStream_t st) {
    const int ks_n = K / 128;
    const int64_t n16 = (rows / 128) * ks_n * 32;
    if (n16 == 0) return cudaSuccess;
    const int64_t want = (n16 + 255) / 256;
    const int grid = static_cast<int>(want < 16L * ctx.num_sms ? want : 16L * ctx.num_sms);
    mx_tile_scales_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint32_t*>(sf_rows), n16,
                                                ks_n, reinterpret_cast<uint4*>(tiled));
    return cudaGetLastError();
}

cudaError_t launch_mx_quantize(const uint16_t* x, int64_t n, int K, int fmt, uint8_t* q,
                               uint8_t* sc, const DevCtx& ctx, cudaStream_t st) {
    const int64_t blocks = n * (K / 32);
    if (blocks == 0) return cudaSuccess;
    const int64_t want = (blocks + 255) / 256;
    const int grid = static_cast<int>(want < 16L * ctx.num_sms ? want : 16L * ctx.num_sms);
    if (fmt == kMxE2M1)
        mx_quantize_kernel<kMxE2M1><<<grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(x),
                                                          blocks, reinterpret_cast<uint4*>(q), sc);
    else
        mx_quantize_kernel<kMxE4M3><<<grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(x),
                                                          blocks, reinterpret_cast<uint4*>(q), sc);
    return cudaGetLastError();
}

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
