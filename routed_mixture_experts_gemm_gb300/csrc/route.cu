// Router scoring and expert selection.
//
// Follows the vLLM-Ascend "Kimi K3 MoE Forward Insight" page, section
// "Stage 2: Select Experts" (softmax / sigmoid / sqrtsoftplus scoring, hash
// routing through tid2eid, grouped top-k, correction bias, top-k,
// renormalisation, routed scaling; settings listed under "Runner
// Initialization") and section "Stage 4: Dispatch, MLP, Combine" step 2
// (logical topk_ids mapped through log2phy).
//
// Reproducibility: the router logit of (t, e) is accumulated in a fixed fp32
// order -- 32 partial sums, partial j takes h = j, j+32, ... ascending with a
// fused multiply-add, then the pairwise tree over the 32 partials (a warp
// xor-butterfly computes exactly that tree) -- and the scoring functions are
// this library's own (exp by Cody-Waite reduction plus the degree-7 Taylor
// polynomial; log1p by the atanh series; IEEE division and sqrt).  With every
// step written with explicitly rounded intrinsics, expert ids and routing
// weights are bit-for-bit reproducible by any implementation of the same
// definitions.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace gbmoe {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();

// ------------------------------------------------ elementary functions
// exp(x) = 2^n e^r, x = n ln2 + r: ln2 split into a 16-significant-bit head
// (n * head exact for |n| <= 256) and an fp32 tail; e^r by the Taylor
// polynomial to degree 7 (Horner, fused multiply-adds); 2^n applied as two
// exact power-of-two scalings.  Results below 2^-126 flush to zero.
__device__ __forceinline__ float pow2_int(int n) { return __int_as_float((n + 127) << 23); }

__device__ __forceinline__ float pinned_exp(float x) {
    if (x != x) return x;
    if (x > 88.72283935546875f) return __int_as_float(0x7f800000);
    if (x < -87.33654022216797f) return 0.0f;
    const float nf = rintf(__fmul_rn(x, 1.44269502162933349609375f));
    const int n = static_cast<int>(nf);
    float r = __fmaf_rn(-nf, 0.693145751953125f, x);
    r = __fmaf_rn(-nf, 1.428606820309417e-06f, r);
    float p = 1.0f / 5040.0f;
    p = __fmaf_rn(p, r, 1.0f / 720.0f);
    p = __fmaf_rn(p, r, 1.0f / 120.0f);
    p = __fmaf_rn(p, r, 1.0f / 24.0f);
    p = __fmaf_rn(p, r, 1.0f / 6.0f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int n1 = n / 2;
    const int n2 = n - n1;
    return __fmul_rn(__fmul_rn(p, pow2_int(n1)), pow2_int(n2));
}

// log(1+y), 0 <= y <= 1: 2 atanh(z), z = y/(2+y), odd series to z^17/17.
__device__ __forceinline__ float pinned_log1p(float y) {
    const float z = __fdiv_rn(y, __fadd_rn(2.0f, y));
    const float w = __fmul_rn(z, z);
    float q = 1.0f / 17.0f;
    q = __fmaf_rn(q, w, 1.0f / 15.0f);
    q = __fmaf_rn(q, w, 1.0f / 13.0f);
    q = __fmaf_rn(q, w, 1.0f / 11.0f);
    q = __fmaf_rn(q, w, 1.0f / 9.0f);
    q = __fmaf_rn(q, w, 1.0f / 7.0f);
    q = __fmaf_rn(q, w, 1.0f / 5.0f);
    q = __fmaf_rn(q, w, 1.0f / 3.0f);
    const float a = __fmaf_rn(__fmul_rn(z, w), q, z);
    return __fmul_rn(2.0f, a);
}

__device__ __forceinline__ float pinned_sigmoid(float l) {
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, pinned_exp(-l)));
}

__device__ __forceinline__ float pinned_sqrtsoftplus(float l) {
    const float sp = __fadd_rn(fmaxf(l, 0.0f), pinned_log1p(pinned_exp(-fabsf(l))));
    return __fsqrt_rn(sp);
}

__device__ __forceinline__ float warp_sum_tree(float v) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, s));
    return v;
}

// ------------------------------------------------------ router logits
// Block = 16 warps arranged 4 (tokens) x 4 (experts); warp tile WT x WE;
// lane j owns h = j, j+32, ... for every (t, e) of its warp tile.
template <int WT, int WE>
__global__ void __launch_bounds__(512) router_logits_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ w, const float* __restrict__ bias,
    int T, int E, int H, float* __restrict__ logits) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * (4 * WT) + (warp >> 2) * WT;
    const int e0 = blockIdx.y * (4 * WE) + (warp & 3) * WE;
    if (t0 >= T || e0 >= E) return;
    int xo[WT], wo[WE];
#pragma unroll
    for (int i = 0; i < WT; ++i) xo[i] = min(t0 + i, T - 1) * H;
#pragma unroll
    for (int j = 0; j < WE; ++j) wo[j] = min(e0 + j, E - 1) * H;
    float acc[WT][WE];
#pragma unroll
    for (int i = 0; i < WT; ++i)
#pragma unroll
        for (int j = 0; j < WE; ++j) acc[i][j] = 0.0f;
    for (int h = lane; h < H; h += 32) {
        float xv[WT], wv[WE];
#pragma unroll
        for (int i = 0; i < WT; ++i) xv[i] = bf16_bits_to_f32(__ldg(x + xo[i] + h));
#pragma unroll
        for (int j = 0; j < WE; ++j) wv[j] = __ldg(w + wo[j] + h);
#pragma unroll
        for (int i = 0; i < WT; ++i)
#pragma unroll
            for (int j = 0; j < WE; ++j) acc[i][j] = __fmaf_rn(xv[i], wv[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < WT; ++i)
#pragma unroll
        for (int j = 0; j < WE; ++j) {
            const float v = warp_sum_tree(acc[i][j]);
            const int t = t0 + i, e = e0 + j;
            if (lane == ((i * WE + j) & 31) && t < T && e < E)
                logits[static_cast<size_t>(t) * E + e] = bias ? __fadd_rn(v, __ldg(bias + e)) : v;
        }
}

// Shared-memory tiled variant (H % 32 == 0, 16-byte aligned x and w).  A
// block of 8 warps covers BT = 8*WT tokens x BE = 8*WE experts; H is walked
// in chunks of 256 (eight h-steps of 32 lanes), double-buffered: router
// weight rows arrive by cp.async in their natural layout (lane j reads
// w[e][h0 + 32 i + j], consecutive words), token rows are transposed on the
// way in so lane j finds its eight values x[t][h0 + j + 32 i], i = 0..7, in
// one 16-byte word.  Lane j still accumulates h = j, j+32, ... ascending, so
// the result is the same pinned sum as router_logits_kernel.
constexpr int kChunk = 256;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Two fp32 fused multiply-adds in one instruction (fma.rn.f32x2): each half
// is an ordinary round-to-nearest fma, so results are those of two fmaf.
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
    return (static_cast<unsigned long long>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}

// Block = 8 warps covering BT = 8*WT tokens x BE = 8*WE experts; each warp
// owns 8 tokens (four pairs, one per 64-bit accumulator) x 8 experts.  Token
// chunks are stored pair-interleaved: for token pair p, lane j and h-step i
// one 32-bit word holds the two tokens' bf16 x[h0 + j + 32 i]; a lane's 8
// words (32 B) are two 16-byte halves, swapped for lanes with bit 2 set so
// that the quarter-warp reading them hits distinct banks.
template <int WT, int WE>
__global__ void __launch_bounds__(256, 2) router_logits_tiled_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ w, const float* __restrict__ bias,
    int T, int E, int H, float* __restrict__ logits) {
    constexpr int TP = 4, TE = 8;          // token pairs and experts per warp
    constexpr int BT = 2 * TP * WT, BE = TE * WE;
    constexpr int BP = BT / 2;             // token pairs per block
    constexpr int XV = BP * (kChunk / 8);  // (pair, 8-h) units per chunk
    constexpr int XR = (XV + 255) / 256;   // per thread
    constexpr int WV = BE * (kChunk / 4);  // 16-byte weight vectors per chunk
    static_assert(WT * WE == 8, "8 warps per block");
    extern __shared__ __align__(16) uint8_t route_smem[];
    // xs: [2][BP][32 lanes][2 halves][4 words]; ws: [2][BE][kChunk] fp32
    uint32_t* xs = reinterpret_cast<uint32_t*>(route_smem);
    auto ws = reinterpret_cast<float(*)[BE][kChunk]>(route_smem + 2 * BP * 32 * 8 * 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wt = warp / WE, we = warp % WE;
    const int t0 = blockIdx.x * BT, e0 = blockIdx.y * BE;
    const int nc = (H + kChunk - 1) / kChunk;

    uint4 xa[XR], xb[XR];
    auto load_x = [&](int c) {
        const int h0 = c * kChunk;
#pragma unroll
        for (int r = 0; r < XR; ++r) {
            const int idx = tid + r * 256;
            xa[r] = xb[r] = make_uint4(0, 0, 0, 0);
            if (idx < XV) {
                const int pr = idx / (kChunk / 8), q = idx % (kChunk / 8);
                const int t = t0 + 2 * pr, h = h0 + 8 * q;
                if (h < H) {
                    if (t < T)
                        xa[r] = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H + h));
                    if (t + 1 < T)
                        xb[r] = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t + 1) * H + h));
                }
            }
        }
    };
    auto store_x = [&](int buf) {
#pragma unroll
        for (int r = 0; r < XR; ++r) {
            const int idx = tid + r * 256;
            if (idx < XV) {
                const int pr = idx / (kChunk / 8), q = idx % (kChunk / 8);
                const int i = q >> 2, j0 = (q & 3) * 8;
                const uint32_t va[4] = {xa[r].x, xa[r].y, xa[r].z, xa[r].w};
                const uint32_t vb[4] = {xb[r].x, xb[r].y, xb[r].z, xb[r].w};
                uint32_t* dst = xs + (buf * BP + pr) * 256;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int j = j0 + jj;
                    const uint32_t lo = (jj & 1) ? (va[jj >> 1] >> 16) : (va[jj >> 1] & 0xffffu);
                    const uint32_t hi = (jj & 1) ? (vb[jj >> 1] >> 16) : (vb[jj >> 1] & 0xffffu);
                    const int half = (i >> 2) ^ ((j >> 2) & 1);
                    dst[j * 8 + half * 4 + (i & 3)] = lo | (hi << 16);
                }
            }
        }
    };
    auto load_w = [&](int c, int buf) {
        const int h0 = c * kChunk;
        for (int idx = tid; idx < WV; idx += 256) {
            const int row = idx / (kChunk / 4), q = idx % (kChunk / 4);
            const int e = e0 + row, h = h0 + 4 * q;
            if (e < E && h < H) cp_async16(&ws[buf][row][4 * q], w + static_cast<size_t>(e) * H + h);
        }
        cp_async_commit();
    };

    unsigned long long acc[TP][TE];
#pragma unroll
    for (int a = 0; a < TP; ++a)
#pragma unroll
        for (int b = 0; b < TE; ++b) acc[a][b] = 0ull;

    load_w(0, 0);
    load_x(0);
    store_x(0);
    cp_async_wait_all();
    __syncthreads();
    const int sw = (lane >> 2) & 1;
    for (int c = 0; c < nc; ++c) {
        const int buf = c & 1;
        if (c + 1 < nc) {
            load_w(c + 1, buf ^ 1);
            load_x(c + 1);
        }
        const int n_i = min(8, (H - c * kChunk) / 32);
        uint32_t xp[TP][8];  // word i of token pair a: (x[t][h], x[t+1][h]), h = h0 + lane + 32 i
#pragma unroll
        for (int a = 0; a < TP; ++a) {
            const uint32_t* src = xs + (buf * BP + wt * TP + a) * 256 + lane * 8;
            const uint4 v0 = *reinterpret_cast<const uint4*>(src + 4 * sw);
            const uint4 v1 = *reinterpret_cast<const uint4*>(src + 4 * (sw ^ 1));
            xp[a][0] = v0.x; xp[a][1] = v0.y; xp[a][2] = v0.z; xp[a][3] = v0.w;
            xp[a][4] = v1.x; xp[a][5] = v1.y; xp[a][6] = v1.z; xp[a][7] = v1.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < n_i) {
                unsigned long long wd[TE];
#pragma unroll
                for (int b = 0; b < TE; ++b) {
                    const float wv = ws[buf][we * TE + b][32 * i + lane];
                    wd[b] = pack2(wv, wv);
                }
#pragma unroll
                for (int a = 0; a < TP; ++a) {
                    const uint32_t pk = xp[a][i];
                    const unsigned long long xv =
                        pack2(__uint_as_float(pk << 16), __uint_as_float(pk & 0xffff0000u));
#pragma unroll
                    for (int b = 0; b < TE; ++b) acc[a][b] = fma2(xv, wd[b], acc[a][b]);
                }
            }
        }
        if (c + 1 < nc) store_x(buf ^ 1);
        cp_async_wait_all();
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < TP; ++a)
#pragma unroll
        for (int b = 0; b < TE; ++b)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float part = __uint_as_float(static_cast<uint32_t>(acc[a][b] >> (32 * u)));
                const float v = warp_sum_tree(part);
                const int t = t0 + wt * 2 * TP + 2 * a + u, e = e0 + we * TE + b;
                if (lane == ((a * 2 * TE + u * TE + b) & 31) && t < T && e < E)
                    logits[static_cast<size_t>(t) * E + e] = bias ? __fadd_rn(v, __ldg(bias + e)) : v;
            }
}

// ----------------------------------------------------------- selection
struct Cand {
    bool ok;
    float v;
    int idx;
};
__device__ __forceinline__ bool better(const Cand& a, const Cand& b) {
    return a.ok && (!b.ok || a.v > b.v || (a.v == b.v && a.idx < b.idx));
}
__device__ __forceinline__ Cand warp_argmax(Cand c) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        Cand o;
        o.ok = __shfl_xor_sync(0xffffffffu, static_cast<int>(c.ok), s) != 0;
        o.v = __shfl_xor_sync(0xffffffffu, c.v, s);
        o.idx = __shfl_xor_sync(0xffffffffu, c.idx, s);
        if (better(o, c)) c = o;
    }
    return c;
}

template <int EPL>
__device__ __forceinline__ float pick(const float (&a)[EPL], int idx) {
    float v = 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
        if (i == idx) v = a[i];
    return v;
}

// One warp per token.  Lane L holds experts e = L + 32 i, i < EPL.
template <int EPL>
__global__ void __launch_bounds__(256) route_select_kernel(const RouteArgs a, int* status) {
    const int lane = threadIdx.x & 31;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= a.T) return;
    const gbmoe_route_cfg& c = a.cfg;
    const int E = c.E_log, k = c.top_k;
    const float* lrow = a.logits + static_cast<size_t>(t) * E;

    float sc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        sc[i] = e < E ? lrow[e] : 0.0f;
    }
    if (c.scoring == GBMOE_SCORE_SOFTMAX) {
        float m = kNegInf;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (lane + 32 * i < E) m = fmaxf(m, sc[i]);
#pragma unroll
        for (int s = 16; s >= 1; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (lane + 32 * i < E) {
                sc[i] = pinned_exp(__fsub_rn(sc[i], m));
                part = __fadd_rn(part, sc[i]);
            }
        const float S = warp_sum_tree(part);
#pragma unroll
        for (int i = 0; i < EPL; ++i) sc[i] = __fdiv_rn(sc[i], S);
    } else if (c.scoring == GBMOE_SCORE_SIGMOID) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) sc[i] = pinned_sigmoid(sc[i]);
    } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) sc[i] = pinned_sqrtsoftplus(sc[i]);
    }

    int my_e = 0;        // slot `lane` (lane < k): chosen logical expert
    float my_s = 0.0f;   // and its unbiased score
    if (c.use_hash) {
        int v = a.input_ids[t];
        if (v < 0 || static_cast<int64_t>(v) >= a.tid2eid_rows) {
            record_error(status, GBMOE_ERR_DEVICE);
            v = 0;
        }
        int e = 0;
        if (lane < k) {
            e = a.tid2eid[static_cast<int64_t>(v) * k + lane];
            if (e < 0 || e >= E) {
                record_error(status, GBMOE_ERR_DEVICE);
                e = 0;
            }
        }
        for (int j = 0; j < k; ++j) {
            const int ej = __shfl_sync(0xffffffffu, e, j);
            const float s = __shfl_sync(0xffffffffu, pick<EPL>(sc, ej >> 5), ej & 31);
            if (lane == j) {
                my_e = ej;
                my_s = s;
            }
        }
    } else {
        float sel[EPL];
        uint32_t allowed = 0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            sel[i] = kNegInf;
            if (e < E) {
                sel[i] = a.corr_bias ? __fadd_rn(sc[i], __ldg(a.corr_bias + e)) : sc[i];
                allowed |= 1u << i;
            }
        }
        if (c.n_group > 1) {
            const int G = c.n_group, gs = E / G;
            float my_g = 0.0f;
            for (int g = 0; g < G; ++g) {
                float b1 = kNegInf, b2 = kNegInf;
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const int e = lane + 32 * i;
                    if (e < E && e / gs == g) {
                        const float v = sel[i];
                        if (v > b1) {
                            b2 = b1;
                            b1 = v;
                        } else if (v > b2) {
                            b2 = v;
                        }
                    }
                }
#pragma unroll
                for (int s = 16; s >= 1; s >>= 1) {
                    const float o1 = __shfl_xor_sync(0xffffffffu, b1, s);
                    const float o2 = __shfl_xor_sync(0xffffffffu, b2, s);
                    const float n2 = fmaxf(fminf(b1, o1), fmaxf(b2, o2));
                    b1 = fmaxf(b1, o1);
                    b2 = n2;
                }
                const float gsc =
                    (c.group_score == GBMOE_GROUP_TOP2SUM && gs > 1) ? __fadd_rn(b1, b2) : b1;
                if (lane == g) my_g = gsc;
            }
            uint32_t keep = 0;
            for (int r = 0; r < c.topk_group; ++r) {
                Cand cd{lane < G && !((keep >> lane) & 1u), my_g, lane};
                cd = warp_argmax(cd);
                keep |= 1u << cd.idx;
            }
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !((keep >> (e / gs)) & 1u)) allowed &= ~(1u << i);
            }
        }
        for (int j = 0; j < k; ++j) {
            Cand cd{false, 0.0f, 0};
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                if ((allowed >> i) & 1u) {
                    const Cand o{true, sel[i], lane + 32 * i};
                    if (better(o, cd)) cd = o;
                }
            }
            cd = warp_argmax(cd);
            const int be = cd.idx;
            if (lane == (be & 31)) allowed &= ~(1u << (be >> 5));
            const float s = __shfl_sync(0xffffffffu, pick<EPL>(sc, be >> 5), be & 31);
            if (lane == j) {
                my_e = be;
                my_s = s;
            }
        }
    }

    float sum = 0.0f;
    for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, my_s, j));
    const float wgt = c.renormalize ? __fmul_rn(__fdiv_rn(my_s, sum), c.routed_scaling)
                                    : __fmul_rn(my_s, c.routed_scaling);
    if (lane < k) {
        int p = my_e;
        if (a.log2phy) {
            int n = a.replica_cnt[my_e];
            if (n < 1 || n > a.R_max) {
                record_error(status, GBMOE_ERR_DEVICE);
                n = 1;
            }
            p = a.log2phy[static_cast<int64_t>(my_e) * a.R_max + (t % n)];
            if (p < 0 || p >= c.E_phys) {
                record_error(status, GBMOE_ERR_DEVICE);
                p = 0;
            }
        }
        const size_t o = static_cast<size_t>(t) * k + lane;
        a.ids_log[o] = my_e;
        a.ids_phys[o] = p;
        a.weights[o] = wgt;
        if (a.counts) atomicAdd(a.counts + p, 1);
    }
}

__global__ void expert_counts_kernel(const int32_t* __restrict__ ids, int64_t n, int E_phys,
                                     int32_t* __restrict__ counts, int* status) {
    for (int64_t f = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; f < n;
         f += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int p = ids[f];
        if (p < 0 || p >= E_phys) {
            record_error(status, GBMOE_ERR_DEVICE);
            continue;
        }
        atomicAdd(counts + p, 1);
    }
}

template <int WT, int WE>
constexpr int tiled_smem_bytes() {
    return 2 * (4 * WT) * 32 * 8 * 4 + 2 * (8 * WE) * kChunk * 4;
}

template <int WT, int WE>
cudaError_t launch_tiled(const RouteArgs& a, const DevCtx& ctx, cudaStream_t s) {
    static bool attr_done[64];
    static std::mutex mu;
    constexpr int smem = tiled_smem_bytes<WT, WE>();
    {
        std::lock_guard<std::mutex> lk(mu);
        if (ctx.device < 0 || ctx.device >= 64 || !attr_done[ctx.device]) {
            cudaError_t e = cudaFuncSetAttribute(router_logits_tiled_kernel<WT, WE>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            if (ctx.device >= 0 && ctx.device < 64) attr_done[ctx.device] = true;
        }
    }
    dim3 grid((a.T + 8 * WT - 1) / (8 * WT), (a.cfg.E_log + 8 * WE - 1) / (8 * WE));
    router_logits_tiled_kernel<WT, WE><<<grid, 256, smem, s>>>(a.x, a.w_router, a.router_bias, a.T,
                                                               a.cfg.E_log, a.H, a.logits);
    return cudaGetLastError();
}

template <int EPL>
cudaError_t launch_select(const RouteArgs& a, const DevCtx& ctx, cudaStream_t s) {
    const int warps_per_block = 8;
    const int blocks = (a.T + warps_per_block - 1) / warps_per_block;
    route_select_kernel<EPL><<<blocks, 32 * warps_per_block, 0, s>>>(a, ctx.status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, const DevCtx& ctx, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    const int E = a.cfg.E_log;
    const bool tiled = a.w_router && a.H % 32 == 0 &&
                       (reinterpret_cast<uintptr_t>(a.x) & 15u) == 0 &&
                       (reinterpret_cast<uintptr_t>(a.w_router) & 15u) == 0;
    if (tiled) {
        // few tokens: one token tile of 8, 64 experts per block; many tokens:
        // 16 x 32 tiles (more blocks, router weight re-read less often)
        const cudaError_t err =
            static_cast<long>((a.T + 15) / 16) * ((E + 31) / 32) >= 4L * ctx.num_sms
                ? launch_tiled<2, 4>(a, ctx, s)
                : launch_tiled<1, 8>(a, ctx, s);
        if (err != cudaSuccess) return err;
    } else if (a.w_router) {
        // small batches: thin token tiles so the grid still covers the GPU
        const long big_blocks = ((a.T + 31) / 32) * static_cast<long>((E + 31) / 32);
        if (big_blocks >= 2L * ctx.num_sms) {
            dim3 grid((a.T + 31) / 32, (E + 31) / 32);
            router_logits_kernel<8, 8><<<grid, 512, 0, s>>>(a.x, a.w_router, a.router_bias, a.T,
                                                            E, a.H, a.logits);
        } else {
            dim3 grid((a.T + 7) / 8, (E + 31) / 32);
            router_logits_kernel<2, 8><<<grid, 512, 0, s>>>(a.x, a.w_router, a.router_bias, a.T,
                                                            E, a.H, a.logits);
        }
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    const int epl = (E + 31) / 32;
    if (epl <= 1) return launch_select<1>(a, ctx, s);
    if (epl <= 2) return launch_select<2>(a, ctx, s);
    if (epl <= 4) return launch_select<4>(a, ctx, s);
    if (epl <= 8) return launch_select<8>(a, ctx, s);
    if (epl <= 12) return launch_select<12>(a, ctx, s);
    if (epl <= 16) return launch_select<16>(a, ctx, s);
    if (epl <= 24) return launch_select<24>(a, ctx, s);
    return launch_select<32>(a, ctx, s);
}

cudaError_t launch_expert_counts(const int32_t* ids, int64_t n, int E_phys, int32_t* counts,
                                 const DevCtx& ctx, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int64_t want = (n + 255) / 256;
    const int blocks = static_cast<int>(std::min<int64_t>(want, 4L * ctx.num_sms));
    expert_counts_kernel<<<blocks, 256, 0, s>>>(ids, n, E_phys, counts, ctx.status);
    return cudaGetLastError();
}

}  // namespace gbmoe
