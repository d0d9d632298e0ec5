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
// order -- 32 partial sums, partial j takes h = 2j, 2j+1, 64+2j, 65+2j, ...
// ascending with a fused multiply-add, then the pairwise tree over the 32
// partials (a warp xor-butterfly computes exactly that tree) -- and the
// scoring functions are
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
// Generic path (any H, any alignment).  Block = 16 warps arranged 4 (tokens)
// x 4 (experts); warp tile WT x WE; lane j owns partial j of every (t, e) of
// its warp tile: h = 2j, 2j+1, 64+2j, 65+2j, ... ascending.
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
    for (int h0 = 2 * lane; h0 < H; h0 += 64) {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int h = h0 + m;
            if (h < H) {
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
        }
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

// Hash routing with an elementwise score (sigmoid, sqrtsoftplus): the
// selection reads only the logits of each token's k hashed experts, so only
// those are computed -- each in the pinned order of the full router (lane j's
// partial over h = 2j, 2j+1, 64+2j, 65+2j, ... with fused multiply-adds, the
// pairwise tree over the 32 partials, the router bias added last), so the
// logits, ids and weights are those of the full computation bit for bit, for
// k / E of its work.  Block = one token, warp j = slot j (the token's x row
// is shared through L1).  Out-of-range token ids or table entries compute
// nothing here; the selection kernel records them.
__global__ void __launch_bounds__(32 * kMaxTopK) router_logits_hash_kernel(const RouteArgs a) {
    const int t = blockIdx.x, j = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.cfg.E_log, k = a.cfg.top_k, H = a.H;
    if (t >= a.T || j >= k) return;
    const int v = a.input_ids[t];
    if (v < 0 || static_cast<int64_t>(v) >= a.tid2eid_rows) return;
    const int e = a.tid2eid[static_cast<int64_t>(v) * k + j];
    if (e < 0 || e >= E) return;
    const uint16_t* xr = a.x + static_cast<size_t>(t) * H;
    const float* wr = a.w_router + static_cast<size_t>(e) * H;
    float acc = 0.0f;
    const bool pairs = (H & 1) == 0 && (reinterpret_cast<uintptr_t>(a.x) & 3u) == 0 &&
                       (reinterpret_cast<uintptr_t>(a.w_router) & 7u) == 0;
    if (pairs) {
#pragma unroll 8
        for (int h = 2 * lane; h < H; h += 64) {
            const uint32_t xp = __ldg(reinterpret_cast<const uint32_t*>(xr + h));
            const float2 wp = __ldg(reinterpret_cast<const float2*>(wr + h));
            acc = __fmaf_rn(bf16_bits_to_f32(static_cast<uint16_t>(xp & 0xffffu)), wp.x, acc);
            acc = __fmaf_rn(bf16_bits_to_f32(static_cast<uint16_t>(xp >> 16)), wp.y, acc);
        }
    } else {
        for (int h0 = 2 * lane; h0 < H; h0 += 64)
            for (int h = h0; h < h0 + 2 && h < H; ++h)
                acc = __fmaf_rn(bf16_bits_to_f32(__ldg(xr + h)), __ldg(wr + h), acc);
    }
    const float sum = warp_sum_tree(acc);
    if (lane == 0)
        a.logits[static_cast<size_t>(t) * E + e] =
            a.router_bias ? __fadd_rn(sum, __ldg(a.router_bias + e)) : sum;
}

// Two fp32 fused multiply-adds in one instruction (fma.rn.f32x2): each half
// is an ordinary round-to-nearest fma, so results are those of two fmaf.
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long pair_u32(uint32_t lo, uint32_t hi) {
    unsigned long long d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ float pair_lo(unsigned long long v) {
    return __uint_as_float(static_cast<uint32_t>(v));
}
__device__ __forceinline__ float pair_hi(unsigned long long v) {
    return __uint_as_float(static_cast<uint32_t>(v >> 32));
}

// TMA-fed path (H % KC == 0, 16-byte aligned rows).  KC-wide column chunks
// of a BT-token x tile (bf16, [BT][KC]) and a BE-expert router-weight tile
// (fp32, [BE][KC]) stream through a STAGES-deep ring in their natural
// layout; WTW x WEW warps each own TT tokens x 8 experts.  Lane 0 of warp 0
// also keeps the ring full: at chunk c it refills the stage of chunk c - 2
// once every warp has released it, so the ring runs STAGES - 2 chunks ahead
// and no warp is spent on loads alone (a block of 8 warps leaves each SM
// sub-partition two warps and the full register budget).  In every 64-wide
// round of a chunk lane j reads its pair h = 2j, 2j+1 as one 32-bit word
// per token (both bf16 values) and one 64-bit word per expert --
// conflict-free, since the 32 lanes cover consecutive words.  Two tokens
// share one fma.rn.f32x2 (x of both tokens times the weight duplicated into
// both halves), so a lane accumulates TT/2 x 8 packed pairs = TT x 8 partial
// sums, each in exactly the pinned order.  The 32 partials of every logit
// are then reduced by a transposing xor-butterfly: at level s lanes l and l^s
// add their halves of the remaining values, which is the pinned pairwise
// tree, and each lane ends with TT/4 finished logits.  Every ring wait is
// bounded: a wait that gives up raises an abort flag, records
// GBMOE_ERR_TIMEOUT and the block stores nothing.
// Level S of the transposing butterfly over the first N values: the lane
// keeps the upper half iff (lane & S) and adds the partner's copy of it.
template <int NV, int N, int S>
__device__ __forceinline__ void transpose_butterfly(float (&v)[NV], int lane) {
    const bool up = (lane & S) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float send = up ? v[i] : v[i + N / 2];
        const float keep = up ? v[i + N / 2] : v[i];
        v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, S));
    }
    if constexpr (S > 1) transpose_butterfly<NV, N / 2, S / 2>(v, lane);
}

template <int TT, int WTW, int WEW, int KC, int STAGES, int LAG_ = 1>
struct RouterTile {
    static constexpr int TE = 8;
    static constexpr int KC_ = KC;
    static constexpr int LAG = LAG_;  // chunks between a stage's release and its refill
    static constexpr int BT = TT * WTW, BE = TE * WEW;
    static constexpr int WARPS = WTW * WEW;
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int X_BYTES = BT * KC * 2;
    static constexpr int W_BYTES = BE * KC * 4;
    static constexpr int STAGE_BYTES = X_BYTES + W_BYTES;
    static constexpr int OFF_BARS = STAGES * STAGE_BYTES;
    static constexpr int SMEM_BYTES = OFF_BARS + 2 * STAGES * 8 + 16 + 128;  // + base alignment
    static_assert(TT % 4 == 0 && TT * TE >= 32, "the transposing reduction needs >= 32 values");
    static_assert(KC % 64 == 0 && KC <= 256, "chunks are whole 64-wide rounds, <= 256 (TMA box)");
    static_assert(STAGE_BYTES % 128 == 0, "stage alignment");
    static_assert(STAGES > LAG && STAGES <= 32, "ring depth");
};

constexpr uint64_t kRouteWaitNs = 2000000000ull;

template <int TT, int WTW, int WEW, int KC, int STAGES, int LAG_ = 1>
__global__ void __launch_bounds__(RouterTile<TT, WTW, WEW, KC, STAGES, LAG_>::THREADS, 1)
router_logits_tma_kernel(const __grid_constant__ CUtensorMap mx,
                         const __grid_constant__ CUtensorMap mw, const float* __restrict__ bias,
                         int T, int E, int H, float* __restrict__ logits, int* status) {
    using L = RouterTile<TT, WTW, WEW, KC, STAGES, LAG_>;
    constexpr int TE = L::TE, NP = TT / 2, NV = TT * TE;
    extern __shared__ uint8_t route_smem[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(route_smem) + 127) & ~static_cast<uintptr_t>(127));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BARS);
    uint64_t* empty = full + STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STAGES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * L::BT, e0 = blockIdx.y * L::BE;
    const int nc = H / KC;
    const bool producer = warp == 0 && lane == 0;
    const uint64_t pol = l2_policy_evict_last();  // both tiles are re-read by other blocks

    auto issue = [&](int c) {
        const int st = c % STAGES;
        mbar_arrive_expect_tx(full + st, L::STAGE_BYTES);
        uint8_t* xs = smem + st * L::STAGE_BYTES;
        tma_load_2d(xs, &mx, full + st, c * KC, t0, pol);
        tma_load_2d(xs + L::X_BYTES, &mw, full + st, c * KC, e0, pol);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, L::WARPS);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    int issued = 0;  // chunks whose loads lane 0 of warp 0 has issued
    if (producer) {
        tma_prefetch_desc(&mx);
        tma_prefetch_desc(&mw);
        for (; issued < min(STAGES, nc); ++issued) issue(issued);
    }

    const int wt = warp / WEW, we = warp % WEW;
    unsigned long long acc[NP][TE];
#pragma unroll
    for (int a = 0; a < NP; ++a)
#pragma unroll
        for (int e = 0; e < TE; ++e) acc[a][e] = 0ull;
    bool ok = true;
    for (int c = 0; c < nc; ++c) {
        const int stage = c % STAGES;
        const uint32_t phase = static_cast<uint32_t>(c / STAGES) & 1u;
        if (warp == 0) {
            if (lane == 0 && c >= L::LAG && issued < nc) {
                const int cp = c - L::LAG;  // issued == cp + STAGES here
                if (mbar_wait_bounded(empty + cp % STAGES, static_cast<uint32_t>(cp / STAGES) & 1u,
                                      abort_flag, status, kRouteWaitNs))
                    issue(issued++);
            }
            __syncwarp();
        }
        // every lane waits; the vote keeps the warp together if one gives up
        if (!__all_sync(0xffffffffu,
                        mbar_wait_bounded(full + stage, phase, abort_flag, status, kRouteWaitNs))) {
            ok = false;
            break;
        }
        const uint8_t* xs = smem + stage * L::STAGE_BYTES;
        const uint32_t* xrow = reinterpret_cast<const uint32_t*>(xs) + (wt * TT) * (KC / 2) + lane;
        const unsigned long long* wrow =
            reinterpret_cast<const unsigned long long*>(xs + L::X_BYTES) + (we * TE) * (KC / 2) +
            lane;
#pragma unroll
        for (int r = 0; r < KC / 64; ++r) {
            uint32_t xw[TT];
#pragma unroll
            for (int t = 0; t < TT; ++t) xw[t] = xrow[t * (KC / 2) + r * 32];
            unsigned long long wp[TE];
#pragma unroll
            for (int e = 0; e < TE; ++e) wp[e] = wrow[e * (KC / 2) + r * 32];
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                unsigned long long xv[NP];
#pragma unroll
                for (int a = 0; a < NP; ++a) {
                    const uint32_t u0 = xw[2 * a], u1 = xw[2 * a + 1];
                    xv[a] = m ? pair_u32(u0 & 0xffff0000u, u1 & 0xffff0000u)
                              : pair_u32(u0 << 16, u1 << 16);
                }
#pragma unroll
                for (int e = 0; e < TE; ++e) {
                    const uint32_t v = m ? __float_as_uint(pair_hi(wp[e]))
                                         : __float_as_uint(pair_lo(wp[e]));
                    const unsigned long long wd = pair_u32(v, v);
#pragma unroll
                    for (int a = 0; a < NP; ++a) acc[a][e] = fma2(xv[a], wd, acc[a][e]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + stage);
    }
    if (!ok) {
        if (producer) {  // let every copy this thread issued land before the block exits
            for (int c = max(0, issued - STAGES); c < issued; ++c)
                mbar_wait_timeout(full + c % STAGES, static_cast<uint32_t>(c / STAGES) & 1u,
                                  200000000ull);
        }
        return;
    }

    // v[(a*8 + e)*2 + u]: token wt*TT + 2a + u, expert we*8 + e
    float v[NV];
#pragma unroll
    for (int a = 0; a < NP; ++a)
#pragma unroll
        for (int e = 0; e < TE; ++e) {
            v[(a * TE + e) * 2] = pair_lo(acc[a][e]);
            v[(a * TE + e) * 2 + 1] = pair_hi(acc[a][e]);
        }
    transpose_butterfly<NV, NV, 16>(v, lane);
    // the lane holds values p = base + i, i < NV/32, base from its lane bits
    constexpr int NL = NV / 32;
    const int base = (((lane >> 4) & 1) * (NV / 2)) + (((lane >> 3) & 1) * (NV / 4)) +
                     (((lane >> 2) & 1) * (NV / 8)) + (((lane >> 1) & 1) * (NV / 16)) +
                     ((lane & 1) * (NV / 32));
#pragma unroll
    for (int i = 0; i < NL; ++i) {
        const int p = base + i;
        const int u = p & 1, e = (p >> 1) % TE, a = (p >> 1) / TE;
        const int t = t0 + wt * TT + 2 * a + u, ex = e0 + we * TE + e;
        if (t < T && ex < E)
            logits[static_cast<size_t>(t) * E + ex] = bias ? __fadd_rn(v[i], __ldg(bias + ex)) : v[i];
    }
}

// ----------------------------------------------------------- selection
// Monotone map of fp32 onto u32 (a larger value gives a larger key; -0 is
// folded onto +0 so that equal values tie).  Key 0 means "no candidate".
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Lane holding the largest key, the lowest such lane on ties; -1 if no lane
// has a candidate.
__device__ __forceinline__ int warp_pick(uint32_t key) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, key);
    if (m == 0u) return -1;
    return __ffs(__ballot_sync(0xffffffffu, key == m)) - 1;
}

template <int EPL>
__device__ __forceinline__ float pick(const float (&a)[EPL], int idx) {
    float v = 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
        if (i == idx) v = a[i];
    return v;
}

// One warp per token.  Lane L holds the EPL consecutive experts
// e = EPL*L + i, so expert order is (lane, slot) order: a warp-wide
// "largest key, lowest lane" pick after an in-lane "largest value, lowest
// slot" pick is exactly "largest value, lowest expert index".  When every
// expert group spans a power-of-two block of whole lanes (E = 256 in 8 groups:
// 4 lanes of 8 experts each) the group top-2 is an in-lane top-2 merged
// across the block; other shapes take a loop over the groups.
template <int EPL>
__global__ void __launch_bounds__(256) route_select_kernel(const RouteArgs a, int* status) {
    const int lane = threadIdx.x & 31;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= a.T) return;
    const gbmoe_route_cfg& c = a.cfg;
    const int E = c.E_log, k = c.top_k;
    const float* lrow = a.logits + static_cast<size_t>(t) * E;
    const int eb = EPL * lane;

    float sc[EPL];
    if (EPL % 4 == 0 && E % 4 == 0 && eb + EPL <= E &&
        (reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0) {
#pragma unroll
        for (int i = 0; i < EPL; i += 4) {
            const float4 v = *reinterpret_cast<const float4*>(lrow + eb + i);
            sc[i] = v.x;
            sc[i + 1] = v.y;
            sc[i + 2] = v.z;
            sc[i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) sc[i] = eb + i < E ? lrow[eb + i] : 0.0f;
    }
    if (c.scoring == GBMOE_SCORE_SOFTMAX) {
        float m = kNegInf;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (eb + i < E) m = fmaxf(m, sc[i]);
#pragma unroll
        for (int s = 16; s >= 1; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
        // denominator in the pinned order: partial j takes e = j, j+32, ...
        float part = 0.0f;
        for (int e = lane; e < E; e += 32) part = __fadd_rn(part, pinned_exp(__fsub_rn(lrow[e], m)));
        const float S = warp_sum_tree(part);
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (eb + i < E) sc[i] = __fdiv_rn(pinned_exp(__fsub_rn(sc[i], m)), S);
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
            const float s = __shfl_sync(0xffffffffu, pick<EPL>(sc, ej % EPL), ej / EPL);
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
            const int e = eb + i;
            sel[i] = kNegInf;
            if (e < E) {
                sel[i] = a.corr_bias ? __fadd_rn(sc[i], __ldg(a.corr_bias + e)) : sc[i];
                allowed |= 1u << i;
            }
        }
        if (c.n_group > 1) {
            const int G = c.n_group, gs = E / G;
            const bool top2 = c.group_score == GBMOE_GROUP_TOP2SUM && gs > 1;
            const int lpg = gs / EPL;  // lanes per group on the fast path
            if (gs % EPL == 0 && lpg <= 32 && (lpg & (lpg - 1)) == 0) {
                float b1 = kNegInf, b2 = kNegInf;
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    if ((allowed >> i) & 1u) {
                        const float v = sel[i];
                        if (v > b1) {
                            b2 = b1;
                            b1 = v;
                        } else if (v > b2) {
                            b2 = v;
                        }
                    }
                }
                for (int s = 1; s < lpg; s <<= 1) {
                    const float o1 = __shfl_xor_sync(0xffffffffu, b1, s);
                    const float o2 = __shfl_xor_sync(0xffffffffu, b2, s);
                    const float n2 = fmaxf(fminf(b1, o1), fmaxf(b2, o2));
                    b1 = fmaxf(b1, o1);
                    b2 = n2;
                }
                const float gsc = top2 ? __fadd_rn(b1, b2) : b1;
                const bool leader = (lane % lpg) == 0 && eb < E;
                bool kept = false;
                for (int r = 0; r < c.topk_group; ++r) {
                    const int wl = warp_pick(leader && !kept ? order_key(gsc) : 0u);
                    if (lane == wl) kept = true;
                }
                kept = __shfl_sync(0xffffffffu, kept, lane & ~(lpg - 1));
                if (!kept) allowed = 0;
            } else {
                int gid[EPL];
#pragma unroll
                for (int i = 0; i < EPL; ++i) gid[i] = (eb + i) / gs;
                float my_g = 0.0f;
                for (int g = 0; g < G; ++g) {
                    float b1 = kNegInf, b2 = kNegInf;
#pragma unroll
                    for (int i = 0; i < EPL; ++i) {
                        if (((allowed >> i) & 1u) && gid[i] == g) {
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
                    if (lane == g) my_g = top2 ? __fadd_rn(b1, b2) : b1;
                }
                uint32_t keep = 0;
                for (int r = 0; r < c.topk_group; ++r) {
                    const int wl = warp_pick(lane < G && !((keep >> lane) & 1u) ? order_key(my_g) : 0u);
                    if (wl >= 0) keep |= 1u << wl;
                }
#pragma unroll
                for (int i = 0; i < EPL; ++i)
                    if (!((keep >> gid[i]) & 1u)) allowed &= ~(1u << i);
            }
        }
        for (int j = 0; j < k; ++j) {
            int bi = -1;
            float bv = 0.0f;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                if (((allowed >> i) & 1u) && (bi < 0 || sel[i] > bv)) {
                    bi = i;
                    bv = sel[i];
                }
            }
            const int wl = warp_pick(bi >= 0 ? order_key(bv) : 0u);
            if (wl < 0) {  // fewer allowed experts than k (excluded by validation)
                record_error(status, GBMOE_ERR_DEVICE);
                break;
            }
            const int wi = __shfl_sync(0xffffffffu, bi, wl);
            if (lane == wl) allowed &= ~(1u << bi);
            const float s = __shfl_sync(0xffffffffu, pick<EPL>(sc, wi), wl);
            if (lane == j) {
                my_e = EPL * wl + wi;
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

// Router-logit tile variants (measured on the 8192- and 128-token routers):
// many tokens -> 16-token x 8-expert warp tiles, 2 x 4 warps (32 x 32
// blocks); few tokens -> 4 x 8 warp tiles, 4 x 2 warps (16 x 16 blocks), so
// that a decode batch still spreads over the GPU.  256-wide chunks (4-deep
// ring) when H allows, else 128-wide (6-deep): fewer ring hand-offs per FMA.
using RouterBig256 = RouterTile<16, 2, 4, 256, 4>;
using RouterBig128 = RouterTile<16, 2, 4, 128, 6>;
using RouterSmall256 = RouterTile<4, 4, 2, 256, 4>;
using RouterSmall128 = RouterTile<4, 4, 2, 128, 6>;
#define ROUTER_BIG256 router_logits_tma_kernel<16, 2, 4, 256, 4>
#define ROUTER_BIG128 router_logits_tma_kernel<16, 2, 4, 128, 6>
#define ROUTER_SMALL256 router_logits_tma_kernel<4, 4, 2, 256, 4>
#define ROUTER_SMALL128 router_logits_tma_kernel<4, 4, 2, 128, 6>

std::mutex g_route_attr_mu;
bool g_route_attr_done[kMaxDevices];

cudaError_t ensure_route_attrs(int device) {
    std::lock_guard<std::mutex> lk(g_route_attr_mu);
    if (device >= 0 && device < kMaxDevices && g_route_attr_done[device]) return cudaSuccess;
    const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaFuncSetAttribute(ROUTER_BIG256, a, RouterBig256::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ROUTER_BIG128, a, RouterBig128::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ROUTER_SMALL256, a, RouterSmall256::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ROUTER_SMALL128, a, RouterSmall128::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (device >= 0 && device < kMaxDevices) g_route_attr_done[device] = true;
    return cudaSuccess;
}

template <class L, class K>
cudaError_t launch_router_tma(K kernel, const RouteArgs& a, const DevCtx& ctx, cudaStream_t s,
                              bool* launched) {
    *launched = false;
    const int E = a.cfg.E_log;
    CUtensorMap mx, mw;
    if (!encode_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, a.H, a.T,
                       static_cast<uint64_t>(a.H) * 2, L::KC_, L::BT, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.w_router, a.H, E,
                       static_cast<uint64_t>(a.H) * 4, L::KC_, L::BE, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaSuccess;  // not encodable: the caller takes the generic path
    const cudaError_t e = ensure_route_attrs(ctx.device);
    if (e != cudaSuccess) return e;
    dim3 grid((a.T + L::BT - 1) / L::BT, (E + L::BE - 1) / L::BE);
    kernel<<<grid, L::THREADS, L::SMEM_BYTES, s>>>(mx, mw, a.router_bias, a.T, E, a.H, a.logits,
                                                   ctx.status);
    *launched = true;
    return cudaGetLastError();
}

template <int EPL>
cudaError_t launch_select(const RouteArgs& a, const DevCtx& ctx, cudaStream_t s) {
    // small batches: two tokens per block so that the warps spread over the SMs
    const int warps_per_block = a.T >= 8 * ctx.num_sms ? 8 : 2;
    const int blocks = (a.T + warps_per_block - 1) / warps_per_block;
    route_select_kernel<EPL><<<blocks, 32 * warps_per_block, 0, s>>>(a, ctx.status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, const DevCtx& ctx, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    const int E = a.cfg.E_log;
    bool done = false;
    if (a.w_router && a.hash_logits_only && a.cfg.use_hash &&
        a.cfg.scoring != GBMOE_SCORE_SOFTMAX) {
        router_logits_hash_kernel<<<a.T, 32 * a.cfg.top_k, 0, s>>>(a);
        const cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        done = true;
    }
    if (a.w_router && !done && a.H % 128 == 0 && (reinterpret_cast<uintptr_t>(a.x) & 15u) == 0 &&
        (reinterpret_cast<uintptr_t>(a.w_router) & 15u) == 0) {
        const long big_blocks =
            static_cast<long>((a.T + RouterBig256::BT - 1) / RouterBig256::BT) *
            ((E + RouterBig256::BE - 1) / RouterBig256::BE);
        const bool big = big_blocks >= 2L * ctx.num_sms, wide = a.H % 256 == 0;
        const cudaError_t err =
            big ? (wide ? launch_router_tma<RouterBig256>(ROUTER_BIG256, a, ctx, s, &done)
                        : launch_router_tma<RouterBig128>(ROUTER_BIG128, a, ctx, s, &done))
                : (wide ? launch_router_tma<RouterSmall256>(ROUTER_SMALL256, a, ctx, s, &done)
                        : launch_router_tma<RouterSmall128>(ROUTER_SMALL128, a, ctx, s, &done));
        if (err != cudaSuccess) return err;
    }
    if (a.w_router && !done) {
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
