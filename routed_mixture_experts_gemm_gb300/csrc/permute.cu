// Token dispatch as a local permutation.
//
// Follows the vLLM-Ascend "Kimi K3 MoE Forward Insight" page, section
// "Stage 4: Dispatch, MLP, Combine", AllGather row of the mode table: sort
// tokens by expert and return expert token counts.
//
// Stable counting sort of the N = T*k flat indices f = t*k + j by physical
// expert p = ids_phys[f]; row r = offsets[p] + (rank of f among the indices
// routed to p).  No atomic operation decides an order, so the result is
// bit-exact and run-to-run identical:
//   1. hist:    worker w (one warp, flat range [w*256, (w+1)*256)) counts
//               its indices per expert -> hist[w][p]            (counts only)
//   2. colscan: one block per expert p turns hist[.][p] into an exclusive
//               prefix over workers and writes counts[p]; the last block to
//               finish scans counts into offsets
//   3. scatter: each worker walks its range in order, 32 indices at a time;
//               __match_any_sync groups equal experts, the rank inside the
//               group is the popcount of lower lanes
//   4. gather:  x_perm[r] = x[row_to_token[r]] with 16-byte vector copies
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace gbmoe {
namespace {

constexpr int kWarpsPerBlock = 4;

struct PermWs {
    int32_t* hist;      // [W][P]
    uint32_t* done;     // last-block counter
};

__host__ __device__ inline int64_t n_workers(int64_t N) { return (N + kPermChunk - 1) / kPermChunk; }

__host__ __device__ inline PermWs perm_ws(void* ws, int64_t N, int P) {
    PermWs w;
    w.hist = reinterpret_cast<int32_t*>(ws);
    const size_t hist_bytes = ((static_cast<size_t>(n_workers(N)) * P * 4 + 255) / 256) * 256;
    w.done = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + hist_bytes);
    return w;
}

__global__ void __launch_bounds__(32 * kWarpsPerBlock) perm_hist_kernel(
    const int32_t* __restrict__ ids, int64_t N, int P, int32_t* __restrict__ hist,
    uint32_t* __restrict__ done, int* status) {
    extern __shared__ int32_t cnt_all[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* cnt = cnt_all + warp * P;
    const int64_t w = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp;
    if (blockIdx.x == 0 && threadIdx.x == 0) *done = 0u;
    for (int p = lane; p < P; p += 32) cnt[p] = 0;
    __syncwarp();
    if (w < n_workers(N)) {
        const int64_t f0 = w * kPermChunk;
        for (int it = 0; it < kPermChunk / 32; ++it) {
            const int64_t f = f0 + it * 32 + lane;
            if (f < N) {
                const int p = ids[f];
                if (p >= 0 && p < P)
                    atomicAdd(cnt + p, 1);
                else
                    record_error(status, GBMOE_ERR_DEVICE);
            }
        }
        __syncwarp();
        int32_t* dst = hist + w * P;
        for (int p = lane; p < P; p += 32) dst[p] = cnt[p];
    }
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 256).
__device__ __forceinline__ int block_exclusive_scan(int v, int* smem_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, s);
        if (lane >= s) incl += o;
    }
    if (lane == 31) smem_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int wv = lane < 8 ? smem_warp[lane] : 0;
        int wi = wv;
#pragma unroll
        for (int s = 1; s < 8; s <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wi, s);
            if (lane >= s) wi += o;
        }
        if (lane < 8) smem_warp[lane] = wi - wv;  // exclusive warp offsets
        if (lane == 7) smem_warp[8] = wi;
    }
    __syncthreads();
    const int res = smem_warp[warp] + incl - v;
    *total = smem_warp[8];
    __syncthreads();
    return res;
}

__global__ void __launch_bounds__(256) perm_colscan_kernel(int32_t* __restrict__ hist, int64_t W,
                                                           int P, int32_t* __restrict__ counts,
                                                           int32_t* __restrict__ offsets,
                                                           uint32_t* __restrict__ done) {
    __shared__ int sw[9];
    __shared__ bool last;
    const int p = blockIdx.x;
    int carry = 0;
    for (int64_t w0 = 0; w0 < W; w0 += 256) {
        const int64_t w = w0 + threadIdx.x;
        const int v = w < W ? hist[w * P + p] : 0;
        int tot;
        const int ex = block_exclusive_scan(v, sw, &tot);
        if (w < W) hist[w * P + p] = carry + ex;
        carry += tot;
    }
    if (threadIdx.x == 0) {
        counts[p] = carry;
        __threadfence();
        last = atomicAdd(done, 1u) == static_cast<uint32_t>(P - 1);
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    int run = 0;
    for (int p0 = 0; p0 < P; p0 += 256) {
        const int q = p0 + threadIdx.x;
        const int v = q < P ? __ldcg(counts + q) : 0;
        int tot;
        const int ex = block_exclusive_scan(v, sw, &tot);
        if (q < P) offsets[q] = run + ex;
        run += tot;
    }
    if (threadIdx.x == 0) offsets[P] = run;
}

__global__ void __launch_bounds__(32 * kWarpsPerBlock) perm_scatter_kernel(
    const int32_t* __restrict__ ids, int64_t N, int k, int P, const int32_t* __restrict__ hist,
    const int32_t* __restrict__ offsets, int32_t* __restrict__ row_to_token,
    int32_t* __restrict__ flat_to_row) {
    extern __shared__ int32_t run_all[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* run = run_all + warp * P;
    const int64_t w = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp;
    for (int p = lane; p < P; p += 32) run[p] = 0;
    __syncwarp();
    if (w >= n_workers(N)) return;
    const int32_t* base = hist + w * P;
    const unsigned lt = (1u << lane) - 1u;
    const int64_t f0 = w * kPermChunk;
    for (int it = 0; it < kPermChunk / 32; ++it) {
        const int64_t f = f0 + it * 32 + lane;
        int p = -1;
        if (f < N) {
            p = ids[f];
            if (p < 0 || p >= P) p = -1;  // reported by the histogram pass
        }
        const unsigned peers = __match_any_sync(0xffffffffu, p);
        const int rank = __popc(peers & lt);
        if (p >= 0) {
            const int r = offsets[p] + base[p] + run[p] + rank;
            row_to_token[r] = static_cast<int32_t>(f / k);
            flat_to_row[f] = r;
        } else if (f < N) {
            flat_to_row[f] = -1;  // id outside [0, P): no row
        }
        __syncwarp();
        if (p >= 0 && rank == 0) run[p] += __popc(peers);
        __syncwarp();
    }
}

// Small batches (N <= kSmallPermMaxN, P <= 1024): the whole permutation in
// one block of 32 warps.  Warp w takes the contiguous flat range
// [w*per, (w+1)*per); its per-expert counts, turned into an exclusive prefix
// over warps, then the running count of its own earlier indices, give every
// index its stable rank -- the same order as the multi-kernel path.
constexpr int64_t kSmallPermMaxN = 4096;
constexpr int kSmallPermMaxP = 1024;

__global__ void __launch_bounds__(1024) perm_small_kernel(
    const int32_t* __restrict__ ids, int64_t N, int k, int P, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ row_to_token,
    int32_t* __restrict__ flat_to_row, int* status) {
    extern __shared__ int32_t perm_sm[];
    int32_t* hist = perm_sm;           // [32][P]: counts, then exclusive prefix, then running
    int32_t* offs = perm_sm + 32 * P;  // [P]
    __shared__ int wsum[32];
    __shared__ int total;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 32 * P; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int64_t per = (N + 31) / 32;
    const int64_t f0 = min(N, warp * per), f1 = min(N, f0 + per);
    const unsigned lt = (1u << lane) - 1u;
    int32_t* h = hist + warp * P;
    auto expert_of = [&](int64_t f) {
        int p = -1;
        if (f < f1) {
            p = ids[f];
            if (p < 0 || p >= P) p = -1;
        }
        return p;
    };
    // 1. per-warp counts
    for (int64_t b0 = f0; b0 < f1; b0 += 32) {
        const int64_t f = b0 + lane;
        const int p = expert_of(f);
        if (p < 0 && f < f1) record_error(status, GBMOE_ERR_DEVICE);
        const unsigned peers = __match_any_sync(0xffffffffu, p);
        if (p >= 0 && __popc(peers & lt) == 0) h[p] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // 2. exclusive prefix over warps, per expert; totals are the counts
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            const int v = hist[w * P + p];
            hist[w * P + p] = run;
            run += v;
        }
        offs[p] = run;
    }
    __syncthreads();
    // 3. offsets = exclusive scan of the counts (one expert per thread)
    {
        const int p = threadIdx.x;
        const int v = p < P ? offs[p] : 0;
        int incl = v;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, s);
            if (lane >= s) incl += o;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int wv = wsum[lane];
            int wi = wv;
#pragma unroll
            for (int s = 1; s < 32; s <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, wi, s);
                if (lane >= s) wi += o;
            }
            wsum[lane] = wi - wv;
            if (lane == 31) total = wi;
        }
        __syncthreads();
        const int ex = wsum[warp] + incl - v;
        if (p < P) {
            counts[p] = v;
            offsets[p] = ex;
            offs[p] = ex;
        }
        if (p == 0) offsets[P] = total;
    }
    __syncthreads();
    // 4. rows, walking each range again in order
    for (int64_t b0 = f0; b0 < f1; b0 += 32) {
        const int64_t f = b0 + lane;
        const int p = expert_of(f);
        const unsigned peers = __match_any_sync(0xffffffffu, p);
        const int rank = __popc(peers & lt);
        if (p >= 0) {
            const int r = offs[p] + h[p] + rank;
            row_to_token[r] = static_cast<int32_t>(f / k);
            flat_to_row[f] = r;
        } else if (f < f1) {
            flat_to_row[f] = -1;  // id outside [0, P): no row
        }
        __syncwarp();
        if (p >= 0 && rank == 0) h[p] += __popc(peers);
        __syncwarp();
    }
}

// x_perm[r] = x[row_to_token[r]]: one warp per row, four 16-byte loads in
// flight per lane; x rows are kept in L2 (each is read k times), x_perm is
// streamed out.  Only the offsets[P] rows the permutation wrote carry a token
// (ids outside [0, P) get no row): the rows after them are zero-filled and
// x is not read for them.
__device__ __forceinline__ uint4 ld_keep(const uint4* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_stream(uint4* p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(32 * kGatherWarps) perm_gather_kernel(
    const uint4* __restrict__ x, int64_t N, int vec_per_row,
    const int32_t* __restrict__ row_to_token, const int32_t* __restrict__ rows_written,
    uint4* __restrict__ x_perm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t keep = l2_policy_evict_last(), stream = l2_policy_evict_first();
    const int64_t n_rows = min(N, static_cast<int64_t>(max(0, *rows_written)));
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kGatherWarps + warp; r < N;
         r += static_cast<int64_t>(gridDim.x) * kGatherWarps) {
        uint4* dst = x_perm + r * vec_per_row;
        if (r >= n_rows) {
            for (int v = lane; v < vec_per_row; v += 32) st_stream(dst + v, make_uint4(0, 0, 0, 0), stream);
            continue;
        }
        const int64_t t = row_to_token[r];
        const uint4* src = x + t * vec_per_row;
        for (int v0 = 0; v0 < vec_per_row; v0 += 128) {
            uint4 buf[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + 32 * u + lane;
                if (v < vec_per_row) buf[u] = ld_keep(src + v, keep);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + 32 * u + lane;
                if (v < vec_per_row) st_stream(dst + v, buf[u], stream);
            }
        }
    }
}

// The small kernel's shared-memory limit is raised once per device (under a
// lock: first calls may come from several host threads at once).
std::mutex g_small_attr_mu;
bool g_small_attr_done[kMaxDevices];

cudaError_t ensure_small_attr(int device) {
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_small_attr_mu);
    if (g_small_attr_done[device]) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(
        perm_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(sizeof(int32_t) * 33 * kSmallPermMaxP));
    if (e == cudaSuccess) g_small_attr_done[device] = true;
    return e;
}

}  // namespace

size_t permute_ws_bytes(int64_t N, int E_phys) {
    const size_t hist_bytes = ((static_cast<size_t>(n_workers(N)) * E_phys * 4 + 255) / 256) * 256;
    return hist_bytes + 256;
}

cudaError_t launch_permute(const int32_t* ids_phys, int64_t N, int k, int E_phys,
                           const uint16_t* x, int H, int32_t* counts, int32_t* offsets,
                           int32_t* row_to_token, int32_t* flat_to_row, uint16_t* x_perm,
                           void* ws, const DevCtx& ctx, cudaStream_t s) {
    const int P = E_phys;
    if (N == 0) {
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * P, s);
        if (e != cudaSuccess) return e;
        return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (P + 1), s);
    }
    if (N <= kSmallPermMaxN && P <= kSmallPermMaxP) {
        const size_t smem = sizeof(int32_t) * 33 * P;
        const cudaError_t e = ensure_small_attr(ctx.device);
        if (e != cudaSuccess) return e;
        perm_small_kernel<<<1, 1024, smem, s>>>(ids_phys, N, k, P, counts, offsets, row_to_token,
                                                flat_to_row, ctx.status);
    } else {
        const PermWs w = perm_ws(ws, N, P);
        const int64_t W = n_workers(N);
        const int blocks = static_cast<int>((W + kWarpsPerBlock - 1) / kWarpsPerBlock);
        const size_t smem = sizeof(int32_t) * P * kWarpsPerBlock;
        perm_hist_kernel<<<blocks, 32 * kWarpsPerBlock, smem, s>>>(ids_phys, N, P, w.hist, w.done,
                                                                   ctx.status);
        perm_colscan_kernel<<<P, 256, 0, s>>>(w.hist, W, P, counts, offsets, w.done);
        perm_scatter_kernel<<<blocks, 32 * kWarpsPerBlock, smem, s>>>(ids_phys, N, k, P, w.hist,
                                                                      offsets, row_to_token,
                                                                      flat_to_row);
    }
    if (x_perm) {
        const int vec = H / 8;
        const int64_t want = (N + kGatherWarps - 1) / kGatherWarps;
        const int grid = static_cast<int>(std::min<int64_t>(want, 8L * ctx.num_sms));
        perm_gather_kernel<<<grid, 32 * kGatherWarps, 0, s>>>(
            reinterpret_cast<const uint4*>(x), N, vec, row_to_token, offsets + P,
            reinterpret_cast<uint4*>(x_perm));
    }
    return cudaGetLastError();
}

}  // namespace gbmoe
