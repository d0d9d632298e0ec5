// Grouped expert GEMMs on 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Follows the vLLM-Ascend "Kimi K3 MoE Forward Insight" page, section
// "Stage 4: Dispatch, MLP, Combine": expert input -> grouped matmul gate/up
// -> activation (SwiGLU) -> grouped matmul down, over per-expert token groups.
//
// Orientation ("weights as M"): every tile is D[128 weight rows x n tokens] =
// W[128 x K] . X[n x K]^T, with the expert weight rows as the MMA's M = 128
// operand and the expert's tokens as its N operand (N = 16..BN, a multiple of
// 16, chosen per tile from the expert's row count).  Decode-sized groups (a
// handful of rows per expert) then waste no tensor-core rows on padding and
// every CTA streams distinct weight tiles; prefill-sized groups use N = BN.
//
// Gate/up: two A operands (W_gate and W_up rows of the same intermediate
// block) feed two TMEM accumulators, so each thread of the epilogue holds g
// and u of the same output and applies act = bf16(silu(g) * u) in registers.
// Down: one A operand (W_down rows), or two consecutive 128-row blocks
// sharing one token operand; y = acc kept in fp32 (only the activation is
// rounded to bf16 inside the layer).
//
// One persistent CTA per SM with four roles: warp 0 streams the weight boxes
// by TMA (128B-swizzled K-major tiles) through the A ring; warps 10-13 fill
// the B ring with the token rows -- by TMA from a row-contiguous operand, or,
// for the gate/up GEMM of the layer, gathered straight from the unpermuted
// hidden states: row r of the tile is x[row_to_token[r]], copied in 16-byte
// pieces (cp.async) into the same swizzled layout, so the permuted copy of x
// is never written; warp 1 issues tcgen05.mma and owns TMEM (2 accumulator
// buffers so the epilogue of tile i overlaps the main loop of tile i+1,
// except for the 256-token tiles whose accumulators fill TMEM); warps 2-9
// (two per TMEM lane quarter) drain TMEM with tcgen05.ld and write coalesced
// rows straight from registers.  Tiles are ordered (expert, weight block,
// token block) so CTAs working on the token blocks of one expert read the
// same weight tile at the same time (one HBM read, L2 hits after).  The tile
// table is built on the device from the group offsets: no host
// synchronisation.
//
// Fused mode (small groups): one cooperative launch walks every gate/up tile
// and then every down tile; a down tile of expert p waits (bounded) until all
// of p's gate/up tiles have published their activations, so the down GEMM
// fills the last wave of the gate/up GEMM instead of waiting for the launch
// boundary (its weights already stream while it waits: the A ring does not
// depend on the activations).
//
// CTA pairs (prefill-sized groups): two CTAs of a cluster compute one tile
// with tcgen05.mma.cta_group::2 (M = 256 per A operand), issued by the even
// CTA.  Each CTA stages its own 128 rows of every A operand and half of the
// tile's token rows, so a stage per CTA is 48 KB instead of 64 KB (four
// stages fit) and the tensor cores read the B operand once for two SMs.  The
// odd CTA's TMA copies complete on the even CTA's full barriers, whose
// expected byte count the even CTA sets for both halves (no arrival from the
// odd CTA on the critical path); gathered token rows of the odd CTA are
// announced by one relaxed remote arrival once they have landed and been
// fenced; the MMA commits multicast to both CTAs' empty and accumulator
// barriers.  Each CTA's epilogue drains its own 128 rows for all tokens and
// writes whole 16-token blocks of bf16 or fp32 outputs through shared memory
// and TMA stores (prefill down GEMM 1.84 -> 1.71 ms bf16, 1.35 -> 1.21 ms MX).
// The bf16 GEMMs, the FP8-row gate/up and both MX GEMMs (224-token tiles)
// run on CTA pairs for prefill-sized groups.
//
// Every pipeline wait is bounded (wall-clock limit); a wait that gives up
// raises an abort flag seen by all roles, records GBMOE_ERR_TIMEOUT, lets
// in-flight copies and MMAs finish, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace gbmoe {
namespace {

constexpr int BM = 128;          // weight rows per MMA (M)
// K elements per pipeline stage (template parameter BK): 64 = one 128-byte
// swizzled row (128B swizzle), 32 = one 64-byte row (64B swizzle).
constexpr int BOX_ROWS = 16;     // granularity of the token dimension (MMA N step, smallest box)
constexpr int EPI_COLS = 16;     // tokens per epilogue pass (one tcgen05.ld x16)
constexpr int EPI_WARPS = 8;     // two warps per TMEM lane quarter, alternating passes
constexpr int LOADER_WARPS = 4;  // B ring
constexpr int LOADER_THREADS = 32 * LOADER_WARPS;
constexpr int LOADER_WARP0 = 2 + EPI_WARPS;
constexpr int MAX_GROUPS = 1024;
constexpr int NUM_THREADS = 32 * (LOADER_WARP0 + LOADER_WARPS);
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // default limit of the bounded waits
constexpr uint64_t kDrainLimitNs = 200000000ull;
// A CTA pair's odd CTA lands its copies on the even CTA's barriers, so on
// the error path neither CTA can observe all of the pair's copies complete:
// both wait this long (copies take microseconds) before the pair exits.
constexpr uint64_t kPairSettleNs = 2000000ull;
constexpr int kCopyLag = 2;      // token stages in flight on the cp.async path (x2 for rings of 8+)

// Operand / epilogue modes of the kernel template.
//   kSwiGLU:   A0 = W_gate rows, A1 = W_up rows of the same 128-row block;
//              out = bf16(silu(g) * u) (the gate/up GEMM)
//   kDown:     A0 = 128 W_down rows; out = fp32 accumulator
//   kDownPair: A0, A1 = two consecutive 128-row blocks of W_down (256 output
//              columns per tile sharing one token operand); out = fp32
//   kFused:    kSwiGLU tiles, then kDownPair tiles, in one launch
constexpr int kSwiGLU = 0, kDown = 1, kDownPair = 2, kFused = 3;

// Shared memory: a ring of SA weight stages (NUM_A boxes of 128 rows x BK)
// and a ring of SB token stages (up to BN rows x BK); EB bytes per element
// (2: bf16, 1: FP8 E4M3), a stage row is BK * EB = 128 (or 64) bytes.
//
// MX block scales (MXS = 1): TMEM holds, after the accumulators, one group
// of scale columns per token stage: 4 columns per A operand and BN/32 for the
// token rows.  Column j of a group holds, in lane r of every lane quarter,
// the four scale bytes (the stage's four 32-element K blocks, byte b = block
// b) of row 32j + r of that operand.
//
// CTA pairs (CG = 2): a tile is computed by two CTAs of a cluster with one
// tcgen05.mma of M = 256 per A operand, issued by the even CTA; each CTA
// stages its own 128 rows of every A operand and half of the tile's token
// rows (BN / 2 per stage), and holds its 128 output rows for all BN tokens in
// its own tensor memory.  With MX block scales each CTA also stages the scale
// chunks of its own weight rows (by TMA, completing on the even CTA's weight
// barrier) and those of all the tile's token rows; the even CTA's
// tcgen05.cp.cta_group::2 copies each CTA's chunks into its own tensor memory,
// where the pair's block-scaled MMA reads them.
template <int NUM_A, int BN, int SA, int SB, int ACC_BUFS, int BK, int EB = 2, int MXS = 0,
          int CG = 1>
struct Layout {
    static constexpr int ROW_BYTES = BK * EB;
    static constexpr int A_BYTES = BM * ROW_BYTES;
    static constexpr int A_STAGE = NUM_A * A_BYTES;
    static constexpr int B_BYTES = (BN / CG) * ROW_BYTES;
    static constexpr int ACC_COLS = NUM_A * BN;
    static constexpr int SF_BASE = ACC_BUFS * ACC_COLS;
    // MX: per token stage one 512-byte chunk of scale words per A operand and
    // per (up to) 128 token rows, 4 TMEM columns each
    static constexpr int SFB_CHUNKS = (BN + 127) / 128;
    static constexpr int SF_CHUNKS = NUM_A + SFB_CHUNKS;
    static constexpr int SF_STAGE_COLS = 4 * SF_CHUNKS;
    static constexpr int TMEM_USED = SF_BASE + (MXS ? SB * SF_STAGE_COLS : 0);
    static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
    static constexpr int TABLE_INTS = MAX_GROUPS + 4;
    static constexpr int OFF_B = SA * A_STAGE;
    static constexpr int OFF_TBS = OFF_B + SB * B_BYTES;      // prefix of token blocks
    static constexpr int OFF_GSTART = OFF_TBS + TABLE_INTS * 4;
    static constexpr int OFF_GCNT = OFF_GSTART + TABLE_INTS * 4;
    static constexpr int OFF_SCAN = OFF_GCNT + TABLE_INTS * 4;
    static constexpr int OFF_BARS = OFF_SCAN + NUM_THREADS * 4 + 16;
    static constexpr int NUM_BARS = 2 * SA + 2 * SB + 4 + 1;
    static constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;
    // MX: the scale words of a stage's TMEM columns as 512-byte chunks of 32
    // rows x 16 bytes (row r = the four columns of lane r): the token rows'
    // chunks with each token stage (staged by the loaders), the weights'
    // chunks with each weight stage (copied whole by the weight producer from
    // the pre-tiled scale arrays)
    static constexpr int OFF_SFS = (OFF_MISC + 16 + 127) / 128 * 128;
    static constexpr int SFS_BYTES = MXS ? SB * SFB_CHUNKS * 512 : 0;
    static constexpr int OFF_ASF = OFF_SFS + SFS_BYTES;
    static constexpr int ASF_BYTES = MXS ? SA * NUM_A * 512 : 0;
    // CTA pairs and the one-SM FP8 tiles of 128 tokens: per epilogue warp a
    // 2 KB staging block (16 tokens x 32 outputs) for the epilogue's TMA
    // stores (used where the launch encoded the output map)
    static constexpr bool EPI_TMA = CG == 2 || (EB == 1 && !MXS && BN == 128 && ACC_BUFS == 2);
    static constexpr int OFF_EPI = (OFF_ASF + ASF_BYTES + 127) / 128 * 128;
    static constexpr int END = OFF_EPI + (EPI_TMA ? EPI_WARPS * 2048 : 0);
    static constexpr int SMEM_BYTES = END + 1024;  // slack to align the base to 1024
    static_assert(TMEM_USED <= 512 && (MXS || TMEM_USED == TMEM_COLS), "TMEM columns");
    static_assert(!MXS || (EB == 1 && BK == 128), "MX stages hold four 32-element K blocks");
    static_assert(!MXS || BN <= 256, "at most two chunks of 128 token rows' scales");
    static_assert(A_STAGE % 1024 == 0 && B_BYTES % 1024 == 0, "stages keep 1024-byte alignment");
    static_assert(ROW_BYTES == 128 || (EB == 2 && ROW_BYTES == 64),
                  "stage K is one 128- or 64-byte swizzled row");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(SA >= 2 && SB >= 2 && SA <= 16 && SB <= 16, "ring depth");
    static_assert(BN % BOX_ROWS == 0 && BN % (2 * EPI_COLS) == 0 && BN <= 256, "tile width");
    static_assert(CG == 1 || (CG == 2 && BN % 32 == 0 && (MXS || BN % 64 == 0)), "CTA-pair tiles");
};

// Tensor maps of one GEMM: the weight operand (a0, a1) and the token operand
// with 16/32/64/128-row boxes.
struct GemmMaps {
    CUtensorMap a0, a1, b16, b32, b64, b128;
    // MX on CTA pairs: the tiled weight scale chunks (512-byte rows) of a0, a1
    CUtensorMap s0, s1;
    // the output (the down GEMM's fp32 y or the gate/up GEMM's bf16
    // activation) in 16-token x 32-column boxes for the epilogue's TMA
    // stores: encoded by the CTA-pair launches (not the MX gate/up, whose
    // epilogue writes E4M3 codes) and the one-SM FP8-row down launch, which
    // then set GemmArgs::tma_out
    CUtensorMap o;
};

struct GemmArgs {
    const int32_t* offsets;  // [groups + 1] or null: one group of n_rows
    int groups;
    int n_rows;              // rows of the token operand
    int R;                   // weight rows per group (I for gate/up, H for down)
    int K;                   // reduction length
    void* out;               // [n_rows, R]: bf16 (gate/up + SwiGLU) or fp32 (down)
    int* status;
    // Gathered token operand of the first GEMM (null: rows of the B maps):
    // row r of the operand is gather_src[gather_rows[r]], gather_src [src_rows, K].
    const int32_t* gather_rows;
    const void* gather_src;
    int src_rows;
    int act;                 // gated activation of the gate/up epilogue (GBMOE_ACT_*)
    // FP8 operands: the accumulator of output (row r, token column n) is
    // scaled by tok_scale[token of n] and by w_scale0[weight row] (the gate, or
    // the down weight; w_scale1: the up weight); null for bf16 operands
    const float* tok_scale;
    const float* w_scale0;
    const float* w_scale1;
    // MX block scales (UE8M0 bytes, one per 32 K-elements of a row; null
    // otherwise): of the token operand [rows, K/32] (rows of gather_src, or of
    // the operand), of the weights (w_sf0: gate / down, w_sf1: up), and of the
    // activation the gate/up epilogue writes quantized (out_sf [n_rows, R/32];
    // out then holds its E4M3 codes [n_rows, R]); a_fmt: the weights' type
    // code in the instruction descriptor (0 E4M3, 5 E2M1)
    const uint8_t* tok_sf;
    const uint8_t* w_sf0;
    const uint8_t* w_sf1;
    uint8_t* out_sf;
    uint32_t a_fmt;
    // wall-clock limit of every bounded pipeline wait (set at launch from the
    // process-wide setting; the drains of the error path keep their own)
    uint64_t wait_ns;
    // 1: the output tensor map (maps.o) is encoded, so the epilogue may write
    // whole 16-token blocks with TMA stores
    int tma_out;
};

// The second GEMM of the fused mode (paired down tiles) and the per-group
// count of published gate/up tiles (zeroed before the launch).
struct FusedArgs {
    int R, K;                // H, I
    float* out;              // y [n_rows, H]
    int* ready;              // [groups]
};

struct Tile {
    int p, rblk, row0, n_valid;
};

// A group of cnt rows is cut into token blocks of equal size (a multiple of
// G = 16, or 32 for CTA pairs, at most BN): blocks of one weight tile then
// take the same time and the CTAs running them stay in step, sharing the
// weight tile through L2.
__device__ __forceinline__ int block_rows(int cnt, int BN, int G) {
    const int tb = (cnt + BN - 1) / BN;
    return tb == 0 ? BN : ((cnt + tb - 1) / tb + G - 1) / G * G;
}
__device__ __forceinline__ int token_blocks(int cnt, int BN, int G) {
    const int rpb = block_rows(cnt, BN, G);
    return (cnt + rpb - 1) / rpb;
}

// Tile tau of a GEMM with `rb` weight blocks per group; tbs[p] is the number
// of token blocks of groups < p, so group p owns tiles [tbs[p]*rb, tbs[p+1]*rb).
__device__ __forceinline__ Tile decode_tile(int tau, const int* tbs, const int* gstart,
                                            const int* gcnt, int P, int rb, int BN, int G) {
    int lo = 0, hi = P;  // largest p with tbs[p] * rb <= tau
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tbs[mid] * rb <= tau) lo = mid; else hi = mid;
    }
    const int p = lo;
    const int cnt = gcnt[p];
    const int rpb = block_rows(cnt, BN, G);
    const int tb = (cnt + rpb - 1) / rpb;
    const int local = tau - tbs[p] * rb;
    Tile t;
    t.p = p;
    t.rblk = local / tb;
    const int tblk = local - t.rblk * tb;
    t.row0 = gstart[p] + tblk * rpb;
    t.n_valid = min(rpb, cnt - tblk * rpb);
    return t;
}

// Barrier over `NT` threads on named barrier `ID` that also ANDs a flag
// across them, so that all take the same branch after a bounded wait.
template <int ID, int NT>
__device__ __forceinline__ bool bar_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(ID), "n"(NT)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool epi_bar_all(bool v) { return bar_all<1, 32 * EPI_WARPS>(v); }
__device__ __forceinline__ void epi_bar_sync() {
    asm volatile("bar.sync 2, %0;" ::"n"(32 * EPI_WARPS) : "memory");
}
__device__ __forceinline__ bool loader_bar_all(bool v) { return bar_all<3, LOADER_THREADS>(v); }

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add_gpu(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Order this thread's generic-proxy global accesses with its async-proxy
// (TMA) ones.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Order this thread's completed generic-proxy shared-memory writes (cp.async)
// before async-proxy reads of them (tcgen05.mma).
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst),
                 "l"(src), "l"(pol)
                 : "memory");
}
// 4-byte copy; with valid == false the destination is zero-filled and the
// source is not read
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}
// TMA store of one box from shared memory (bulk async-group of this thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global into shared memory, completing its bytes on the mbarrier.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}
template <int N>  // all but the newest N groups landed
__device__ __forceinline__ void cp_async_wait_newest() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The gated activations (the result is rounded to bf16, so the fast
// exponential and division -- a few ulp of fp32 -- are far below its ulp):
// silu(g) * u = g * u / (1 + e^-g); the clipped variant caps the gate at 7,
// clamps the up projection to [-7, 7] and uses sigmoid(1.702 g) (u + 1);
// GeGLU with erf, or with the tanh approximation of the normal CDF.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}
__device__ __forceinline__ float gated_act(int act, float g, float u) {
    switch (act) {
        case GBMOE_ACT_SWIGLU_OAI: {
            const float gc = fminf(g, 7.0f);
            const float uc = fminf(fmaxf(u, -7.0f), 7.0f);
            return __fdividef(gc, 1.0f + __expf(-1.702f * gc)) * (uc + 1.0f);
        }
        case GBMOE_ACT_GEGLU:
            return 0.5f * g * (1.0f + erff(g * 0.70710678118654752f)) * u;
        case GBMOE_ACT_GEGLU_TANH:
            return 0.5f * g * (1.0f + tanhf(0.79788456080286536f * (g + 0.044715f * g * g * g))) *
                   u;
        default:
            return silu_mul(g, u);
    }
}

template <int NUM_A, int BN, int SA, int SB, int MODE, int ACC_BUFS, int BK, int EB = 2,
          int MXS = 0, int CG = 1>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ GemmMaps m1, const __grid_constant__ GemmMaps m2,
                    const GemmArgs args, const FusedArgs fz) {
    constexpr bool FUSED = MODE == kFused;
    constexpr int MODE1 = FUSED ? kSwiGLU : MODE;  // mode of the first GEMM's tiles
    static_assert(MODE1 != kDown || NUM_A == 1, "down tiles have one A operand");
    static_assert(MODE1 == kDown || NUM_A == 2, "gate/up and paired tiles have two");
    constexpr bool PAIR = CG == 2;
    static_assert(!PAIR || !FUSED, "CTA pairs run the two-launch GEMMs");
    constexpr int TG = 16 * CG;  // token-block granularity (an MMA N step per CTA of the tile)
    using L = Layout<NUM_A, BN, SA, SB, ACC_BUFS, BK, EB, MXS, CG>;
    static_assert(EB == 2 || !FUSED, "the FP8 path runs its GEMMs as two launches");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    int* tbs = reinterpret_cast<int*>(smem + L::OFF_TBS);
    int* gstart = reinterpret_cast<int*>(smem + L::OFF_GSTART);
    int* gcnt = reinterpret_cast<int*>(smem + L::OFF_GCNT);
    int* scan = reinterpret_cast<int*>(smem + L::OFF_SCAN);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BARS);
    uint64_t* afull = bars;
    uint64_t* aempty = afull + SA;
    uint64_t* bfull = aempty + SA;
    // with rings of equal depth the two rings advance in lockstep: one
    // barrier frees a weight stage and a token stage (one MMA commit less per
    // K stage; every tcgen05 instruction costs the issuing thread tens of
    // cycles)
    constexpr bool ONE_EMPTY = SA == SB;
    uint64_t* bempty = ONE_EMPTY ? aempty : bfull + SB;
    uint64_t* tfull = bfull + 2 * SB;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = args.groups;
    const uint64_t wait_ns = args.wait_ns;
    // CTA pairs: cluster rank (the even CTA issues the MMAs) and the tile
    // stream shared by the pair
    const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = crank == 0u;
    const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int nunits = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    constexpr int CROWS1 = MODE1 == kDownPair ? 2 * BM : BM;  // weight rows per CTA and tile
    constexpr int WROWS1 = CROWS1 * CG;                       // weight rows per first-GEMM tile
    const int rb1 = args.R / WROWS1;
    const int rb2 = FUSED ? fz.R / (2 * BM) : 0;

    // ---- set-up: barriers, TMEM, tile table
    if (tid == 0) {
        // CTA pairs: the odd CTA's copies complete on the even CTA's full
        // barriers (whose expected bytes the even CTA sets for both halves);
        // gathered token stages also count the odd CTA's publication, and the
        // accumulator barriers the odd CTA's epilogue warps
        const uint32_t peer = (PAIR && leader) ? 1u : 0u;
        for (int s = 0; s < SA; ++s) {
            mbar_init(afull + s, 1);
            mbar_init(aempty + s, 1);
        }
        // MX token stages loaded by TMA complete on two arrivals: the lead
        // thread's (with the copies' bytes) and the published scale columns
        const uint32_t bfull_count = (MXS && args.gather_rows == nullptr) ? 2u : 1u;
        for (int s = 0; s < SB; ++s) {
            mbar_init(bfull + s, bfull_count + ((args.gather_rows != nullptr || MXS) ? peer : 0u));
            if (!ONE_EMPTY) mbar_init(bempty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull + b, 1);
            mbar_init(tempty + b, EPI_WARPS * (1 + peer));
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&m1.a0);
        tma_prefetch_desc(&m1.a1);
        tma_prefetch_desc(&m1.b16);
        tma_prefetch_desc(&m1.b128);
        if (FUSED) {
            tma_prefetch_desc(&m2.a0);
            tma_prefetch_desc(&m2.b16);
            tma_prefetch_desc(&m2.b128);
        }
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(tmem_base_s, L::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_base_s, L::TMEM_COLS);
            tmem_relinquish();
        }
    }
    {
        // tbs[p] = token blocks of groups < p
        const int seg = (P + NUM_THREADS - 1) / NUM_THREADS;
        const int s0 = min(P, tid * seg), s1 = min(P, s0 + seg);
        int local = 0;
        for (int p = s0; p < s1; ++p) {
            int off = 0, cnt = args.n_rows;
            if (args.offsets) {
                off = args.offsets[p];
                cnt = args.offsets[p + 1] - off;
                if (cnt < 0 || off < 0 || off + cnt > args.n_rows) {
                    record_error(args.status, GBMOE_ERR_DEVICE);
                    off = 0;
                    cnt = 0;
                }
            }
            gstart[p] = off;
            gcnt[p] = cnt;
            local += token_blocks(cnt, BN, TG);
        }
        scan[tid] = local;
        __syncthreads();
        if (tid == 0) {
            int run = 0;
            for (int i = 0; i < NUM_THREADS; ++i) {
                const int v = scan[i];
                scan[i] = run;
                run += v;
            }
            scan[NUM_THREADS] = run;
        }
        __syncthreads();
        int run = scan[tid];
        for (int p = s0; p < s1; ++p) {
            tbs[p] = run;
            run += token_blocks(gcnt[p], BN, TG);
        }
        if (tid == 0) tbs[P] = scan[NUM_THREADS];
    }
    tc_fence_before();
    __syncthreads();
    // a pair's barriers are initialised before either CTA arrives on the other's
    if (PAIR) cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_base_s;
    const int T1 = tbs[P] * rb1;                    // tiles of the first GEMM
    const int total = T1 + (FUSED ? tbs[P] * rb2 : 0);

    // tile tau -> (which GEMM, tile); the second GEMM exists only when fused
    auto job = [&](int tau, bool& second, Tile& tl) {
        second = FUSED && tau >= T1;
        tl = second ? decode_tile(tau - T1, tbs, gstart, gcnt, P, rb2, BN, TG)
                    : decode_tile(tau, tbs, gstart, gcnt, P, rb1, BN, TG);
    };

    // ---------------------------------------------------------- roles
    if (warp == 0 && lane == 0) {
        // A producer: weight boxes by TMA.  A weight tile read by one CTA is
        // streamed through L2 (evict first); one shared by several token
        // blocks stays at normal priority until the other CTAs have read it.
        const uint64_t pol_once = l2_policy_evict_first(), pol_shared = l2_policy_evict_normal();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t armed = 0;          // bit s: stage s has been armed at least once
        uint32_t armed_phase = 0;    // bit s: parity of its last armed phase
        for (int tau = unit; tau < total && !*abort_flag; tau += nunits) {
            bool second;
            Tile tl;
            job(tau, second, tl);
            const GemmMaps& m = second ? m2 : m1;
            const int mode = second ? kDownPair : MODE1;
            const int R = second ? fz.R : args.R;
            const int KB = (second ? fz.K : args.K) / BK;
            // this CTA's weight rows of the tile (a pair's odd CTA: the second half)
            const int crows = mode == kDownPair ? 2 * BM : BM;
            const int a_row = tl.p * R + (tl.rblk * CG + static_cast<int>(crank)) * crows;
            const uint64_t pol_w = token_blocks(gcnt[tl.p], BN, TG) > 1 ? pol_shared : pol_once;
            // an E2M1 box lands as one byte per element (16 codes in the first
            // 8 bytes of every 16) but completes with its packed size
            const uint32_t a_tx = ((MXS && args.a_fmt == 5u) ? L::A_BYTES / 2 : L::A_BYTES) +
                                  (MXS ? 512u : 0u);
            // MX: the weight scale chunks of this tile's 128-row blocks, one
            // 512-byte run per (row block, K stage) in the pre-tiled arrays
            const int ks_per_row = args.K / BK;
            const size_t sf_tile0 = static_cast<size_t>(a_row / BM) * ks_per_row;
            bool ok = true;
            for (int kb = 0; kb < KB; ++kb) {
                if (!mbar_wait_bounded(aempty + stage, phase ^ 1u, abort_flag, args.status,
                                       wait_ns)) {
                    ok = false;
                    break;
                }
                uint8_t* sA = smem + stage * L::A_STAGE;
                if (PAIR && !leader) {
                    // the odd CTA's half lands here and completes on the even
                    // CTA's barrier, which expects it
                    const uint32_t lb = mapa_shared(smem_u32(afull + stage), 0u);
                    tma_load_2d_pair(sA, &m.a0, lb, kb * BK, a_row, pol_w);
                    if (mode == kSwiGLU)
                        tma_load_2d_pair(sA + L::A_BYTES, &m.a1, lb, kb * BK, a_row, pol_w);
                    if (mode == kDownPair)
                        tma_load_2d_pair(sA + L::A_BYTES, &m.a0, lb, kb * BK, a_row + BM, pol_w);
                    if (MXS) {
                        uint8_t* sf = smem + L::OFF_ASF + stage * (NUM_A * 512);
                        const int ch = static_cast<int>(sf_tile0) + kb;
                        tma_load_2d_pair(sf, &m.s0, lb, 0, ch, pol_w);
                        if (mode == kSwiGLU) tma_load_2d_pair(sf + 512, &m.s1, lb, 0, ch, pol_w);
                        if (mode == kDownPair)
                            tma_load_2d_pair(sf + 512, &m.s0, lb, 0, ch + ks_per_row, pol_w);
                    }
                } else {
                    mbar_arrive_expect_tx(afull + stage, NUM_A * a_tx * CG);
                    tma_load_2d(sA, &m.a0, afull + stage, kb * BK, a_row, pol_w);
                    if (mode == kSwiGLU)
                        tma_load_2d(sA + L::A_BYTES, &m.a1, afull + stage, kb * BK, a_row, pol_w);
                    if (mode == kDownPair)
                        tma_load_2d(sA + L::A_BYTES, &m.a0, afull + stage, kb * BK, a_row + BM,
                                    pol_w);
                    if (MXS && PAIR) {
                        uint8_t* sf = smem + L::OFF_ASF + stage * (NUM_A * 512);
                        const int ch = static_cast<int>(sf_tile0) + kb;
                        tma_load_2d(sf, &m.s0, afull + stage, 0, ch, pol_w);
                        if (mode == kSwiGLU) tma_load_2d(sf + 512, &m.s1, afull + stage, 0, ch, pol_w);
                        if (mode == kDownPair)
                            tma_load_2d(sf + 512, &m.s0, afull + stage, 0, ch + ks_per_row, pol_w);
                    } else if (MXS) {
                        uint8_t* sf = smem + L::OFF_ASF + stage * (NUM_A * 512);
                        // gate/up: the gate's and the up's chunks of the same
                        // rows; paired down: the two consecutive row blocks
                        const size_t c0 = (sf_tile0 + kb) * 512;
                        bulk_load(sf, args.w_sf0 + c0, 512, afull + stage, pol_w);
                        if (mode == kSwiGLU)
                            bulk_load(sf + 512, args.w_sf1 + c0, 512, afull + stage, pol_w);
                        if (mode == kDownPair)
                            bulk_load(sf + 512, args.w_sf0 + c0 + static_cast<size_t>(ks_per_row) * 512,
                                      512, afull + stage, pol_w);
                    }
                }
                armed |= 1u << stage;
                armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == SA) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
        }
        if (*abort_flag && PAIR) {
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < kPairSettleNs) {
            }
        } else if (*abort_flag) {  // let every copy this thread issued land before exit
            for (int s = 0; s < SA; ++s)
                if ((armed >> s) & 1u)
                    mbar_wait_timeout(afull + s, (armed_phase >> s) & 1u, kDrainLimitNs);
        } else if (PAIR) {
            // every stage consumed: the even CTA's MMA commits to this CTA's
            // barriers have all landed before the pair exits
            for (int i = 0; i < SA; ++i) {
                mbar_wait_timeout(aempty + stage, phase ^ 1u, kDrainLimitNs);
                if (++stage == SA) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp >= LOADER_WARP0) {
        // B loaders: token rows, by TMA (lead thread) or gathered by cp.async
        // (every loader thread copies one fixed 16-byte column of every 16th
        // row of the tile).  A gathered stage is published once a newer one
        // has been issued (two stages in flight) and every loader's
        // copies of it have landed: each thread waits for its own older
        // copies and fences them for the tensor cores' proxy, and the barrier
        // orders all of that before the lead thread's arrive.  A stage is
        // published before the lead thread waits for the slot SB stages
        // later: no cycle.  MX block scales travel the same way (scale words
        // staged by cp.async; with TMA rows the stage completes on the lead
        // thread's arrive and the scales' publishing arrive).
        const int li = tid - 32 * LOADER_WARP0;
        const bool lead = li == 0;
        const int chunk = li & 7;       // 16-byte column of the 128-byte row
        const int rbase = li >> 3;      // rows rbase + 16u
        constexpr int RSTEP = LOADER_THREADS / 8;
        constexpr int RPT = (BN / CG) / RSTEP;  // rows per thread
        static_assert((BN / CG) % RSTEP == 0, "loader rows");
        const uint64_t pol_x = l2_policy_evict_last();
        // without gathered rows the lead thread alone streams the B ring
        // (with MX block scales every loader thread also stages scale words)
        const bool solo = args.gather_rows == nullptr && !MXS;
        const int kq = args.K / 32;     // scale bytes per row
        // MX: loader warp w stages scale column w of every 4-column group
        // (rows 32 w + lane of each A operand; token rows 32 (w + 4 c) + lane)
        const int wi = warp - LOADER_WARP0;
        auto all_agree = [&](bool v) { return solo ? v : loader_bar_all(v); };
        int stage = 0;
        uint32_t phase = 0;
        // staged (cp.async) stages in flight: up to LAG copy groups, the
        // oldest published once a new one is issued; with LAG <= SB a stage
        // is always published before the lead thread waits for a slot that
        // needs it consumed
        constexpr int LAG = SB >= 8 ? 2 * kCopyLag : kCopyLag;
        int npend = 0, last = 0;        // unpublished staged stages: the npend up to `last`
        auto publish_oldest = [&](bool go) {
            const int old = (last - (npend - 1) + SB) % SB;
            fence_proxy_async_shared();
            const bool all = loader_bar_all(go);
            // relaxed arrivals: every loader's copies of the stage have landed
            // and been fenced before the barrier, and a release here would
            // also wait for the newer stage's copies in flight
            if (lead && all) {
                if (PAIR && !leader)  // the pair's MMA waits on the even CTA's barrier
                    mbar_arrive_remote_relaxed(mapa_shared(smem_u32(bfull + old), 0u));
                else
                    mbar_arrive_relaxed(bfull + old);
            }
            --npend;
        };
        uint32_t armed = 0, armed_phase = 0;  // TMA-armed stages (lead thread)
        bool ok = !solo || lead;
        for (int tau = unit; ok && tau < total; tau += nunits) {
            bool second;
            Tile tl;
            job(tau, second, tl);
            const bool gather = !second && args.gather_rows != nullptr && L::ROW_BYTES == 128;
            // this CTA's token rows of the tile: all of them, or for a CTA
            // pair one half of the MMA's N (the odd CTA the second)
            const int n_mma = (tl.n_valid + TG - 1) / TG * TG;
            const int my0 = static_cast<int>(crank) * (n_mma / CG);
            const int my_valid = max(0, min(n_mma / CG, tl.n_valid - my0));
            if (FUSED && second) {
                // publish the pending gathered stages before waiting: the MMA
                // needs them to finish the very gate/up tiles waited for
                if (npend > 0) {
                    cp_async_wait_all();
                    while (npend > 0) publish_oldest(true);
                }
                // all gate/up tiles of this group must have published their rows
                bool got = true;
                if (lead) {
                    const int need = rb1 * token_blocks(gcnt[tl.p], BN, TG);
                    const uint64_t t0 = global_timer_ns();
                    for (uint32_t it = 0; ld_acquire_gpu(fz.ready + tl.p) < need; ++it) {
                        if ((it & 63u) == 63u) {
                            if (*abort_flag) { got = false; break; }
                            if (global_timer_ns() - t0 > wait_ns) {
                                *abort_flag = 1;
                                record_error(args.status, GBMOE_ERR_TIMEOUT);
                                got = false;
                                break;
                            }
                        }
                    }
                    fence_proxy_async_global();
                }
                if (!all_agree(got)) {
                    ok = false;
                    break;
                }
            }
            const GemmMaps& m = second ? m2 : m1;
            const int KB = (second ? fz.K : args.K) / BK;
            const int n_load = (my_valid + BOX_ROWS - 1) / BOX_ROWS * BOX_ROWS;
            // gathered rows of this thread: source element offsets (-1: none)
            int64_t src[RPT];
            if (gather) {
#pragma unroll
                for (int u = 0; u < RPT; ++u) {
                    const int r = rbase + RSTEP * u;
                    src[u] = -1;
                    if (r < my_valid) {
                        int t = args.gather_rows[tl.row0 + my0 + r];
                        if (t < 0 || t >= args.src_rows) {
                            record_error(args.status, GBMOE_ERR_DEVICE);
                            t = 0;
                        }
                        src[u] = static_cast<int64_t>(t) * args.K * EB + chunk * 16;
                    }
                }
            }
            // MX: the token scale rows this thread stages
            int64_t sfb_row[L::SFB_CHUNKS];
            if (MXS) {
#pragma unroll
                for (int j = 0; j < L::SFB_CHUNKS; ++j) {
                    const int n = 32 * (wi + 4 * j) + lane;
                    sfb_row[j] = -1;
                    if (n < tl.n_valid) {
                        int t = tl.row0 + n;
                        if (args.gather_rows) {
                            t = args.gather_rows[t];
                            if (t < 0 || t >= args.src_rows) {
                                record_error(args.status, GBMOE_ERR_DEVICE);
                                t = 0;
                            }
                        }
                        sfb_row[j] = t;
                    }
                }
            }
            for (int kb = 0; kb < KB; ++kb) {
                bool free_ok = true;
                if (lead)
                    free_ok = mbar_wait_bounded(bempty + stage, phase ^ 1u, abort_flag,
                                                args.status, wait_ns);
                if (!all_agree(free_ok)) {
                    ok = false;
                    break;
                }
                if (MXS) {
                    // this stage's token scale words (four K blocks of a row
                    // each) into its chunks, in the stage's copy group
                    const uint32_t sfs = smem_u32(smem + L::OFF_SFS) +
                                         stage * (L::SFB_CHUNKS * 512) + lane * 16 + wi * 4;
#pragma unroll
                    for (int j = 0; j < L::SFB_CHUNKS; ++j) {
                        const bool v = sfb_row[j] >= 0;
                        cp_async4(sfs + j * 512,
                                  args.tok_sf + (v ? sfb_row[j] * kq + kb * 4 : 0), v);
                    }
                }
                uint8_t* sB = smem + L::OFF_B + stage * L::B_BYTES;
                if (gather) {
                    const uint32_t sb = smem_u32(sB);
#pragma unroll
                    for (int u = 0; u < RPT; ++u) {
                        if (src[u] >= 0) {
                            const int r = rbase + RSTEP * u;
                            const uint32_t dst = sb + r * 128 + ((chunk ^ (r & 7)) << 4);
                            cp_async16(dst,
                                       static_cast<const uint8_t*>(args.gather_src) + src[u] +
                                           static_cast<int64_t>(kb) * L::ROW_BYTES,
                                       pol_x);
                        }
                    }
                } else if (lead) {
                    // the even CTA of a pair expects both halves' bytes; the
                    // odd CTA's copies complete on that barrier
                    const uint32_t lb = mapa_shared(smem_u32(bfull + stage), 0u);
                    if (!PAIR || leader) {
                        int n_all = n_load;
                        if (PAIR) {
                            const int pv = max(0, min(n_mma / CG, tl.n_valid - n_mma / CG));
                            n_all += (pv + BOX_ROWS - 1) / BOX_ROWS * BOX_ROWS;
                        }
                        mbar_arrive_expect_tx(bfull + stage, n_all * L::ROW_BYTES);
                    }
                    // token rows in as few boxes as possible (128/64/32/16 rows)
                    for (int off = 0; off < n_load;) {
                        const int rem = n_load - off;
                        const int box = rem >= 128 ? 128 : rem >= 64 ? 64 : rem >= 32 ? 32 : 16;
                        const CUtensorMap* mb = box == 128 ? &m.b128 : box == 64 ? &m.b64
                                              : box == 32 ? &m.b32 : &m.b16;
                        if (PAIR && !leader)
                            tma_load_2d_pair(sB + off * L::ROW_BYTES, mb, lb, kb * BK,
                                             tl.row0 + my0 + off, pol_x);
                        else
                            tma_load_2d(sB + off * L::ROW_BYTES, mb, bfull + stage, kb * BK,
                                        tl.row0 + my0 + off, pol_x);
                        off += box;
                    }
                    armed |= 1u << stage;
                    armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
                }
                if (gather || MXS) {
                    cp_async_commit();
                    last = stage;
                    // publish the oldest staged stage: this thread's copies of
                    // it have landed (only the newest LAG - 1 groups may be in
                    // flight) and are fenced for the tensor cores' proxy, and
                    // the barrier orders every loader's part before the lead
                    // thread's arrive
                    if (++npend == LAG) {
                        cp_async_wait_newest<LAG - 1>();
                        publish_oldest(true);
                    }
                }
                if (++stage == SB) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (npend > 0) {  // publish the last staged stages
            cp_async_wait_all();
            while (npend > 0) publish_oldest(ok);
        }
        cp_async_wait_all();
        if (lead && *abort_flag && PAIR) {
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < kPairSettleNs) {
            }
        } else if (lead && *abort_flag) {  // let every TMA copy issued land before exit
            for (int s = 0; s < SB; ++s)
                if ((armed >> s) & 1u)
                    mbar_wait_timeout(bfull + s, (armed_phase >> s) & 1u, kDrainLimitNs);
        } else if (PAIR && lead) {
            // every stage consumed (the even CTA's commits have landed here)
            for (int i = 0; i < SB; ++i) {
                mbar_wait_timeout(bempty + stage, phase ^ 1u, kDrainLimitNs);
                if (++stage == SB) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // MMA issuer (for a pair: the even CTA, M = 256 over both CTAs'
        // shared memory; its commits signal the stage and accumulator
        // barriers of both CTAs)
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            return mbar_wait_bounded(bar, parity, abort_flag, args.status, wait_ns);
        };
        auto commit = [&](uint64_t* bar) {
            if (PAIR)
                umma_commit_pair_mc(bar, 0x3);
            else
                umma_commit(bar);
        };
        int as = 0, bs = 0, acc = 0;
        uint32_t aph = 0, bph = 0, acc_phase = 0;
        bool issued = false;
        for (int tau = unit; tau < total && !*abort_flag; tau += nunits) {
            bool second;
            Tile tl;
            job(tau, second, tl);
            const int KB = (second ? fz.K : args.K) / BK;
            const int n_mma = ((tl.n_valid + TG - 1) / TG) * TG;
            const uint32_t idesc = MXS ? idesc_mx(BM * CG, n_mma, args.a_fmt, 0u, 0u)
                                 : EB == 2 ? idesc_bf16_f32(BM * CG, n_mma)
                                           : idesc_e4m3_f32(BM * CG, n_mma);
            // the accumulator is free once both CTAs' epilogues have drained it
            if (!(PAIR ? mbar_wait_bounded_cluster(tempty + acc, acc_phase ^ 1u, abort_flag,
                                                   args.status, wait_ns)
                       : wait(tempty + acc, acc_phase ^ 1u)))
                break;
            tc_fence_after();
            const uint32_t d0 = tmem_base + acc * L::ACC_COLS;
            bool ok = true;
            for (int kb = 0; kb < KB; ++kb) {
                if (!wait(afull + as, aph) || !wait(bfull + bs, bph)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sA = smem_u32(smem + as * L::A_STAGE);
                const uint32_t sB = smem_u32(smem + L::OFF_B + bs * L::B_BYTES);
                const uint32_t sf = tmem_base + L::SF_BASE + bs * L::SF_STAGE_COLS;
                if (MXS) {
                    // the stage's scale chunks into its TMEM columns (in order
                    // with the MMAs below)
                    // weight chunks from the weight stage, token chunks from
                    // the token stage
                    const uint32_t asf = smem_u32(smem + L::OFF_ASF) + as * (NUM_A * 512);
                    const uint32_t sfs = smem_u32(smem + L::OFF_SFS) + bs * (L::SFB_CHUNKS * 512);
#pragma unroll
                    for (int a = 0; a < NUM_A; ++a) {
                        if (PAIR)
                            tmem_cp_32x128b_warpx4_pair(sf + 4 * a, smem_desc_rows16(asf + a * 512));
                        else
                            tmem_cp_32x128b_warpx4(sf + 4 * a, smem_desc_rows16(asf + a * 512));
                    }
#pragma unroll
                    for (int c = 0; c < L::SFB_CHUNKS; ++c) {
                        if (PAIR)
                            tmem_cp_32x128b_warpx4_pair(sf + 4 * (NUM_A + c),
                                                        smem_desc_rows16(sfs + c * 512));
                        else
                            tmem_cp_32x128b_warpx4(sf + 4 * (NUM_A + c),
                                                   smem_desc_rows16(sfs + c * 512));
                    }
                }
                // one MMA covers 32 bytes of K (16 bf16 or 32 FP8 elements)
#pragma unroll
                for (int ks = 0; ks < L::ROW_BYTES / 32; ++ks) {
                    const uint64_t bdesc = smem_desc_kmajor<L::ROW_BYTES / 2>(sB + ks * 32);
#pragma unroll
                    for (int a = 0; a < NUM_A; ++a) {
                        const uint64_t adesc =
                            smem_desc_kmajor<L::ROW_BYTES / 2>(sA + a * L::A_BYTES + ks * 32);
                        const uint32_t accum = (kb > 0 || ks > 0) ? 1u : 0u;
                        if (MXS && PAIR)
                            umma_mx_pair(d0 + a * BN, adesc, bdesc,
                                         idesc | (static_cast<uint32_t>(ks) << 4) |
                                             (static_cast<uint32_t>(ks) << 29),
                                         sf + 4 * a, sf + 4 * NUM_A, accum);
                        else if (MXS)
                            umma_mx(d0 + a * BN, adesc, bdesc,
                                    idesc | (static_cast<uint32_t>(ks) << 4) |
                                        (static_cast<uint32_t>(ks) << 29),
                                    sf + 4 * a, sf + 4 * NUM_A, accum);
                        else if (PAIR && EB == 2)
                            umma_bf16_pair(d0 + a * BN, adesc, bdesc, idesc, accum);
                        else if (PAIR)
                            umma_e4m3_pair(d0 + a * BN, adesc, bdesc, idesc, accum);
                        else if (EB == 2)
                            umma_bf16(d0 + a * BN, adesc, bdesc, idesc, accum);
                        else
                            umma_e4m3(d0 + a * BN, adesc, bdesc, idesc, accum);
                    }
                }
                issued = true;
                commit(aempty + as);
                if (!ONE_EMPTY) commit(bempty + bs);
                if (++as == SA) {
                    as = 0;
                    aph ^= 1u;
                }
                if (++bs == SB) {
                    bs = 0;
                    bph ^= 1u;
                }
            }
            if (!ok) break;
            commit(tfull + acc);
            if (++acc == ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (*abort_flag && issued) {  // wait for the MMAs in flight before TMEM is freed
            if (PAIR)
                umma_commit_pair_mc(drain, 0x1);
            else
                umma_commit(drain);
            mbar_wait_timeout(drain, 0u, kDrainLimitNs);
        }
    } else if (warp >= 2 && warp < LOADER_WARP0) {
        // epilogue: TMEM -> registers -> (activation) -> global.  Warp w may
        // only read TMEM lanes 32*(w%4)..+31; the two warps of each lane
        // quarter take alternate 16-token passes.
        const int q = warp & 3;                 // TMEM lane quarter
        const int half = (warp - 2) / 4;        // which of the quarter's two warps
        const int r = q * 32 + lane;            // weight row within the tile
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tau = unit; tau < total; tau += nunits) {
            bool second;
            Tile tl;
            job(tau, second, tl);
            const bool got = mbar_wait_bounded(tfull + acc, acc_phase, abort_flag, args.status,
                                               wait_ns);
            if (!epi_bar_all(got)) break;
            tc_fence_after();
            const int mode = second ? kDownPair : MODE1;
            const bool swiglu = mode == kSwiGLU;
            const bool quant_out = MXS && swiglu;  // MX E4M3 activation codes + scales
            const int out_elem = quant_out ? 1 : swiglu ? 2 : 4;
            const int R = second ? fz.R : args.R;
            uint8_t* outp = static_cast<uint8_t*>(second ? static_cast<void*>(fz.out) : args.out);
            const int wrows = mode == kDownPair ? 2 * BM : BM;
            const int nout = mode == kDownPair ? 2 : 1;
            const uint32_t tb = tmem_base + acc * L::ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
            const size_t row_bytes = static_cast<size_t>(R) * out_elem;
            for (int c0 = half * EPI_COLS; c0 < tl.n_valid; c0 += 2 * EPI_COLS)
#pragma unroll 1
            for (int ob = 0; ob < nout; ++ob) {
                const int nr = min(EPI_COLS, tl.n_valid - c0);
                // output column: this CTA's weight rows of the tile (the odd
                // CTA of a pair holds the second half)
                const size_t col = static_cast<size_t>(tl.rblk * CG + static_cast<int>(crank)) *
                                       wrows + ob * BM + r;
                uint32_t g[16], u[16];
                tmem_ld_32x32b_x16(tb + ob * BN + c0, g);
                if (swiglu) tmem_ld_32x32b_x16(tb + BN + c0, u);
                tmem_ld_wait();
                float gv[16], uv[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    gv[c] = __uint_as_float(g[c]);
                    uv[c] = swiglu ? __uint_as_float(u[c]) : 0.0f;
                }
                if (EB == 1 && !MXS) {
                    // FP8 operands: (acc * token scale) * weight-row scale
                    const size_t wrow = static_cast<size_t>(tl.p) * R + col;
                    const float sw0 = args.w_scale0[wrow];
                    const float sw1 = swiglu ? args.w_scale1[wrow] : 0.0f;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        float st = 0.0f;
                        if (c < nr) {
                            int tok = tl.row0 + c0 + c;
                            if (args.gather_rows) {
                                tok = args.gather_rows[tok];
                                tok = (tok < 0 || tok >= args.src_rows) ? 0 : tok;
                            }
                            st = args.tok_scale[tok];
                        }
                        gv[c] = __fmul_rn(__fmul_rn(gv[c], st), sw0);
                        if (swiglu) uv[c] = __fmul_rn(__fmul_rn(uv[c], st), sw1);
                    }
                }
                float v[16];
                if (swiglu) {
                    if (args.act == GBMOE_ACT_SWIGLU) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) v[c] = silu_mul(gv[c], uv[c]);
                    } else {
#pragma unroll
                        for (int c = 0; c < 16; ++c) v[c] = gated_act(args.act, gv[c], uv[c]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 16; ++c) v[c] = gv[c];
                }
                // Lane r holds output column r for 16 consecutive token rows,
                // so for each row the 32 lanes of a warp write 32 consecutive
                // outputs (128 B of fp32 / 64 B of bf16): coalesced stores
                // straight from registers.
                uint8_t* base = outp + (static_cast<size_t>(tl.row0 + c0) * R + col) * out_elem;
                if (L::EPI_TMA && args.tma_out && !quant_out && c0 + EPI_COLS <= tl.n_valid &&
                    tl.row0 + c0 + EPI_COLS <= args.n_rows) {
                    // a whole 16-token block: staged in shared memory and written
                    // by one TMA store, so the warp hands its accumulator columns
                    // back without waiting on 16 rows of global stores (a block
                    // that would reach past the tile's rows takes the plain
                    // stores below: other tiles own the rows after it)
                    uint8_t* stg = smem + L::OFF_EPI + (warp - 2) * 2048;
                    if (lane == 0) bulk_wait_read_all();  // the previous store has read it
                    __syncwarp();
                    if (swiglu) {
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            reinterpret_cast<uint16_t*>(stg)[c * 32 + lane] = f32_to_bf16_bits(v[c]);
                    } else {
#pragma unroll
                        for (int c = 0; c < 16; ++c) reinterpret_cast<float*>(stg)[c * 32 + lane] = v[c];
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&m1.o, stg, static_cast<int>(col) - lane, tl.row0 + c0);
                        bulk_commit();
                    }
                    continue;
                }
                if (quant_out) {
                    // the activation rounded to bf16, then quantized to MX E4M3:
                    // the warp's 32 lanes are one 32-element block of each
                    // token row (max over the warp, shared exponent, codes)
                    const int blk = ((tl.rblk * CG + static_cast<int>(crank)) * BM + q * 32) / 32;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float a = bf16_bits_to_f32(f32_to_bf16_bits(v[c]));
                        // magnitudes order like their fp32 bit patterns
                        const float m = __uint_as_float(
                            __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(a))));
                        const int e = mx_block_exp(m, 8);
                        const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
                        const uint32_t code = cvt_e4m3x2(__fmul_rn(a, inv), 0.0f) & 0xffu;
                        const int row = tl.row0 + c0 + c;
                        if (c < nr && row < args.n_rows) {
                            base[c * row_bytes] = static_cast<uint8_t>(code);
                            if (lane == 0)
                                args.out_sf[static_cast<size_t>(row) * (R / 32) + blk] =
                                    static_cast<uint8_t>(e + 127);
                        }
                    }
                    continue;
                }
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    if (c < nr && tl.row0 + c0 + c < args.n_rows) {
                        if (swiglu)
                            *reinterpret_cast<uint16_t*>(base + c * row_bytes) = f32_to_bf16_bits(v[c]);
                        else
                            *reinterpret_cast<float*>(base + c * row_bytes) = v[c];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR && !leader)  // the pair's MMA waits on the even CTA's barrier
                    mbar_arrive_remote(mapa_shared(smem_u32(tempty + acc), 0u));
                else
                    mbar_arrive(tempty + acc);
            }
            if (FUSED && !second) {
                // publish this gate/up tile: its activations are in global memory
                __threadfence();
                fence_proxy_async_global();
                epi_bar_sync();
                if (warp == 2 && lane == 0) red_release_add_gpu(fz.ready + tl.p, 1);
            }
            if (++acc == ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    if (L::EPI_TMA && warp >= 2 && warp < LOADER_WARP0 && lane == 0) bulk_wait_all();
    // ---- teardown (a pair: neither CTA leaves while the other may still
    // signal its barriers or read its shared memory)
    __syncthreads();
    if (PAIR) cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

// ----------------------------------------------------------------- host
// Variant choice (measured on the decode, hash, skew and prefill routings):
// once groups average >= 96 rows, gate/up uses 256-token tiles -- on CTA
// pairs when I % 256 == 0 -- and the down GEMM pairs two 128-row W_down
// blocks over 256-token tiles (one accumulator buffer) -- on CTA pairs when
// H % 512 == 0; below 96 rows the down GEMM pairs the blocks over 128-token
// tiles with two buffers (H % 256 == 0), else 128- or 256-token
// single-block tiles.  All variants stream K in 64-wide stages
// (32-wide stages with the 64B swizzle were measured slower: per-stage costs
// outweigh the extra lookahead).  Below 96 rows per group with H % 256 == 0
// moe_forward runs the two GEMMs fused in one launch (their tiles share one
// layout).  Ring depths (weight stages, token stages) fill the shared memory.
constexpr int kBK = 64;
constexpr long kLargeGateUpRows = 96;
constexpr int kG1S_A = 4, kG1S_B = 4;
constexpr int kG1L_A = 3, kG1L_B = 3;
constexpr int kG2S_A = 6, kG2S_B = 6;
constexpr int kG2L_A = 4, kG2L_B = 4;
constexpr int kG2P_A = 4, kG2P_B = 4;
using Gemm1Small = Layout<2, 128, kG1S_A, kG1S_B, 2, kBK>;
using Gemm1Large = Layout<2, 256, kG1L_A, kG1L_B, 1, kBK>;
using Gemm2Small = Layout<1, 128, kG2S_A, kG2S_B, 2, kBK>;
using Gemm2Large = Layout<1, 256, kG2L_A, kG2L_B, 2, kBK>;
using Gemm2Pair = Layout<2, 128, kG2P_A, kG2P_B, 2, kBK>;
#define GEMM1_SMALL grouped_gemm_kernel<2, 128, kG1S_A, kG1S_B, kSwiGLU, 2, kBK>
#define GEMM1_LARGE grouped_gemm_kernel<2, 256, kG1L_A, kG1L_B, kSwiGLU, 1, kBK>
#define GEMM2_SMALL grouped_gemm_kernel<1, 128, kG2S_A, kG2S_B, kDown, 2, kBK>
#define GEMM2_LARGE grouped_gemm_kernel<1, 256, kG2L_A, kG2L_B, kDown, 2, kBK>
#define GEMM2_PAIR grouped_gemm_kernel<2, 128, kG2P_A, kG2P_B, kDownPair, 2, kBK>
// paired down blocks over 256-token tiles (the gate/up 256-token layout)
#define GEMM2_PAIR_LARGE grouped_gemm_kernel<2, 256, kG1L_A, kG1L_B, kDownPair, 1, kBK>
#define GEMM_FUSED grouped_gemm_kernel<2, 128, kG1S_A, kG1S_B, kFused, 2, kBK>
// CTA pairs (prefill-sized groups, I % 256 == 0 / H % 512 == 0): gate/up
// tiles of 2 x 128 gate and up rows x 256 tokens, and down tiles of 2 x 256
// W_down rows x 256 tokens, each CTA staging 128 token rows per stage
constexpr int kPr_A = 4, kPr_B = 4;
using GemmPairLarge = Layout<2, 256, kPr_A, kPr_B, 1, kBK, 2, 0, 2>;
#define GEMM1_CTA_PAIR grouped_gemm_kernel<2, 256, kPr_A, kPr_B, kSwiGLU, 1, kBK, 2, 0, 2>
#define GEMM2_CTA_PAIR grouped_gemm_kernel<2, 256, kPr_A, kPr_B, kDownPair, 1, kBK, 2, 0, 2>
// FP8 E4M3 operands: 128-element stages (the same 128-byte rows)
constexpr int kBK8 = 128;
using Gemm1SmallF8 = Layout<2, 128, kG1S_A, kG1S_B, 2, kBK8, 1>;
using Gemm1LargeF8 = Layout<2, 256, kG1L_A, kG1L_B, 1, kBK8, 1>;
using Gemm2PairF8 = Layout<2, 128, kG2P_A, kG2P_B, 2, kBK8, 1>;
#define GEMM1_SMALL_F8 grouped_gemm_kernel<2, 128, kG1S_A, kG1S_B, kSwiGLU, 2, kBK8, 1>
#define GEMM1_LARGE_F8 grouped_gemm_kernel<2, 256, kG1L_A, kG1L_B, kSwiGLU, 1, kBK8, 1>
#define GEMM2_PAIR_F8 grouped_gemm_kernel<2, 128, kG2P_A, kG2P_B, kDownPair, 2, kBK8, 1>
// ... and the gate/up GEMM on CTA pairs for prefill-sized groups (as bf16)
using GemmPairLargeF8 = Layout<2, 256, kPr_A, kPr_B, 1, kBK8, 1, 0, 2>;
#define GEMM1_CTA_PAIR_F8 grouped_gemm_kernel<2, 256, kPr_A, kPr_B, kSwiGLU, 1, kBK8, 1, 0, 2>

// MX block scales: 224-token tiles for groups averaging >= 96 rows -- on CTA
// pairs (below) when I % 256 == 0 / H % 512 == 0, else on one SM (two
// accumulators of 224 columns and three token stages' scale columns fill
// TMEM) -- else 128-token tiles with one accumulator buffer (the scale
// columns of the four token stages take the rest of TMEM); for groups of at
// most 32 rows on average (decode), 32-token tiles with two accumulator
// buffers and five weight and five token stages (equal depths: one commit
// per K stage)
constexpr int kMx_A = 4, kMx_B = 4;
constexpr int kMxD_A = 5, kMxD_B = 5;
constexpr long kMxDecodeRows = 32;
using GemmMx = Layout<2, 128, kMx_A, kMx_B, 1, kBK8, 1, 1>;
using GemmMxDec = Layout<2, 32, kMxD_A, kMxD_B, 2, kBK8, 1, 1>;
using GemmMxL = Layout<2, 224, 3, 3, 1, kBK8, 1, 1>;
#define GEMM1_MX_L grouped_gemm_kernel<2, 224, 3, 3, kSwiGLU, 1, kBK8, 1, 1>
// MX on CTA pairs for prefill-sized groups: 2 x 128 gate and up rows (or
// 2 x 256 W_down rows) x 224 tokens, four stages (TMEM: 2 x 224 accumulator +
// 4 x 16 scale columns)
using GemmMxPair = Layout<2, 224, 4, 4, 1, kBK8, 1, 1, 2>;
#define GEMM1_MX_PAIR grouped_gemm_kernel<2, 224, 4, 4, kSwiGLU, 1, kBK8, 1, 1, 2>
#define GEMM2_MX_PAIR grouped_gemm_kernel<2, 224, 4, 4, kDownPair, 1, kBK8, 1, 1, 2>
#define GEMM2_MX_L grouped_gemm_kernel<2, 224, 3, 3, kDownPair, 1, kBK8, 1, 1>
#define GEMM1_MX grouped_gemm_kernel<2, 128, kMx_A, kMx_B, kSwiGLU, 1, kBK8, 1, 1>
#define GEMM2_MX grouped_gemm_kernel<2, 128, kMx_A, kMx_B, kDownPair, 1, kBK8, 1, 1>
#define GEMM1_MX_DEC grouped_gemm_kernel<2, 32, kMxD_A, kMxD_B, kSwiGLU, 2, kBK8, 1, 1>
#define GEMM2_MX_DEC grouped_gemm_kernel<2, 32, kMxD_A, kMxD_B, kDownPair, 2, kBK8, 1, 1>

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 map over [rows, K] (K contiguous), box = {bk, box_rows}; bk = 64
// uses the 128B swizzle, bk = 32 the 64B swizzle (matching smem_desc_kmajor).
bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t K, uint32_t box_rows,
              int bk) {
    return encode_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, K, rows, K * 2,
                         static_cast<uint32_t>(bk), box_rows,
                         bk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

// Maps of one GEMM: weights [groups * R, K] (a1 may be null: a copy of a0)
// and token rows [n_rows, K].
bool make_gemm_maps(GemmMaps* g, const void* a0, const void* a1, uint64_t weight_rows,
                    const void* b, uint64_t n_rows, uint64_t K) {
    return make_map(&g->a0, a0, weight_rows, K, BM, kBK) &&
           make_map(&g->a1, a1 ? a1 : a0, weight_rows, K, BM, kBK) &&
           make_map(&g->b16, b, n_rows, K, 16, kBK) && make_map(&g->b32, b, n_rows, K, 32, kBK) &&
           make_map(&g->b64, b, n_rows, K, 64, kBK) && make_map(&g->b128, b, n_rows, K, 128, kBK);
}

// FP8 (one byte per element) maps: 128-element boxes with the 128B swizzle.
bool make_map_u8(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t K, uint32_t box_rows) {
    return encode_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, ptr, K, rows, K, kBK8, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}
bool make_gemm_maps_u8(GemmMaps* g, const void* a0, const void* a1, uint64_t weight_rows,
                       const void* b, uint64_t n_rows, uint64_t K) {
    return make_map_u8(&g->a0, a0, weight_rows, K, BM) &&
           make_map_u8(&g->a1, a1 ? a1 : a0, weight_rows, K, BM) &&
           make_map_u8(&g->b16, b, n_rows, K, 16) && make_map_u8(&g->b32, b, n_rows, K, 32) &&
           make_map_u8(&g->b64, b, n_rows, K, 64) && make_map_u8(&g->b128, b, n_rows, K, 128);
}

// MX weight maps: E4M3 codes as bytes, or E2M1 codes packed two per byte
// expanded by the copy to one element per byte of shared memory (16 codes in
// the first 8 bytes of every 16), the layout kind::mxf8f6f4 reads.
bool make_map_w_mx(CUtensorMap* m, int fmt, const void* ptr, uint64_t rows, uint64_t K) {
    if (fmt == kMxE2M1)
        return encode_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, ptr, K, rows, K / 2, kBK8,
                             BM, CU_TENSOR_MAP_SWIZZLE_128B);
    return make_map_u8(m, ptr, rows, K, BM);
}
bool make_gemm_maps_mx(GemmMaps* g, int fmt, const void* a0, const void* a1,
                       uint64_t weight_rows, const void* b, uint64_t n_rows, uint64_t K) {
    return make_map_w_mx(&g->a0, fmt, a0, weight_rows, K) &&
           make_map_w_mx(&g->a1, fmt, a1 ? a1 : a0, weight_rows, K) &&
           make_map_u8(&g->b16, b, n_rows, K, 16) && make_map_u8(&g->b32, b, n_rows, K, 32) &&
           make_map_u8(&g->b64, b, n_rows, K, 64) && make_map_u8(&g->b128, b, n_rows, K, 128);
}

std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};

// Launch-time settings every grouped-GEMM launch carries.
void stamp(GemmArgs& a) { a.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed); }

std::mutex g_attr_mu;
bool g_attr_done[kMaxDevices];

cudaError_t ensure_attrs(int device) {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (device >= 0 && device < kMaxDevices && g_attr_done[device]) return cudaSuccess;
    const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaFuncSetAttribute(GEMM1_SMALL, a, Gemm1Small::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM1_LARGE, a, Gemm1Large::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM2_SMALL, a, Gemm2Small::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM2_LARGE, a, Gemm2Large::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM2_PAIR, a, Gemm2Pair::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM2_PAIR_LARGE, a, Gemm1Large::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM_FUSED, a, Gemm1Small::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM1_SMALL_F8, a, Gemm1SmallF8::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM1_LARGE_F8, a, Gemm1LargeF8::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM2_PAIR_F8, a, Gemm2PairF8::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(GEMM1_CTA_PAIR_F8, a, GemmPairLargeF8::SMEM_BYTES);

    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM1_MX, a, GemmMx::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM2_MX, a, GemmMx::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM1_MX_DEC, a, GemmMxDec::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM2_MX_DEC, a, GemmMxDec::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM1_MX_L, a, GemmMxL::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM1_MX_PAIR, a, GemmMxPair::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM2_MX_PAIR, a, GemmMxPair::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM2_MX_L, a, GemmMxL::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM1_CTA_PAIR, a, GemmPairLarge::SMEM_BYTES);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(GEMM2_CTA_PAIR, a, GemmPairLarge::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (device >= 0 && device < kMaxDevices) g_attr_done[device] = true;
    return cudaSuccess;
}

int grid_for(int groups, int n_rows, int R, int BN, int num_sms) {
    const long bound = static_cast<long>(R / BM) * ((n_rows + BN - 1) / BN + groups);
    return static_cast<int>(std::max<long>(1, std::min<long>(bound, num_sms)));
}

// Launch of a CTA-pair kernel as clusters of two CTAs, as many clusters as
// can be resident at once (one CTA per SM), at most one per tile.  The
// residency limit is queried once per device and kernel.
std::mutex g_pair_mu;
int g_pair_clusters[kMaxDevices][5];

template <class K>
int launch_pair(K kernel, int slot, int smem, long tiles, const GemmMaps& m, const GemmArgs& a,
                const DevCtx& ctx, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(std::max(2, ctx.num_sms / 2 * 2));
    int clusters = 0;
    {
        std::lock_guard<std::mutex> lk(g_pair_mu);
        int& c = g_pair_clusters[ctx.device][slot];
        if (c == 0 && cudaOccupancyMaxActiveClusters(&c, kernel, &cfg) != cudaSuccess) c = 0;
        clusters = c;
    }
    if (clusters < 1) return GBMOE_ERR_CUDA;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * std::max<long>(1, std::min<long>(clusters, tiles))));
    const FusedArgs none{0, 0, nullptr, nullptr};
    return cudaLaunchKernelEx(&cfg, kernel, m, m, a, none) == cudaSuccess ? GBMOE_OK
                                                                          : GBMOE_ERR_CUDA;
}

}  // namespace

bool encode_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
                   uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gemm_max_groups() { return MAX_GROUPS; }

uint64_t set_gemm_wait_limit_ns(uint64_t ns) {
    return g_wait_limit_ns.exchange(ns ? ns : kWaitLimitNs);
}

bool gemm_fused_eligible(int groups, int n_rows, int H) {
    return n_rows > 0 && n_rows < kLargeGateUpRows * groups && H % 256 == 0;
}

int launch_gemm_gateup(const uint16_t* x_rows, const int32_t* row_to_token, int src_rows,
                       const int32_t* offsets, int groups, int n_rows, int H, int I,
                       const uint16_t* w_gate, const uint16_t* w_up, int activation,
                       uint16_t* act, const DevCtx& ctx, cudaStream_t s) {
    if (n_rows == 0) return GBMOE_OK;
    GemmMaps m;
    // with gathered rows the token maps go unused; they are encoded over the
    // source rows only to be valid
    if (!make_gemm_maps(&m, w_gate, w_up, static_cast<uint64_t>(groups) * I, x_rows,
                        row_to_token ? src_rows : n_rows, H))
        return GBMOE_ERR_CUDA;
    if (ensure_attrs(ctx.device) != cudaSuccess) return GBMOE_ERR_CUDA;
    GemmArgs a{offsets, groups, n_rows, I, H, act, ctx.status,
               row_to_token, row_to_token ? x_rows : nullptr, src_rows, activation};
    stamp(a);
    const FusedArgs none{0, 0, nullptr, nullptr};
    if (n_rows >= kLargeGateUpRows * groups && I % 256 == 0) {
        if (!encode_map_2d(&m.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act, I, n_rows,
                           static_cast<uint64_t>(I) * 2, 32, EPI_COLS, CU_TENSOR_MAP_SWIZZLE_NONE))
            return GBMOE_ERR_CUDA;
        a.tma_out = 1;
        const long tiles = static_cast<long>(I / 256) * ((n_rows + 255) / 256 + groups);
        return launch_pair(GEMM1_CTA_PAIR, 0, GemmPairLarge::SMEM_BYTES, tiles, m, a, ctx, s);
    } else if (n_rows >= kLargeGateUpRows * groups) {
        const int grid = grid_for(groups, n_rows, I, 256, ctx.num_sms);
        GEMM1_LARGE<<<grid, NUM_THREADS, Gemm1Large::SMEM_BYTES, s>>>(m, m, a, none);
    } else {
        const int grid = grid_for(groups, n_rows, I, 128, ctx.num_sms);
        GEMM1_SMALL<<<grid, NUM_THREADS, Gemm1Small::SMEM_BYTES, s>>>(m, m, a, none);
    }
    return cudaGetLastError() == cudaSuccess ? GBMOE_OK : GBMOE_ERR_CUDA;
}

int launch_gemm_down(const uint16_t* act, const int32_t* offsets, int groups, int n_rows, int H,
                     int I, const uint16_t* w_down, float* y, const DevCtx& ctx,
                     cudaStream_t s) {
    if (n_rows == 0) return GBMOE_OK;
    GemmMaps m;
    if (!make_gemm_maps(&m, w_down, nullptr, static_cast<uint64_t>(groups) * H, act, n_rows, I))
        return GBMOE_ERR_CUDA;
    if (ensure_attrs(ctx.device) != cudaSuccess) return GBMOE_ERR_CUDA;
    GemmArgs a{offsets, groups, n_rows, H, I, y, ctx.status, nullptr, nullptr, 0, 0};
    stamp(a);
    const FusedArgs none{0, 0, nullptr, nullptr};
    if (H % 512 == 0 && n_rows >= kLargeGateUpRows * groups) {
        if (!encode_map_2d(&m.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, y, H, n_rows,
                           static_cast<uint64_t>(H) * 4, 32, EPI_COLS, CU_TENSOR_MAP_SWIZZLE_NONE))
            return GBMOE_ERR_CUDA;
        a.tma_out = 1;
        const long tiles = static_cast<long>(H / 512) * ((n_rows + 255) / 256 + groups);
        return launch_pair(GEMM2_CTA_PAIR, 1, GemmPairLarge::SMEM_BYTES, tiles, m, a, ctx, s);
    } else if (H % 256 == 0 && n_rows >= kLargeGateUpRows * groups) {
        const int grid = grid_for(groups, n_rows, H / 2, 256, ctx.num_sms);
        GEMM2_PAIR_LARGE<<<grid, NUM_THREADS, Gemm1Large::SMEM_BYTES, s>>>(m, m, a, none);
    } else if (H % 256 == 0) {
        const int grid = grid_for(groups, n_rows, H / 2, 128, ctx.num_sms);
        GEMM2_PAIR<<<grid, NUM_THREADS, Gemm2Pair::SMEM_BYTES, s>>>(m, m, a, none);
    } else if (n_rows >= 128L * groups) {
        const int grid = grid_for(groups, n_rows, H, 256, ctx.num_sms);
        GEMM2_LARGE<<<grid, NUM_THREADS, Gemm2Large::SMEM_BYTES, s>>>(m, m, a, none);
    } else {
        const int grid = grid_for(groups, n_rows, H, 128, ctx.num_sms);
        GEMM2_SMALL<<<grid, NUM_THREADS, Gemm2Small::SMEM_BYTES, s>>>(m, m, a, none);
    }
    return cudaGetLastError() == cudaSuccess ? GBMOE_OK : GBMOE_ERR_CUDA;
}

int launch_gemm_mlp_fused(const uint16_t* x_rows, const int32_t* row_to_token, int src_rows,
                          const int32_t* offsets, int groups, int n_rows, int H, int I,
                          const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                          int activation, uint16_t* act, float* y, int* ready,
                          const DevCtx& ctx, cudaStream_t s) {
    if (n_rows == 0) return GBMOE_OK;
    GemmMaps m1, m2;
    if (!make_gemm_maps(&m1, w_gate, w_up, static_cast<uint64_t>(groups) * I, x_rows,
                        row_to_token ? src_rows : n_rows, H) ||
        !make_gemm_maps(&m2, w_down, nullptr, static_cast<uint64_t>(groups) * H, act, n_rows, I))
        return GBMOE_ERR_CUDA;
    if (ensure_attrs(ctx.device) != cudaSuccess) return GBMOE_ERR_CUDA;
    if (cudaMemsetAsync(ready, 0, sizeof(int) * groups, s) != cudaSuccess) return GBMOE_ERR_CUDA;
    GemmArgs a{offsets, groups, n_rows, I, H, act, ctx.status,
               row_to_token, row_to_token ? x_rows : nullptr, src_rows, activation};
    stamp(a);
    const FusedArgs f{H, I, y, ready};
    // every CTA must be resident (down tiles wait on gate/up tiles of other
    // CTAs): a cooperative launch of at most one CTA per SM
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctx.num_sms);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = Gemm1Small::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, GEMM_FUSED, m1, m2, a, f);
    return e == cudaSuccess ? GBMOE_OK : GBMOE_ERR_CUDA;
}

int launch_gemm_gateup_fp8(const uint8_t* xq, const float* sx, const int32_t* row_to_token,
                           int src_rows, const int32_t* offsets, int groups, int n_rows, int H,
                           int I, const uint8_t* wg, const float* sg, const uint8_t* wu,
                           const float* su, int activation, uint16_t* act, const DevCtx& ctx,
                           cudaStream_t s) {
    if (n_rows == 0) return GBMOE_OK;
    GemmMaps m;
    if (!make_gemm_maps_u8(&m, wg, wu, static_cast<uint64_t>(groups) * I, xq,
                           row_to_token ? src_rows : n_rows, H))
        return GBMOE_ERR_CUDA;
    if (ensure_attrs(ctx.device) != cudaSuccess) return GBMOE_ERR_CUDA;
    GemmArgs a{offsets, groups, n_rows, I, H, act, ctx.status,
               row_to_token, row_to_token ? xq : nullptr, src_rows, activation};
    stamp(a);
    a.tok_scale = sx;
    a.w_scale0 = sg;
    a.w_scale1 = su;
    const FusedArgs none{0, 0, nullptr, nullptr};
    if (n_rows >= kLargeGateUpRows * groups && I % 256 == 0) {
        if (!encode_map_2d(&m.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act, I, n_rows,
                           static_cast<uint64_t>(I) * 2, 32, EPI_COLS, CU_TENSOR_MAP_SWIZZLE_NONE))
            return GBMOE_ERR_CUDA;
        a.tma_out = 1;
        const long tiles = static_cast<long>(I / 256) * ((n_rows + 255) / 256 + groups);
        return launch_pair(GEMM1_CTA_PAIR_F8, 2, GemmPairLargeF8::SMEM_BYTES, tiles, m, a, ctx, s);
    } else if (n_rows >= kLargeGateUpRows * groups) {
        const int grid = grid_for(groups, n_rows, I, 256, ctx.num_sms);
        GEMM1_LARGE_F8<<<grid, NUM_THREADS, Gemm1LargeF8::SMEM_BYTES, s>>>(m, m, a, none);
    } else {
        const int grid = grid_for(groups, n_rows, I, 128, ctx.num_sms);
        GEMM1_SMALL_F8<<<grid, NUM_THREADS, Gemm1SmallF8::SMEM_BYTES, s>>>(m, m, a, none);
    }
    return cudaGetLastError() == cudaSuccess ? GBMOE_OK : GBMOE_ERR_CUDA;
}

int launch_gemm_down_fp8(const uint8_t* aq, const float* sa, const int32_t* offsets, int groups,
                         int n_rows, int H, int I, const uint8_t* wd, const float* sd, float* y,
                         const DevCtx& ctx, cudaStream_t s) {
    if (n_rows == 0) return GBMOE_OK;
    if (H % 256) return GBMOE_ERR_UNSUPPORTED;
    GemmMaps m;
    if (!make_gemm_maps_u8(&m, wd, nullptr, static_cast<uint64_t>(groups) * H, aq, n_rows, I))
        return GBMOE_ERR_CUDA;
    if (ensure_attrs(ctx.device) != cudaSuccess) return GBMOE_ERR_CUDA;
    GemmArgs a{offsets, groups, n_rows, H, I, y, ctx.status, nullptr, nullptr, 0, 0};
    stamp(a);
    a.tok_scale = sa;
    a.w_scale0 = sd;
    const FusedArgs none{0, 0, nullptr, nullptr};
    // (256-token paired tiles, on one SM or on CTA pairs, both faster for
    // bf16, were measured slower here: 1.37 and 1.30 vs 1.22 ms at prefill;
    // these 128-token tiles on CTA pairs gained nothing)
    if (!encode_map_2d(&m.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, y, H, n_rows,
                       static_cast<uint64_t>(H) * 4, 32, EPI_COLS, CU_TENSOR_MAP_SWIZZLE_NONE))
        return GBMOE_ERR_CUDA;
    a.tma_out = 1;
    const int grid = grid_for(groups, n_rows, H / 2, 128, ctx.num_sms);
    GEMM2_PAIR_F8<<<grid, NUM_THREADS, Gemm2PairF8::SMEM_BYTES, s>>>(m, m, a, none);
    return cudaGetLastError() == cudaSuccess ? GBMOE_OK : GBMOE_ERR_CUDA;
}

int launch_gemm_gateup_mx(const uint8_t* xq, const uint8_t* xs, const int32_t* row_to_token,
                          int src_rows, const int32_t* offsets, int groups, int n_rows, int H,
                          int I, int w_fmt, const uint8_t* wg, const uint8_t* sg,
                          const uint8_t* wu, const uint8_t* su, int activation, uint8_t* aq,
                          uint8_t* as, const DevCtx& ctx, cudaStream_t s) {
    if (n_rows == 0) return GBMOE_OK;
    GemmMaps m;
    if (!make_gemm_maps_mx(&m, w_fmt, wg, wu, static_cast<uint64_t>(groups) * I, xq,
                           row_to_token ? src_rows : n_rows, H))
        return GBMOE_ERR_CUDA;
    if (ensure_attrs(ctx.device) != cudaSuccess) return GBMOE_ERR_CUDA;
    GemmArgs a{offsets, groups, n_rows, I, H, aq, ctx.status,
               row_to_token, row_to_token ? xq : nullptr, src_rows, activation};
    stamp(a);
    a.tok_sf = xs;
    a.w_sf0 = sg;
    a.w_sf1 = su;
    a.out_sf = as;
    a.a_fmt = w_fmt == kMxE2M1 ? 5u : 0u;
    const FusedArgs none{0, 0, nullptr, nullptr};
    if (n_rows <= kMxDecodeRows * groups) {
        const int grid = grid_for(groups, n_rows, I, 32, ctx.num_sms);
        GEMM1_MX_DEC<<<grid, NUM_THREADS, GemmMxDec::SMEM_BYTES, s>>>(m, m, a, none);
    } else if (n_rows >= kLargeGateUpRows * groups && I % 256 == 0) {
        // the weight scale chunks as 512-byte rows for the pair's TMA copies
        const uint64_t chunks = static_cast<uint64_t>(groups) * (I / 128) * (H / 128);
        if (!encode_map_2d(&m.s0, CU_TENSOR_MAP_DATA_TYPE_UINT32, sg, 128, chunks, 512, 128, 1,
                           CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_map_2d(&m.s1, CU_TENSOR_MAP_DATA_TYPE_UINT32, su, 128, chunks, 512, 128, 1,
                           CU_TENSOR_MAP_SWIZZLE_NONE))
            return GBMOE_ERR_CUDA;
        const long tiles = static_cast<long>(I / 256) * ((n_rows + 223) / 224 + groups);
        return launch_pair(GEMM1_MX_PAIR, 3, GemmMxPair::SMEM_BYTES, tiles, m, a, ctx, s);
    } else if (n_rows >= kLargeGateUpRows * groups) {
        const int grid = grid_for(groups, n_rows, I, 224, ctx.num_sms);
        GEMM1_MX_L<<<grid, NUM_THREADS, GemmMxL::SMEM_BYTES, s>>>(m, m, a, none);
    } else {
        const int grid = grid_for(groups, n_rows, I, 128, ctx.num_sms);
        GEMM1_MX<<<grid, NUM_THREADS, GemmMx::SMEM_BYTES, s>>>(m, m, a, none);
    }
    return cudaGetLastError() == cudaSuccess ? GBMOE_OK : GBMOE_ERR_CUDA;
}

int launch_gemm_down_mx(const uint8_t* aq, const uint8_t* as, const int32_t* offsets, int groups,
                        int n_rows, int H, int I, int w_fmt, const uint8_t* wd,
                        const uint8_t* sd, float* y, const DevCtx& ctx, cudaStream_t s) {
    if (n_rows == 0) return GBMOE_OK;
    if (H % 256) return GBMOE_ERR_UNSUPPORTED;
    GemmMaps m;
    if (!make_gemm_maps_mx(&m, w_fmt, wd, nullptr, static_cast<uint64_t>(groups) * H, aq, n_rows,
                           I))
        return GBMOE_ERR_CUDA;
    if (ensure_attrs(ctx.device) != cudaSuccess) return GBMOE_ERR_CUDA;
    GemmArgs a{offsets, groups, n_rows, H, I, y, ctx.status, nullptr, nullptr, 0, 0};
    stamp(a);
    a.tok_sf = as;
    a.w_sf0 = sd;
    a.a_fmt = w_fmt == kMxE2M1 ? 5u : 0u;
    const FusedArgs none{0, 0, nullptr, nullptr};
    if (n_rows <= kMxDecodeRows * groups) {
        const int grid = grid_for(groups, n_rows, H / 2, 32, ctx.num_sms);
        GEMM2_MX_DEC<<<grid, NUM_THREADS, GemmMxDec::SMEM_BYTES, s>>>(m, m, a, none);
    } else if (n_rows >= kLargeGateUpRows * groups && H % 512 == 0) {
        const uint64_t chunks = static_cast<uint64_t>(groups) * (H / 128) * (I / 128);
        if (!encode_map_2d(&m.s0, CU_TENSOR_MAP_DATA_TYPE_UINT32, sd, 128, chunks, 512, 128, 1,
                           CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_map_2d(&m.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, y, H, n_rows,
                           static_cast<uint64_t>(H) * 4, 32, EPI_COLS, CU_TENSOR_MAP_SWIZZLE_NONE))
            return GBMOE_ERR_CUDA;
        a.tma_out = 1;
        const long tiles = static_cast<long>(H / 512) * ((n_rows + 223) / 224 + groups);
        return launch_pair(GEMM2_MX_PAIR, 4, GemmMxPair::SMEM_BYTES, tiles, m, a, ctx, s);
    } else if (n_rows >= kLargeGateUpRows * groups) {
        const int grid = grid_for(groups, n_rows, H / 2, 224, ctx.num_sms);
        GEMM2_MX_L<<<grid, NUM_THREADS, GemmMxL::SMEM_BYTES, s>>>(m, m, a, none);
    } else {
        const int grid = grid_for(groups, n_rows, H / 2, 128, ctx.num_sms);
        GEMM2_MX<<<grid, NUM_THREADS, GemmMx::SMEM_BYTES, s>>>(m, m, a, none);
    }
    return cudaGetLastError() == cudaSuccess ? GBMOE_OK : GBMOE_ERR_CUDA;
}

}  // namespace gbmoe
