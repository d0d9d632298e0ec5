// Host-side launchers shared between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gbmoe.h"

namespace gbmoe {

// Per-device host state (contexts, kernel attributes, scratch addresses) is
// kept for device ordinals below this bound.
constexpr int kMaxDevices = 64;
constexpr int kMaxTopK = 32;  // largest top_k a route configuration may ask for

struct DevCtx {
    int device;
    int num_sms;
    int* status;  // device address of this device's status word
};

// Lazily created per-device context for the current device (nullptr on failure).
const DevCtx* device_ctx();

// 2-D TMA tensor map over a row-major [rows, inner] array whose rows are
// row_bytes apart; box {box_inner, box_rows}.  False if the driver entry point
// is unavailable or the encode rejects the arguments (gemm.cu).
bool encode_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
                   uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle);

// --- routing (route.cu) ---
struct RouteArgs {
    gbmoe_route_cfg cfg;
    int T, H;
    const uint16_t* x;
    const float* w_router;
    float* logits;
    const float* router_bias;
    const float* corr_bias;
    const int32_t* input_ids;
    const int32_t* tid2eid;
    int64_t tid2eid_rows;
    const int32_t* log2phy;
    const int32_t* replica_cnt;
    int R_max;
    int32_t* ids_log;
    int32_t* ids_phys;
    float* weights;
    int32_t* counts;  // may be null; zeroed by the caller beforehand
    // the logits are scratch (moe_forward): with hash routing and an
    // elementwise score only the hashed experts' logits are computed
    int hash_logits_only;
};
cudaError_t launch_route(const RouteArgs& a, const DevCtx& ctx, cudaStream_t s);
cudaError_t launch_expert_counts(const int32_t* ids, int64_t n, int E_phys, int32_t* counts,
                                 const DevCtx& ctx, cudaStream_t s);

// --- permutation (permute.cu) ---
constexpr int kPermChunk = 256;  // flat (token, slot) pairs per scatter worker
// Argument checks shared by moe_permute and moe_permute_static (api.cu):
// GBMOE_OK or the status the entry point returns; *N receives T * k.
int check_permute_args(const int32_t* ids_phys, int T, int k, int E_phys, const uint16_t* x,
                       int H, const int32_t* counts, const int32_t* offsets,
                       const int32_t* row_to_token, const int32_t* flat_to_row,
                       const uint16_t* x_perm, int64_t* N);
size_t permute_ws_bytes(int64_t N, int E_phys);
cudaError_t launch_permute(const int32_t* ids_phys, int64_t N, int k, int E_phys,
                           const uint16_t* x, int H, int32_t* counts, int32_t* offsets,
                           int32_t* row_to_token, int32_t* flat_to_row, uint16_t* x_perm,
                           void* ws, const DevCtx& ctx, cudaStream_t s);

// --- grouped GEMMs (gemm.cu) ---
// Returns GBMOE_OK or an error status (tensor-map encode or launch failure).
// x_rows: the token operand [n_rows, H]; or, with row_to_token, the source
// rows [src_rows, H] that row r of the operand is gathered from.
int launch_gemm_gateup(const uint16_t* x_rows, const int32_t* row_to_token, int src_rows,
                       const int32_t* offsets, int groups, int n_rows, int H, int I,
                       const uint16_t* w_gate, const uint16_t* w_up, int activation,
                       uint16_t* act, const DevCtx& ctx, cudaStream_t s);
int launch_gemm_down(const uint16_t* act, const int32_t* offsets, int groups, int n_rows, int H,
                     int I, const uint16_t* w_down, float* y, const DevCtx& ctx,
                     cudaStream_t s);
int gemm_max_groups();
// Limit of the bounded pipeline waits of grouped-GEMM launches made from now
// on (0: the default, 4 s); returns the previous limit.
uint64_t set_gemm_wait_limit_ns(uint64_t ns);
// Whether moe_forward runs both GEMMs in one fused cooperative launch (small
// groups: decode-like batches).
bool gemm_fused_eligible(int groups, int n_rows, int H);
// Gate/up + SwiGLU and down in one launch; `ready` is [groups] int scratch.
int launch_gemm_mlp_fused(const uint16_t* x_rows, const int32_t* row_to_token, int src_rows,
                          const int32_t* offsets, int groups, int n_rows, int H, int I,
                          const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                          int activation, uint16_t* act, float* y, int* ready,
                          const DevCtx& ctx, cudaStream_t s);

// FP8 E4M3 grouped GEMMs (two launches; one fp32 scale per token / routed
// row and per weight row): act = bf16(f((xq.wg^T) sx sg, (xq.wu^T) sx su)),
// y = (aq.wd^T) sa sd.  H % 256 == 0 for the down GEMM.
int launch_gemm_gateup_fp8(const uint8_t* xq, const float* sx, const int32_t* row_to_token,
                           int src_rows, const int32_t* offsets, int groups, int n_rows, int H,
                           int I, const uint8_t* wg, const float* sg, const uint8_t* wu,
                           const float* su, int activation, uint16_t* act, const DevCtx& ctx,
                           cudaStream_t s);
int launch_gemm_down_fp8(const uint8_t* aq, const float* sa, const int32_t* offsets, int groups,
                         int n_rows, int H, int I, const uint8_t* wd, const float* sd, float* y,
                         const DevCtx& ctx, cudaStream_t s);

// MX block-scaled grouped GEMMs (kind::mxf8f6f4 block_scale): tokens /
// activations as MX E4M3 (codes [rows, K], scale bytes [rows, K/32]),
// weights as MX E4M3 or E2M1 (w_fmt: kMxE4M3 / kMxE2M1; E2M1 codes packed two
// per byte).  The gate/up GEMM writes the activation already quantized to MX
// E4M3 (act codes [n_rows, I] + scales [n_rows, I/32]); the down GEMM writes
// y fp32.  H % 256 == 0, I % 128 == 0.
int launch_gemm_gateup_mx(const uint8_t* xq, const uint8_t* xs, const int32_t* row_to_token,
                          int src_rows, const int32_t* offsets, int groups, int n_rows, int H,
                          int I, int w_fmt, const uint8_t* wg, const uint8_t* sg,
                          const uint8_t* wu, const uint8_t* su, int activation, uint8_t* aq,
                          uint8_t* as, const DevCtx& ctx, cudaStream_t s);
int launch_gemm_down_mx(const uint8_t* aq, const uint8_t* as, const int32_t* offsets, int groups,
                        int n_rows, int H, int I, int w_fmt, const uint8_t* wd,
                        const uint8_t* sd, float* y, const DevCtx& ctx, cudaStream_t s);

// --- FP8 row quantization and MX block quantization (quant.cu) ---
cudaError_t launch_quantize_rows(const uint16_t* x, int64_t n, int K, uint8_t* q, float* s,
                                 const DevCtx& ctx, cudaStream_t st);
// rows [n, K] bf16 (K % 32 == 0) -> codes (E4M3 [n, K] or E2M1 [n, K/2]) and
// UE8M0 scale bytes [n, K/32]
cudaError_t launch_mx_quantize(const uint16_t* x, int64_t n, int K, int fmt, uint8_t* q,
                               uint8_t* sc, const DevCtx& ctx, cudaStream_t st);

// MX weight scales row-major [rows, K/32] -> the GEMMs' tiled layout
// (rows % 128 == 0, K % 128 == 0)
cudaError_t launch_mx_tile_scales(const uint8_t* sf_rows, int64_t rows, int K, uint8_t* tiled,
                                  const DevCtx& ctx, cudaStream_t st);

// --- latent-MoE tail (tail.cu) ---
size_t latent_tail_ws_bytes(int T, int L, int Hm);
int launch_latent_tail(const uint16_t* latent, int T, int L, const uint16_t* norm_w, float eps,
                       const uint16_t* up_proj, int Hm, const uint16_t* shared, uint16_t* out,
                       void* ws, const DevCtx& ctx, cudaStream_t s);

// --- combine (combine.cu) ---
cudaError_t launch_combine(const float* y, const int32_t* flat_to_row, const float* weights,
                           const float* shared_y, int T, int k, int H, uint16_t* out,
                           const DevCtx& ctx, cudaStream_t s);

}  // namespace gbmoe
