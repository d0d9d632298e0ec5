// C ABI of libgbmoe.so (declared in include/gbmoe.h): argument validation,
// the per-device context, workspace layout and the layer orchestration.
// Follows the routed-MoE forward of the vLLM-Ascend "Kimi K3 MoE Forward
// Insight" page ("Forward Skeleton"; "Stage 4: Dispatch, MLP, Combine" steps
// 1-9), specialised to one GPU: dispatch is a local permutation.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "gbmoe.h"
#include "internal.h"

namespace gbmoe {

// One status word per device: first device-side error since the last check.
__device__ int g_status_word = 0;

namespace {

std::mutex g_ctx_mu;
DevCtx g_ctx[kMaxDevices];
bool g_ctx_ok[kMaxDevices];

constexpr int kMaxE = 1024;
constexpr int kMaxGroups = 32;

bool valid_activation(int a) { return a >= GBMOE_ACT_SWIGLU && a <= GBMOE_ACT_GEGLU_TANH; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
// E2M1 weights are read by 32-byte-aligned tensor copies
inline bool mx_weights_aligned(int fmt, const void* p) {
    return (reinterpret_cast<uintptr_t>(p) & (fmt == GBMOE_MX_E2M1 ? 31u : 15u)) == 0;
}
inline size_t align256(size_t b) { return (b + 255) / 256 * 256; }

int status_from(cudaError_t e) { return e == cudaSuccess ? GBMOE_OK : GBMOE_ERR_CUDA; }

int check_cfg(const gbmoe_route_cfg* c) {
    if (!c) return GBMOE_ERR_INVALID_ARG;
    if (c->E_log < 1 || c->E_log > kMaxE) return GBMOE_ERR_INVALID_ARG;
    if (c->E_phys < c->E_log || c->E_phys > kMaxE) return GBMOE_ERR_INVALID_ARG;
    if (c->top_k < 1 || c->top_k > c->E_log || c->top_k > kMaxTopK) return GBMOE_ERR_INVALID_ARG;
    if (c->n_group < 1 || c->n_group > kMaxGroups || c->E_log % c->n_group) return GBMOE_ERR_INVALID_ARG;
    if (c->topk_group < 1 || c->topk_group > c->n_group) return GBMOE_ERR_INVALID_ARG;
    if (c->n_group > 1 && c->topk_group * (c->E_log / c->n_group) < c->top_k)
        return GBMOE_ERR_INVALID_ARG;
    if (c->scoring < GBMOE_SCORE_SOFTMAX || c->scoring > GBMOE_SCORE_SQRTSOFTPLUS)
        return GBMOE_ERR_INVALID_ARG;
    if (c->group_score != GBMOE_GROUP_MAX && c->group_score != GBMOE_GROUP_TOP2SUM)
        return GBMOE_ERR_INVALID_ARG;
    if (c->use_hash && c->n_group != 1) return GBMOE_ERR_INVALID_ARG;
    if (!(c->routed_scaling == c->routed_scaling)) return GBMOE_ERR_INVALID_ARG;
    return GBMOE_OK;
}

struct WsCursor {
    char* base;
    size_t off;
    template <typename T>
    T* take(size_t count) {
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += align256(count * sizeof(T));
        return p;
    }
};

// Workspace of moe_forward for T tokens (nullptr base: sizing only).
struct FwdWs {
    float* logits;
    int32_t *ids_log, *ids_phys, *counts, *offsets, *row_to_token, *flat_to_row, *ready;
    float* weights;
    void* perm;
    uint16_t *act, *act_s;
    float *y, *ys;
    uint8_t *xq, *aq;  // FP8 / MX layers: hidden-state and activation codes
    float *sx, *sa;    // and their per-row scales (FP8)
    uint8_t *xs, *as;  // or block-scale bytes (MX)
    size_t bytes;
};

FwdWs layout_fwd(const gbmoe_layer* L, int T, void* ws) {
    const gbmoe_route_cfg& c = L->route;
    const size_t N = static_cast<size_t>(T) * c.top_k;
    WsCursor w{static_cast<char*>(ws), 0};
    FwdWs f;
    f.logits = w.take<float>(static_cast<size_t>(T) * c.E_log);
    f.ids_log = w.take<int32_t>(N);
    f.ids_phys = w.take<int32_t>(N);
    f.weights = w.take<float>(N);
    f.counts = w.take<int32_t>(c.E_phys);
    f.offsets = w.take<int32_t>(c.E_phys + 1);
    f.ready = w.take<int32_t>(c.E_phys);
    f.row_to_token = w.take<int32_t>(N);
    f.flat_to_row = w.take<int32_t>(N);
    f.perm = w.take<char>(permute_ws_bytes(static_cast<int64_t>(N), c.E_phys));
    f.act = w.take<uint16_t>(N * L->I);
    f.y = w.take<float>(N * L->H);
    f.act_s = w.take<uint16_t>(static_cast<size_t>(T) * L->I_shared);
    f.ys = w.take<float>(L->I_shared ? static_cast<size_t>(T) * L->H : 0);
    const bool fp8 = L->w_gate_q != nullptr;
    const bool mx = !fp8 && L->w_gate_mx != nullptr;
    f.xq = w.take<uint8_t>(fp8 || mx ? static_cast<size_t>(T) * L->H : 0);
    f.sx = w.take<float>(fp8 ? static_cast<size_t>(T) : 0);
    f.aq = w.take<uint8_t>(fp8 || mx ? N * L->I : 0);
    f.sa = w.take<float>(fp8 ? N : 0);
    f.xs = w.take<uint8_t>(mx ? static_cast<size_t>(T) * (L->H / 32) : 0);
    f.as = w.take<uint8_t>(mx ? N * (L->I / 32) : 0);
    f.bytes = w.off;
    return f;
}

int check_layer(const gbmoe_layer* L) {
    if (!L) return GBMOE_ERR_INVALID_ARG;
    int st = check_cfg(&L->route);
    if (st) return st;
    const gbmoe_route_cfg& c = L->route;
    if (L->H <= 0 || L->I <= 0 || L->I_shared < 0) return GBMOE_ERR_INVALID_ARG;
    if (L->H % 128 || L->I % 128 || L->I_shared % 128) return GBMOE_ERR_UNSUPPORTED;
    if (!L->w_router) return GBMOE_ERR_INVALID_ARG;
    if (L->w_gate_q) {  // FP8 routed experts
        if (!L->w_up_q || !L->w_down_q || !L->s_gate || !L->s_up || !L->s_down)
            return GBMOE_ERR_INVALID_ARG;
        if (!aligned16(L->w_gate_q) || !aligned16(L->w_up_q) || !aligned16(L->w_down_q))
            return GBMOE_ERR_INVALID_ARG;
        if (L->H % 256) return GBMOE_ERR_UNSUPPORTED;
    } else if (L->w_gate_mx) {  // MX block-scaled routed experts
        if (!L->w_up_mx || !L->w_down_mx || !L->sf_gate || !L->sf_up || !L->sf_down)
            return GBMOE_ERR_INVALID_ARG;
        if (L->mx_format != GBMOE_MX_E4M3 && L->mx_format != GBMOE_MX_E2M1)
            return GBMOE_ERR_UNSUPPORTED;
        if (!mx_weights_aligned(L->mx_format, L->w_gate_mx) ||
            !mx_weights_aligned(L->mx_format, L->w_up_mx) ||
            !mx_weights_aligned(L->mx_format, L->w_down_mx) || !aligned16(L->sf_gate) ||
            !aligned16(L->sf_up) || !aligned16(L->sf_down))
            return GBMOE_ERR_INVALID_ARG;
        if (L->H % 256) return GBMOE_ERR_UNSUPPORTED;
    } else {
        if (!L->w_gate || !L->w_up || !L->w_down) return GBMOE_ERR_INVALID_ARG;
        if (!aligned16(L->w_gate) || !aligned16(L->w_up) || !aligned16(L->w_down))
            return GBMOE_ERR_INVALID_ARG;
    }
    if (c.use_hash && (!L->tid2eid || L->tid2eid_rows <= 0 || L->corr_bias))
        return GBMOE_ERR_INVALID_ARG;
    if (L->log2phy && (!L->replica_cnt || L->R_max < 1)) return GBMOE_ERR_INVALID_ARG;
    if (!L->log2phy && c.E_phys != c.E_log) return GBMOE_ERR_INVALID_ARG;
    if (L->I_shared && (!L->w_gate_shared || !L->w_up_shared || !L->w_down_shared))
        return GBMOE_ERR_INVALID_ARG;
    if (!valid_activation(L->activation)) return GBMOE_ERR_UNSUPPORTED;
    return GBMOE_OK;
}

}  // namespace

int check_permute_args(const int32_t* ids_phys, int T, int k, int E_phys, const uint16_t* x,
                       int H, const int32_t* counts, const int32_t* offsets,
                       const int32_t* row_to_token, const int32_t* flat_to_row,
                       const uint16_t* x_perm, int64_t* N) {
    if (T < 0 || k < 1 || E_phys < 1 || E_phys > kMaxE) return GBMOE_ERR_INVALID_ARG;
    if (!counts || !offsets) return GBMOE_ERR_INVALID_ARG;
    if (T > 0 && (!ids_phys || !row_to_token || !flat_to_row)) return GBMOE_ERR_INVALID_ARG;
    if (x_perm && (!x || H <= 0 || H % 8 || !aligned16(x) || !aligned16(x_perm)))
        return GBMOE_ERR_INVALID_ARG;
    *N = static_cast<int64_t>(T) * k;
    if (*N > INT32_MAX) return GBMOE_ERR_UNSUPPORTED;
    return GBMOE_OK;
}

const DevCtx* device_ctx() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_ctx_mu);
    if (!g_ctx_ok[dev]) {
        DevCtx c;
        c.device = dev;
        if (cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        c.status = static_cast<int*>(p);
        g_ctx[dev] = c;
        g_ctx_ok[dev] = true;
    }
    return &g_ctx[dev];
}

}  // namespace gbmoe

using namespace gbmoe;

extern "C" {

const char* gbmoe_status_string(int status) {
    switch (status) {
        case GBMOE_OK: return "ok";
        case GBMOE_ERR_INVALID_ARG: return "invalid argument";
        case GBMOE_ERR_UNSUPPORTED: return "unsupported shape or option";
        case GBMOE_ERR_WORKSPACE: return "workspace missing or too small";
        case GBMOE_ERR_CUDA: return "CUDA runtime error";
        case GBMOE_ERR_DEVICE: return "device-side check failed (bad id or table entry)";
        case GBMOE_ERR_TIMEOUT: return "GEMM pipeline wait timed out";
        default: return "unknown status";
    }
}

int gbmoe_validate_route_cfg(const gbmoe_route_cfg* cfg) { return check_cfg(cfg); }

uint64_t gbmoe_set_wait_limit_ns(uint64_t ns) { return set_gemm_wait_limit_ns(ns); }

int gbmoe_validate_log2phy(const int32_t* log2phy_host, const int32_t* replica_cnt_host,
                           int E_log, int R_max, int E_phys) {
    if (!log2phy_host || !replica_cnt_host || E_log < 1 || R_max < 1 || E_phys < E_log)
        return GBMOE_ERR_INVALID_ARG;
    std::vector<int> owner(E_phys, -1);
    for (int e = 0; e < E_log; ++e) {
        const int n = replica_cnt_host[e];
        if (n < 1 || n > R_max) return GBMOE_ERR_INVALID_ARG;
        for (int r = 0; r < n; ++r) {
            const int p = log2phy_host[static_cast<size_t>(e) * R_max + r];
            if (p < 0 || p >= E_phys) return GBMOE_ERR_INVALID_ARG;
            if (owner[p] != -1 && owner[p] != e) return GBMOE_ERR_INVALID_ARG;
            if (owner[p] == e) return GBMOE_ERR_INVALID_ARG;  // same slot twice
            owner[p] = e;
        }
    }
    return GBMOE_OK;
}

int gbmoe_check_device_status(gbmoe_stream_t stream, int* status) {
    if (!status) return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GBMOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, ctx->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GBMOE_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(ctx->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
        return GBMOE_ERR_CUDA;
    *status = v;
    return GBMOE_OK;
}

int moe_route(const gbmoe_route_cfg* cfg, const uint16_t* x, int T, int H,
              const float* w_router, float* logits, const float* router_bias,
              const float* corr_bias, const int32_t* input_ids, const int32_t* tid2eid,
              int64_t tid2eid_rows, const int32_t* log2phy, const int32_t* replica_cnt,
              int R_max, int32_t* ids_log, int32_t* ids_phys, float* weights, int32_t* counts,
              gbmoe_stream_t stream) {
    int st = check_cfg(cfg);
    if (st) return st;
    if (T < 0) return GBMOE_ERR_INVALID_ARG;
    if (!logits || !ids_log || !ids_phys || !weights) return GBMOE_ERR_INVALID_ARG;
    if (w_router && (!x || H <= 0)) return GBMOE_ERR_INVALID_ARG;
    if (cfg->use_hash && (!input_ids || !tid2eid || tid2eid_rows <= 0 || corr_bias))
        return GBMOE_ERR_INVALID_ARG;
    if (log2phy && (!replica_cnt || R_max < 1)) return GBMOE_ERR_INVALID_ARG;
    if (!log2phy && cfg->E_phys != cfg->E_log) return GBMOE_ERR_INVALID_ARG;
    if (T == 0) return GBMOE_OK;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (counts) {
        st = status_from(cudaMemsetAsync(counts, 0, sizeof(int32_t) * cfg->E_phys, s));
        if (st) return st;
    }
    RouteArgs a{*cfg, T, H, x, w_router, logits, router_bias, corr_bias, input_ids, tid2eid,
                tid2eid_rows, log2phy, replica_cnt, R_max, ids_log, ids_phys, weights, counts};
    return status_from(launch_route(a, *ctx, s));
}

int moe_expert_counts(const int32_t* ids_phys, int T, int k, int E_phys, int32_t* counts,
                      int accumulate, gbmoe_stream_t stream) {
    if (T < 0 || k < 1 || E_phys < 1 || !counts || (T > 0 && !ids_phys))
        return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!accumulate) {
        int st = status_from(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E_phys, s));
        if (st) return st;
    }
    return status_from(
        launch_expert_counts(ids_phys, static_cast<int64_t>(T) * k, E_phys, counts, *ctx, s));
}

size_t gbmoe_permute_workspace_size(int T, int k, int E_phys) {
    if (T < 0 || k < 1 || E_phys < 1) return 0;
    return permute_ws_bytes(static_cast<int64_t>(T) * k, E_phys);
}

int moe_permute(const int32_t* ids_phys, int T, int k, int E_phys, const uint16_t* x, int H,
                int32_t* counts, int32_t* offsets, int32_t* row_to_token, int32_t* flat_to_row,
                uint16_t* x_perm, void* ws, size_t ws_bytes, gbmoe_stream_t stream) {
    int64_t N = 0;
    const int st = check_permute_args(ids_phys, T, k, E_phys, x, H, counts, offsets,
                                      row_to_token, flat_to_row, x_perm, &N);
    if (st) return st;
    if (N > 0 && (!ws || ws_bytes < permute_ws_bytes(N, E_phys))) return GBMOE_ERR_WORKSPACE;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return status_from(launch_permute(ids_phys, N, k, E_phys, x, H, counts, offsets, row_to_token,
                                      flat_to_row, x_perm, ws, *ctx,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

int moe_gemm_gateup_act(const uint16_t* x_perm, const int32_t* offsets, int E_phys, int N, int H,
                        int I, const uint16_t* w_gate, const uint16_t* w_up, int activation,
                        uint16_t* act, gbmoe_stream_t stream) {
    if (!valid_activation(activation)) return GBMOE_ERR_UNSUPPORTED;
    if (N < 0 || H <= 0 || I <= 0 || E_phys < 1) return GBMOE_ERR_INVALID_ARG;
    if (E_phys > gemm_max_groups()) return GBMOE_ERR_UNSUPPORTED;
    if (!offsets && E_phys != 1) return GBMOE_ERR_INVALID_ARG;
    if (H % 128 || I % 128) return GBMOE_ERR_UNSUPPORTED;
    if (N == 0) return GBMOE_OK;
    if (!x_perm || !w_gate || !w_up || !act) return GBMOE_ERR_INVALID_ARG;
    if (!aligned16(x_perm) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(act))
        return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return launch_gemm_gateup(x_perm, nullptr, 0, offsets, E_phys, N, H, I, w_gate, w_up,
                              activation, act, *ctx, reinterpret_cast<cudaStream_t>(stream));
}

int moe_gemm_gateup_act_rows(const uint16_t* x, const int32_t* row_to_token, int T,
                             const int32_t* offsets, int E_phys, int N, int H, int I,
                             const uint16_t* w_gate, const uint16_t* w_up, int activation,
                             uint16_t* act, gbmoe_stream_t stream) {
    if (!valid_activation(activation)) return GBMOE_ERR_UNSUPPORTED;
    if (N < 0 || T < 0 || H <= 0 || I <= 0 || E_phys < 1) return GBMOE_ERR_INVALID_ARG;
    if (E_phys > gemm_max_groups()) return GBMOE_ERR_UNSUPPORTED;
    if (!offsets && E_phys != 1) return GBMOE_ERR_INVALID_ARG;
    if (H % 128 || I % 128) return GBMOE_ERR_UNSUPPORTED;
    if (N == 0) return GBMOE_OK;
    if (T < 1 || !x || !row_to_token || !w_gate || !w_up || !act) return GBMOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(act))
        return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return launch_gemm_gateup(x, row_to_token, T, offsets, E_phys, N, H, I, w_gate, w_up,
                              activation, act, *ctx, reinterpret_cast<cudaStream_t>(stream));
}

int moe_gemm_down(const uint16_t* act, const int32_t* offsets, int E_phys, int N, int H, int I,
                  const uint16_t* w_down, float* y, gbmoe_stream_t stream) {
    if (N < 0 || H <= 0 || I <= 0 || E_phys < 1) return GBMOE_ERR_INVALID_ARG;
    if (E_phys > gemm_max_groups()) return GBMOE_ERR_UNSUPPORTED;
    if (!offsets && E_phys != 1) return GBMOE_ERR_INVALID_ARG;
    if (H % 128 || I % 128) return GBMOE_ERR_UNSUPPORTED;
    if (N == 0) return GBMOE_OK;
    if (!act || !w_down || !y) return GBMOE_ERR_INVALID_ARG;
    if (!aligned16(act) || !aligned16(w_down) || !aligned16(y)) return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return launch_gemm_down(act, offsets, E_phys, N, H, I, w_down, y, *ctx,
                            reinterpret_cast<cudaStream_t>(stream));
}

int gbmoe_expert_mlp_fused(int E_phys, int N, int H) {
    return gemm_fused_eligible(E_phys, N, H) ? 1 : 0;
}

int moe_expert_mlp(const uint16_t* x_rows, const int32_t* row_to_token, int T,
                   const int32_t* offsets, int E_phys, int N, int H, int I,
                   const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                   int activation, uint16_t* act, float* y, int32_t* ready,
                   gbmoe_stream_t stream) {
    if (!valid_activation(activation)) return GBMOE_ERR_UNSUPPORTED;
    if (N < 0 || H <= 0 || I <= 0 || E_phys < 1) return GBMOE_ERR_INVALID_ARG;
    if (E_phys > gemm_max_groups()) return GBMOE_ERR_UNSUPPORTED;
    if (!offsets && E_phys != 1) return GBMOE_ERR_INVALID_ARG;
    if (H % 128 || I % 128) return GBMOE_ERR_UNSUPPORTED;
    if (row_to_token && T < 1) return GBMOE_ERR_INVALID_ARG;
    if (N == 0) return GBMOE_OK;
    if (!x_rows || !w_gate || !w_up || !w_down || !act || !y) return GBMOE_ERR_INVALID_ARG;
    if (!aligned16(x_rows) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
        !aligned16(act) || !aligned16(y))
        return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int src_rows = row_to_token ? T : N;
    if (ready && gemm_fused_eligible(E_phys, N, H))
        return launch_gemm_mlp_fused(x_rows, row_to_token, src_rows, offsets, E_phys, N, H, I,
                                     w_gate, w_up, w_down, activation, act, y, ready, *ctx, s);
    int st = launch_gemm_gateup(x_rows, row_to_token, src_rows, offsets, E_phys, N, H, I, w_gate,
                                w_up, activation, act, *ctx, s);
    if (st) return st;
    return launch_gemm_down(act, offsets, E_phys, N, H, I, w_down, y, *ctx, s);
}

int moe_combine(const float* y, const int32_t* flat_to_row, const float* weights,
                const float* shared_y, int T, int k, int H, uint16_t* out,
                gbmoe_stream_t stream) {
    if (T < 0 || k < 1 || k > kMaxTopK || H <= 0 || H % 8) return GBMOE_ERR_INVALID_ARG;
    if (T == 0) return GBMOE_OK;
    if (!y || !flat_to_row || !weights || !out) return GBMOE_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(out) || (shared_y && !aligned16(shared_y)))
        return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return status_from(launch_combine(y, flat_to_row, weights, shared_y, T, k, H, out, *ctx,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

int moe_gemm_gateup_act_fp8(const uint8_t* xq, const float* sx, const int32_t* row_to_token,
                            int T, const int32_t* offsets, int E_phys, int N, int H, int I,
                            const uint8_t* wgq, const float* sg, const uint8_t* wuq,
                            const float* su, int activation, uint16_t* act,
                            gbmoe_stream_t stream) {
    if (!valid_activation(activation)) return GBMOE_ERR_UNSUPPORTED;
    if (N < 0 || H <= 0 || I <= 0 || E_phys < 1) return GBMOE_ERR_INVALID_ARG;
    if (E_phys > gemm_max_groups()) return GBMOE_ERR_UNSUPPORTED;
    if (!offsets && E_phys != 1) return GBMOE_ERR_INVALID_ARG;
    if (H % 256 || I % 128) return GBMOE_ERR_UNSUPPORTED;
    if (N == 0) return GBMOE_OK;
    if (row_to_token && T < 1) return GBMOE_ERR_INVALID_ARG;
    if (!xq || !sx || !wgq || !sg || !wuq || !su || !act) return GBMOE_ERR_INVALID_ARG;
    if (!aligned16(xq) || !aligned16(wgq) || !aligned16(wuq) || !aligned16(act))
        return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return launch_gemm_gateup_fp8(xq, sx, row_to_token, row_to_token ? T : N, offsets, E_phys, N,
                                  H, I, wgq, sg, wuq, su, activation, act, *ctx,
                                  reinterpret_cast<cudaStream_t>(stream));
}

int moe_gemm_down_fp8(const uint8_t* aq, const float* sa, const int32_t* offsets, int E_phys,
                      int N, int H, int I, const uint8_t* wdq, const float* sd, float* y,
                      gbmoe_stream_t stream) {
    if (N < 0 || H <= 0 || I <= 0 || E_phys < 1) return GBMOE_ERR_INVALID_ARG;
    if (E_phys > gemm_max_groups()) return GBMOE_ERR_UNSUPPORTED;
    if (!offsets && E_phys != 1) return GBMOE_ERR_INVALID_ARG;
    if (H % 256 || I % 128) return GBMOE_ERR_UNSUPPORTED;
    if (N == 0) return GBMOE_OK;
    if (!aq || !sa || !wdq || !sd || !y) return GBMOE_ERR_INVALID_ARG;
    if (!aligned16(aq) || !aligned16(wdq) || !aligned16(y)) return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return launch_gemm_down_fp8(aq, sa, offsets, E_phys, N, H, I, wdq, sd, y, *ctx,
                                reinterpret_cast<cudaStream_t>(stream));
}

int moe_quantize_fp8_rows(const uint16_t* x, int64_t n, int K, uint8_t* q, float* scales,
                          gbmoe_stream_t stream) {
    if (n < 0 || K <= 0) return GBMOE_ERR_INVALID_ARG;
    if (K % 8) return GBMOE_ERR_UNSUPPORTED;
    if (n == 0) return GBMOE_OK;
    if (!x || !q || !scales || !aligned16(x) || (reinterpret_cast<uintptr_t>(q) & 7u))
        return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return status_from(launch_quantize_rows(x, n, K, q, scales, *ctx,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

int moe_quantize_mx_rows(const uint16_t* x, int64_t n, int K, int fmt, uint8_t* q,
                         uint8_t* scales, gbmoe_stream_t stream) {
    if (n < 0 || K <= 0) return GBMOE_ERR_INVALID_ARG;
    if (fmt != GBMOE_MX_E4M3 && fmt != GBMOE_MX_E2M1) return GBMOE_ERR_UNSUPPORTED;
    if (K % 32) return GBMOE_ERR_UNSUPPORTED;
    if (n == 0) return GBMOE_OK;
    if (!x || !q || !scales || !aligned16(x) || !aligned16(q)) return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return status_from(launch_mx_quantize(x, n, K, fmt, q, scales, *ctx,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int moe_mx_tile_scales(const uint8_t* sf_rows, int64_t rows, int K, uint8_t* sf_tiled,
                       gbmoe_stream_t stream) {
    if (rows < 0 || K <= 0) return GBMOE_ERR_INVALID_ARG;
    if (rows % 128 || K % 128) return GBMOE_ERR_UNSUPPORTED;
    if (rows == 0) return GBMOE_OK;
    if (!sf_rows || !sf_tiled || !aligned4(sf_rows) || !aligned16(sf_tiled))
        return GBMOE_ERR_INVALID_ARG;
    const size_t bytes = static_cast<size_t>(rows) * (K / 32);
    const uintptr_t a = reinterpret_cast<uintptr_t>(sf_rows), b = reinterpret_cast<uintptr_t>(sf_tiled);
    if (a < b + bytes && b < a + bytes) return GBMOE_ERR_INVALID_ARG;  // must not overlap
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return status_from(launch_mx_tile_scales(sf_rows, rows, K, sf_tiled, *ctx,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int moe_gemm_gateup_act_mx(const uint8_t* xq, const uint8_t* xs, const int32_t* row_to_token,
                           int T, const int32_t* offsets, int E_phys, int N, int H, int I,
                           int w_fmt, const uint8_t* wgq, const uint8_t* sg, const uint8_t* wuq,
                           const uint8_t* su, int activation, uint8_t* act_q, uint8_t* act_s,
                           gbmoe_stream_t stream) {
    if (!valid_activation(activation)) return GBMOE_ERR_UNSUPPORTED;
    if (w_fmt != GBMOE_MX_E4M3 && w_fmt != GBMOE_MX_E2M1) return GBMOE_ERR_UNSUPPORTED;
    if (N < 0 || H <= 0 || I <= 0 || E_phys < 1) return GBMOE_ERR_INVALID_ARG;
    if (E_phys > gemm_max_groups()) return GBMOE_ERR_UNSUPPORTED;
    if (!offsets && E_phys != 1) return GBMOE_ERR_INVALID_ARG;
    if (H % 256 || I % 128) return GBMOE_ERR_UNSUPPORTED;
    if (N == 0) return GBMOE_OK;
    if (row_to_token && T < 1) return GBMOE_ERR_INVALID_ARG;
    if (!xq || !xs || !wgq || !sg || !wuq || !su || !act_q || !act_s)
        return GBMOE_ERR_INVALID_ARG;
    if (!aligned16(xq) || !mx_weights_aligned(w_fmt, wgq) || !mx_weights_aligned(w_fmt, wuq) ||
        !aligned4(xs) || !aligned16(sg) || !aligned16(su))
        return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return launch_gemm_gateup_mx(xq, xs, row_to_token, row_to_token ? T : N, offsets, E_phys, N,
                                 H, I, w_fmt, wgq, sg, wuq, su, activation, act_q, act_s, *ctx,
                                 reinterpret_cast<cudaStream_t>(stream));
}

int moe_gemm_down_mx(const uint8_t* aq, const uint8_t* as, const int32_t* offsets, int E_phys,
                     int N, int H, int I, int w_fmt, const uint8_t* wdq, const uint8_t* sd,
                     float* y, gbmoe_stream_t stream) {
    if (w_fmt != GBMOE_MX_E4M3 && w_fmt != GBMOE_MX_E2M1) return GBMOE_ERR_UNSUPPORTED;
    if (N < 0 || H <= 0 || I <= 0 || E_phys < 1) return GBMOE_ERR_INVALID_ARG;
    if (E_phys > gemm_max_groups()) return GBMOE_ERR_UNSUPPORTED;
    if (!offsets && E_phys != 1) return GBMOE_ERR_INVALID_ARG;
    if (H % 256 || I % 128) return GBMOE_ERR_UNSUPPORTED;
    if (N == 0) return GBMOE_OK;
    if (!aq || !as || !wdq || !sd || !y) return GBMOE_ERR_INVALID_ARG;
    if (!aligned16(aq) || !mx_weights_aligned(w_fmt, wdq) || !aligned4(as) || !aligned16(sd) ||
        !aligned16(y))
        return GBMOE_ERR_INVALID_ARG;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return launch_gemm_down_mx(aq, as, offsets, E_phys, N, H, I, w_fmt, wdq, sd, y, *ctx,
                               reinterpret_cast<cudaStream_t>(stream));
}

size_t gbmoe_latent_tail_workspace_size(int T, int L, int Hm) {
    if (T < 0 || L <= 0 || Hm <= 0) return 0;
    return latent_tail_ws_bytes(T, L, Hm);
}

int moe_latent_tail(const uint16_t* latent, int T, int L, const uint16_t* norm_w, float eps,
                    const uint16_t* up_proj, int Hm, const uint16_t* shared, uint16_t* out,
                    void* ws, size_t ws_bytes, gbmoe_stream_t stream) {
    if (T < 0 || L <= 0 || Hm <= 0) return GBMOE_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || eps > 1e30f) return GBMOE_ERR_INVALID_ARG;
    if (L % 128 || Hm % 128) return GBMOE_ERR_UNSUPPORTED;
    if (T == 0) return GBMOE_OK;
    if (!latent || !up_proj || !out || !ws) return GBMOE_ERR_INVALID_ARG;
    if (!aligned16(latent) || !aligned16(up_proj) || !aligned16(out) || !aligned16(ws) ||
        (shared && !aligned16(shared)))
        return GBMOE_ERR_INVALID_ARG;
    if (ws_bytes < latent_tail_ws_bytes(T, L, Hm)) return GBMOE_ERR_WORKSPACE;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    return launch_latent_tail(latent, T, L, norm_w, eps, up_proj, Hm, shared, out, ws, *ctx,
                              reinterpret_cast<cudaStream_t>(stream));
}

size_t gbmoe_forward_workspace_size(const gbmoe_layer* L, int T_max) {
    if (check_layer(L) || T_max < 0) return 0;
    return layout_fwd(L, T_max, nullptr).bytes;
}

int moe_forward(const gbmoe_layer* L, const uint16_t* x, int T, const int32_t* input_ids,
                uint16_t* out, int32_t* ids_log, int32_t* ids_phys, float* weights,
                int32_t* counts, void* ws, size_t ws_bytes, gbmoe_stream_t stream) {
    int st = check_layer(L);
    if (st) return st;
    if (T < 0) return GBMOE_ERR_INVALID_ARG;
    if (T == 0) return GBMOE_OK;
    if (!x || !out || !aligned16(x) || !aligned16(out)) return GBMOE_ERR_INVALID_ARG;
    if (L->route.use_hash && !input_ids) return GBMOE_ERR_INVALID_ARG;
    const gbmoe_route_cfg& c = L->route;
    const int64_t N64 = static_cast<int64_t>(T) * c.top_k;
    if (N64 > INT32_MAX / 8) return GBMOE_ERR_UNSUPPORTED;
    const int N = static_cast<int>(N64);
    if (!ws) return GBMOE_ERR_WORKSPACE;
    FwdWs f = layout_fwd(L, T, ws);
    if (ws_bytes < f.bytes) return GBMOE_ERR_WORKSPACE;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t* il = ids_log ? ids_log : f.ids_log;
    int32_t* ip = ids_phys ? ids_phys : f.ids_phys;
    float* wt = weights ? weights : f.weights;
    int32_t* cn = counts ? counts : f.counts;

    // 1. router logits + selection + log2phy ("Stage 2", "Stage 4" step 2)
    RouteArgs ra{c, T, L->H, x, L->w_router, f.logits, L->router_bias, L->corr_bias, input_ids,
                 L->tid2eid, L->tid2eid_rows, L->log2phy, L->replica_cnt, L->R_max, il, ip, wt,
                 nullptr};
    ra.hash_logits_only = 1;  // f.logits is scratch: only the selection reads it
    st = status_from(launch_route(ra, *ctx, s));
    if (st) return st;
    // 2. dispatch: counts, offsets, stable permutation ("Stage 4" AllGather
    // row); the permuted rows are not materialised: the gate/up GEMM gathers
    // them from x through row_to_token
    st = status_from(launch_permute(ip, N, c.top_k, c.E_phys, x, L->H, cn, f.offsets,
                                    f.row_to_token, f.flat_to_row, nullptr, f.perm, *ctx, s));
    if (st) return st;
    // 3-4. grouped gate/up + SwiGLU, grouped down ("Stage 4": unified_apply_mlp);
    // one fused launch for small groups
    if (L->w_gate_q) {
        // FP8 routed experts: hidden states and activations quantized per row
        st = status_from(launch_quantize_rows(x, T, L->H, f.xq, f.sx, *ctx, s));
        if (st) return st;
        st = launch_gemm_gateup_fp8(f.xq, f.sx, f.row_to_token, T, f.offsets, c.E_phys, N, L->H,
                                    L->I, L->w_gate_q, L->s_gate, L->w_up_q, L->s_up,
                                    L->activation, f.act, *ctx, s);
        if (st) return st;
        st = status_from(launch_quantize_rows(f.act, N, L->I, f.aq, f.sa, *ctx, s));
        if (st) return st;
        st = launch_gemm_down_fp8(f.aq, f.sa, f.offsets, c.E_phys, N, L->H, L->I, L->w_down_q,
                                  L->s_down, f.y, *ctx, s);
        if (st) return st;
    } else if (L->w_gate_mx) {
        // MX routed experts: hidden states quantized per 32-element block; the
        // gate/up GEMM writes the activation already quantized
        st = status_from(launch_mx_quantize(x, T, L->H, GBMOE_MX_E4M3, f.xq, f.xs, *ctx, s));
        if (st) return st;
        st = launch_gemm_gateup_mx(f.xq, f.xs, f.row_to_token, T, f.offsets, c.E_phys, N, L->H,
                                   L->I, L->mx_format, L->w_gate_mx, L->sf_gate, L->w_up_mx,
                                   L->sf_up, L->activation, f.aq, f.as, *ctx, s);
        if (st) return st;
        st = launch_gemm_down_mx(f.aq, f.as, f.offsets, c.E_phys, N, L->H, L->I, L->mx_format,
                                 L->w_down_mx, L->sf_down, f.y, *ctx, s);
        if (st) return st;
    } else if (gemm_fused_eligible(c.E_phys, N, L->H)) {
        st = launch_gemm_mlp_fused(x, f.row_to_token, T, f.offsets, c.E_phys, N, L->H, L->I,
                                   L->w_gate, L->w_up, L->w_down, L->activation, f.act, f.y,
                                   f.ready, *ctx, s);
        if (st) return st;
    } else {
        st = launch_gemm_gateup(x, f.row_to_token, T, f.offsets, c.E_phys, N, L->H, L->I,
                                L->w_gate, L->w_up, L->activation, f.act, *ctx, s);
        if (st) return st;
        st = launch_gemm_down(f.act, f.offsets, c.E_phys, N, L->H, L->I, L->w_down, f.y, *ctx,
                              s);
        if (st) return st;
    }
    // 5. shared expert over all tokens in order (one group)
    const float* ys = nullptr;
    if (L->I_shared) {
        st = launch_gemm_gateup(x, nullptr, 0, nullptr, 1, T, L->H, L->I_shared,
                                L->w_gate_shared, L->w_up_shared, L->activation, f.act_s, *ctx,
                                s);
        if (st) return st;
        st = launch_gemm_down(f.act_s, nullptr, 1, T, L->H, L->I_shared, L->w_down_shared, f.ys,
                              *ctx, s);
        if (st) return st;
        ys = f.ys;
    }
    // 6. combine: restore token order, apply weights, add the shared expert
    return status_from(launch_combine(f.y, f.flat_to_row, wt, ys, T, c.top_k, L->H, out, *ctx, s));
}

size_t gbmoe_forward_host_workspace_size(const gbmoe_layer* L, int T_max) {
    const size_t base = gbmoe_forward_workspace_size(L, T_max);
    if (!base) return 0;
    const size_t TH = static_cast<size_t>(T_max) * L->H;
    return base + 2 * align256(TH * 2) + align256(static_cast<size_t>(T_max) * 4) +
           align256(static_cast<size_t>(T_max) * L->route.top_k * 4);
}

int moe_forward_host(const gbmoe_layer* L, const uint16_t* x_host, int T,
                     const int32_t* input_ids_host, uint16_t* out_host, int32_t* ids_log_host,
                     void* ws, size_t ws_bytes, gbmoe_stream_t stream) {
    int st = check_layer(L);
    if (st) return st;
    if (T < 0) return GBMOE_ERR_INVALID_ARG;
    if (T == 0) return GBMOE_OK;
    if (!x_host || !out_host || (L->route.use_hash && !input_ids_host)) return GBMOE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < gbmoe_forward_host_workspace_size(L, T)) return GBMOE_ERR_WORKSPACE;
    const size_t fw = gbmoe_forward_workspace_size(L, T);
    const size_t TH = static_cast<size_t>(T) * L->H;
    WsCursor w{static_cast<char*>(ws) + fw, 0};
    uint16_t* x_dev = w.take<uint16_t>(TH);
    uint16_t* out_dev = w.take<uint16_t>(TH);
    int32_t* ids_dev = w.take<int32_t>(T);
    int32_t* il_dev = w.take<int32_t>(static_cast<size_t>(T) * L->route.top_k);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = status_from(cudaMemcpyAsync(x_dev, x_host, TH * 2, cudaMemcpyHostToDevice, s));
    if (st) return st;
    if (L->route.use_hash) {
        st = status_from(cudaMemcpyAsync(ids_dev, input_ids_host, static_cast<size_t>(T) * 4,
                                         cudaMemcpyHostToDevice, s));
        if (st) return st;
    }
    st = moe_forward(L, x_dev, T, L->route.use_hash ? ids_dev : nullptr, out_dev, il_dev, nullptr,
                     nullptr, nullptr, ws, fw, stream);
    if (st) return st;
    st = status_from(cudaMemcpyAsync(out_host, out_dev, TH * 2, cudaMemcpyDeviceToHost, s));
    if (st) return st;
    if (ids_log_host)
        st = status_from(cudaMemcpyAsync(ids_log_host, il_dev,
                                         static_cast<size_t>(T) * L->route.top_k * 4,
                                         cudaMemcpyDeviceToHost, s));
    return st;
}

}  // extern "C"
