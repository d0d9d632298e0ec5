/*
 * gbmoe — routed mixture-of-experts layer forward for GB300 (sm_103a).
 *
 * C ABI of libgbmoe.so.  The operations follow the routed-MoE forward traced
 * on the vLLM-Ascend "Kimi K3 MoE Forward Insight" page: expert selection
 * (section "Stage 2: Select Experts", with the routing settings listed under
 * "Runner Initialization"), logical-to-physical mapping and token dispatch
 * (section "Stage 4: Dispatch, MLP, Combine", AllGather row of its table),
 * the grouped gate/up -> activation -> down expert MLP (same section), the
 * combine that restores token order and applies the routing probabilities
 * (same table), and per-expert token counts for load tracking (section
 * "Stage 6: Dynamic EPLB").  On one GPU the dispatch is a local permutation:
 * no expert parallelism and no collectives.  The same section's quantized
 * expert paths are provided as FP8 E4M3 with per-row scales (W8A8FP) and MX
 * block-scaled experts (MXFP8, and W4A8 read as E2M1 weights with E4M3
 * activations); the NVIDIA LatentMoERunner page's post-MoE tail (RMSNorm,
 * up-projection, shared-expert add) is provided for one GPU.
 *
 * Conventions shared by every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller (except where a
 *    name ends in _host), row-major and contiguous with the stated shapes.
 *    bf16 tensors are passed as uint16_t* (raw bf16 bits).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and performs no host synchronisation.  It returns
 *    a gbmoe_status.  Argument errors are detected on the host before any
 *    work is enqueued and leave all outputs untouched.  Errors that only the
 *    device can see (an out-of-range id in a caller table, a pipeline wait
 *    that gave up) are recorded in a per-device status word and reported by
 *    gbmoe_check_device_status(); the affected outputs are then unspecified.
 *  - T = 0 is valid and enqueues nothing (outputs of size 0).
 *  - No exception crosses the ABI.  The library keeps one lazily created
 *    context per device (its status word and SM count); it is thread-safe.
 */
#ifndef GBMOE_H
#define GBMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gbmoe_stream_t; /* == cudaStream_t */

enum gbmoe_status {
    GBMOE_OK = 0,
    GBMOE_ERR_INVALID_ARG = 1, /* bad shape, pointer or configuration */
    GBMOE_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels handle */
    GBMOE_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
    GBMOE_ERR_CUDA = 4,        /* a CUDA runtime call failed */
    GBMOE_ERR_DEVICE = 5,      /* a device-side check tripped (bad table entry / id) */
    GBMOE_ERR_TIMEOUT = 6      /* a GEMM pipeline wait gave up (bounded wait) */
};

/* scoring function ("Stage 2: Select Experts": softmax, sigmoid, sqrtsoftplus) */
enum { GBMOE_SCORE_SOFTMAX = 0, GBMOE_SCORE_SIGMOID = 1, GBMOE_SCORE_SQRTSOFTPLUS = 2 };
/* group score used by grouped top-k */
enum { GBMOE_GROUP_MAX = 0, GBMOE_GROUP_TOP2SUM = 1 };
/* Gated activation of the gate/up GEMM epilogue, act = f(g, u) on the fp32
 * gate and up projections, rounded to bf16 ("Stage 4" activation branches):
 *   GBMOE_ACT_SWIGLU       silu(g) * u, silu(g) = g / (1 + e^-g)
 *   GBMOE_ACT_SWIGLU_OAI   clipped: g' = min(g, 7), u' = clamp(u, -7, 7),
 *                          g' * sigmoid(1.702 g') * (u' + 1)
 *   GBMOE_ACT_GEGLU        0.5 g (1 + erf(g / sqrt 2)) * u
 *   GBMOE_ACT_GEGLU_TANH   0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) * u */
enum {
    GBMOE_ACT_SWIGLU = 0,
    GBMOE_ACT_SWIGLU_OAI = 1,
    GBMOE_ACT_GEGLU = 2,
    GBMOE_ACT_GEGLU_TANH = 3
};

/*
 * Routing settings ("Runner Initialization": grouped top-k settings,
 * renormalisation, scoring function, correction bias, routed scaling; "Entry
 * Point": tid2eid for hash routing).
 *   E_log       logical experts (1..1024)
 *   E_phys      physical slots (E_log..1024); E_phys == E_log without log2phy
 *   top_k       experts per token (1..min(E_log, 32))
 *   n_group     expert groups for grouped top-k (1 = flat); divides E_log
 *   topk_group  groups kept (1..n_group); topk_group * E_log/n_group >= top_k
 *   scoring     GBMOE_SCORE_*
 *   group_score GBMOE_GROUP_*
 *   renormalize 1: w_j = s_j / sum_j s_j * routed_scaling; 0: s_j * routed_scaling
 *   use_hash    1: ids come from tid2eid[input_ids[t]] (requires n_group == 1
 *               and no correction bias)
 * Scores s are the unbiased scoring-function values; a correction bias, when
 * given, enters the selection only.
 */
typedef struct gbmoe_route_cfg {
    int E_log;
    int E_phys;
    int top_k;
    int n_group;
    int topk_group;
    int scoring;
    int group_score;
    int renormalize;
    float routed_scaling;
    int use_hash;
} gbmoe_route_cfg;

/* One layer: routing settings, sizes and (device) weights. */
typedef struct gbmoe_layer {
    gbmoe_route_cfg route;
    int H;                        /* hidden size, multiple of 128 */
    int I;                        /* expert intermediate size, multiple of 128 */
    int I_shared;                 /* shared-expert intermediate (0: none), multiple of 128 */
    const float* w_router;        /* [E_log, H] fp32 router weight */
    const float* router_bias;     /* [E_log] fp32 added to the logits, or NULL */
    const float* corr_bias;       /* [E_log] fp32 selection-only bias, or NULL */
    const int32_t* tid2eid;       /* [tid2eid_rows, top_k] (use_hash) */
    int64_t tid2eid_rows;
    const int32_t* log2phy;       /* [E_log, R_max] physical slot of each replica, or NULL */
    const int32_t* replica_cnt;   /* [E_log] replicas per logical expert (1..R_max) */
    int R_max;
    const uint16_t* w_gate;       /* [E_phys, I, H] bf16 */
    const uint16_t* w_up;         /* [E_phys, I, H] bf16 */
    const uint16_t* w_down;       /* [E_phys, H, I] bf16 */
    const uint16_t* w_gate_shared;/* [I_shared, H] bf16 or NULL */
    const uint16_t* w_up_shared;  /* [I_shared, H] bf16 or NULL */
    const uint16_t* w_down_shared;/* [H, I_shared] bf16 or NULL */
    int activation;               /* GBMOE_ACT_*, of the routed and the shared experts */
    /* FP8 routed experts (W8A8FP, see moe_gemm_gateup_act_fp8): when w_gate_q
     * is non-NULL the routed expert MLP runs on these E4M3 codes and per-row
     * scales (hidden states and activations are quantized per row on the fly)
     * and w_gate / w_up / w_down may be NULL; H % 256 == 0.  The shared expert
     * stays bf16. */
    const uint8_t* w_gate_q;      /* [E_phys, I, H] E4M3 codes */
    const float* s_gate;          /* [E_phys, I] */
    const uint8_t* w_up_q;        /* [E_phys, I, H] */
    const float* s_up;            /* [E_phys, I] */
    const uint8_t* w_down_q;      /* [E_phys, H, I] */
    const float* s_down;          /* [E_phys, H] */
    /* MX block-scaled routed experts (MXFP8 / W4A8, see moe_gemm_gateup_act_mx):
     * when w_gate_mx is non-NULL (and w_gate_q is NULL) the routed expert MLP
     * runs on these codes in format mx_format (GBMOE_MX_E4M3 or
     * GBMOE_MX_E2M1) with UE8M0 scale bytes per 32 elements along K; hidden
     * states and activations are MX E4M3 (quantized on the fly).  H % 256 ==
     * 0.  The shared expert stays bf16. */
    int mx_format;
    const uint8_t* w_gate_mx;     /* [E_phys, I, H] (E4M3) or [E_phys, I, H/2] (E2M1) */
    const uint8_t* sf_gate;       /* [E_phys, I, H/32], tiled (moe_mx_tile_scales) */
    const uint8_t* w_up_mx;       /* as w_gate_mx */
    const uint8_t* sf_up;         /* [E_phys, I, H/32], tiled */
    const uint8_t* w_down_mx;     /* [E_phys, H, I] (E4M3) or [E_phys, H, I/2] (E2M1) */
    const uint8_t* sf_down;       /* [E_phys, H, I/32], tiled */
} gbmoe_layer;

/* Text for a status code (static storage). */
const char* gbmoe_status_string(int status);

/* Host-side check of a routing configuration (GBMOE_OK or INVALID_ARG). */
int gbmoe_validate_route_cfg(const gbmoe_route_cfg* cfg);

/*
 * Host-side check of a placement table ("Stage 6: Dynamic EPLB": every
 * logical expert stays placed; no physical slot is shared by two logical
 * experts).  log2phy_host [E_log, R_max], replica_cnt_host [E_log] in host
 * memory.  Returns GBMOE_OK or GBMOE_ERR_INVALID_ARG.
 */
int gbmoe_validate_log2phy(const int32_t* log2phy_host, const int32_t* replica_cnt_host,
                           int E_log, int R_max, int E_phys);

/*
 * Synchronises `stream`, then reads and clears this device's status word.
 * *status receives GBMOE_OK or the first device-side error recorded since
 * the last check (GBMOE_ERR_DEVICE / GBMOE_ERR_TIMEOUT).  Not for hot loops.
 */
int gbmoe_check_device_status(gbmoe_stream_t stream, int* status);

/*
 * gbmoe_set_wait_limit_ns — wall-clock limit of every bounded wait inside
 * the grouped-GEMM kernels launched after this call (the pipeline's stage
 * waits, and the fused launch's wait for an expert's activations).  A wait
 * that runs out records GBMOE_ERR_TIMEOUT in the device status; the launch
 * then lets its in-flight copies and MMAs finish (under a fixed limit of its
 * own), frees its tensor memory and returns, leaving the context usable.
 * The vLLM-Ascend page's "Where It Breaks" section traces hangs of the MoE
 * path; this library turns such a stall into a reported error.
 *   ns = 0 restores the default (4 s).  Process-wide, thread-safe; launches
 *   already enqueued keep the limit they were launched with.  A very small
 *   limit makes healthy launches give up too (that is how the timeout path
 *   is tested); their outputs are then unspecified.  Waits on a pipeline
 *   barrier compare the clock between suspended polls of the barrier, so
 *   their effective limit can exceed a very small setting; the fused
 *   launch's wait for an expert's activations polls memory and keeps to it.
 * Returns the previous limit in nanoseconds.
 */
uint64_t gbmoe_set_wait_limit_ns(uint64_t ns);

/*
 * moe_route — router scoring and expert selection ("Stage 2: Select
 * Experts"), then the logical -> physical mapping ("Stage 4", step 2: map
 * logical topk_ids through log2phy).
 *   x            [T, H] bf16 hidden states (read when w_router != NULL)
 *   w_router     [E_log, H] fp32, or NULL when the caller supplies logits
 *   logits       [T, E_log] fp32: OUTPUT (router logits) when w_router is
 *                given, INPUT otherwise; always required
 *   router_bias  [E_log] fp32 added to computed logits, or NULL
 *   corr_bias    [E_log] fp32 selection-only bias, or NULL
 *   input_ids    [T] token ids (use_hash), tid2eid [tid2eid_rows, top_k]
 *   log2phy      [E_log, R_max] + replica_cnt [E_log], or NULL (identity);
 *                token t uses replica (t mod replica_cnt[e])
 *   ids_log      [T, top_k] int32 logical expert ids in user token order
 *                (the routed-expert capture of "Stage 5")
 *   ids_phys     [T, top_k] int32 physical slots
 *   weights      [T, top_k] fp32 routing weights
 *   counts       [E_phys] int32 tokens per physical slot (overwritten), or NULL
 * Selection order: slots hold experts in descending selection score, ties
 * to the lower expert id.  Logits use a fixed fp32 summation order, so ids
 * and weights are reproducible bit for bit.
 */
int moe_route(const gbmoe_route_cfg* cfg, const uint16_t* x, int T, int H,
              const float* w_router, float* logits, const float* router_bias,
              const float* corr_bias, const int32_t* input_ids, const int32_t* tid2eid,
              int64_t tid2eid_rows, const int32_t* log2phy, const int32_t* replica_cnt,
              int R_max, int32_t* ids_log, int32_t* ids_phys, float* weights, int32_t* counts,
              gbmoe_stream_t stream);

/*
 * moe_expert_counts — tokens per physical expert ("Stage 6": expert_tokens
 * converted to per-expert counts and added into moe_load).
 *   ids_phys [T, k] int32; counts [E_phys] int32, overwritten (accumulate=0)
 *   or incremented (accumulate=1).  Integer counts: deterministic.
 */
int moe_expert_counts(const int32_t* ids_phys, int T, int k, int E_phys, int32_t* counts,
                      int accumulate, gbmoe_stream_t stream);

/* Scratch bytes moe_permute needs for T tokens, k slots, E_phys experts. */
size_t gbmoe_permute_workspace_size(int T, int k, int E_phys);

/*
 * moe_permute — dispatch as a local permutation ("Stage 4" table, AllGather
 * row: sort tokens by expert and return expert token counts).
 * Stable: row r = offsets[p] + (rank of flat index t*k+j among the pairs
 * routed to p), so rows of one expert keep token order.  Bit-exact and
 * deterministic (no atomics decide an order).
 *   ids_phys     [T, k] int32 in [0, E_phys)
 *   x            [T, H] bf16 (read only when x_perm != NULL)
 *   counts       [E_phys] int32 out
 *   offsets      [E_phys + 1] int32 out (exclusive scan; offsets[E_phys] = T*k)
 *   row_to_token [T*k] int32 out; flat_to_row [T*k] int32 out
 *   x_perm       [T*k, H] bf16 out (x_perm[r] = x[row_to_token[r]]), or NULL
 *   ws           device scratch of ws_bytes >= gbmoe_permute_workspace_size()
 * An id outside [0, E_phys) sets GBMOE_ERR_DEVICE and is skipped: it is not
 * counted, gets no row (its flat_to_row entry is -1), and offsets[E_phys] is
 * then below T*k; row_to_token entries from offsets[E_phys] on are not written
 * and those x_perm rows are zero-filled (x is read only through rows that the
 * permutation wrote).
 */
int moe_permute(const int32_t* ids_phys, int T, int k, int E_phys, const uint16_t* x, int H,
                int32_t* counts, int32_t* offsets, int32_t* row_to_token, int32_t* flat_to_row,
                uint16_t* x_perm, void* ws, size_t ws_bytes, gbmoe_stream_t stream);

/*
 * moe_permute_static — the same permutation as moe_permute, for callers that
 * cannot allocate device memory (cudaMalloc/cudaFree can synchronise the
 * device and stall every stream, and a process whose GPU memory belongs to
 * another framework's pool must not allocate behind it).  The pages have no
 * counterpart to this entry point; it is an addition of this library.
 *
 * Arguments, outputs and results are those of moe_permute, without the
 * workspace: the scratch lives in a 1 MiB array inside the library, one per
 * device, held until the process exits.  The library allocates nothing.
 *   Limit: ceil(T*k/256) * E_phys * 4 + 256 bytes must fit in 1 MiB
 *   (e.g. E_phys = 256 allows T*k up to 261,888); larger requests return
 *   GBMOE_ERR_WORKSPACE and enqueue nothing.
 *   The first call on each device resolves the array's device address
 *   (cudaGetSymbolAddress with that device current); make it before any
 *   stream capture.
 *   All calls share the array and it keeps the last call's contents; calls
 *   that overlap on the GPU (several streams or threads) race on it, so the
 *   caller must serialise them.
 */
int moe_permute_static(const int32_t* ids_phys, int T, int k, int E_phys, const uint16_t* x,
                       int H, int32_t* counts, int32_t* offsets, int32_t* row_to_token,
                       int32_t* flat_to_row, uint16_t* x_perm, gbmoe_stream_t stream);

/*
 * moe_gemm_gateup_act — grouped gate/up GEMM with the activation fused into
 * its epilogue ("Stage 4": grouped matmul gate/up -> activation).
 * For each expert p and each row r in [offsets[p], offsets[p+1]):
 *   g = x_perm[r] . w_gate[p]^T,  u = x_perm[r] . w_up[p]^T   (fp32 accumulate)
 *   act[r, i] = bf16(f(g_i, u_i)), f the GBMOE_ACT_* `activation`
 *   (GBMOE_ERR_UNSUPPORTED for any other value)
 *   x_perm [N, H] bf16; offsets [E_phys + 1] int32 on the device, or NULL for a
 *   single group of N rows (E_phys must then be 1); w_gate, w_up [E_phys, I, H]
 *   bf16; act [N, I] bf16 out.  H, I multiples of 128; 16-byte aligned pointers.
 * Runs on tcgen05 tensor cores (TMEM accumulators, TMA-fed shared memory).
 */
int moe_gemm_gateup_act(const uint16_t* x_perm, const int32_t* offsets, int E_phys, int N, int H,
                        int I, const uint16_t* w_gate, const uint16_t* w_up, int activation,
                        uint16_t* act, gbmoe_stream_t stream);

/*
 * moe_gemm_gateup_act_rows — moe_gemm_gateup_act with the token operand
 * gathered inside the GEMM: row r of the operand is x[row_to_token[r]], so no
 * permuted copy of x is needed ("Stage 4": the dispatch's expert-sorted rows,
 * read in place).
 *   x [T, H] bf16; row_to_token [N] int32 (as written by moe_permute); the
 *   other arguments as for moe_gemm_gateup_act.  An entry outside [0, T) is
 *   read as row 0 and reported as GBMOE_ERR_DEVICE through the device status.
 */
int moe_gemm_gateup_act_rows(const uint16_t* x, const int32_t* row_to_token, int T,
                             const int32_t* offsets, int E_phys, int N, int H, int I,
                             const uint16_t* w_gate, const uint16_t* w_up, int activation,
                             uint16_t* act, gbmoe_stream_t stream);

/*
 * moe_gemm_down — grouped down GEMM ("Stage 4": grouped matmul down).
 *   y[r] = act[r] . w_down[p]^T for r in expert p's rows, fp32 accumulate,
 *   written in fp32 (inside the layer only the activation is rounded to bf16).
 *   act [N, I] bf16; w_down [E_phys, H, I] bf16; y [N, H] fp32 out;
 *   offsets as for moe_gemm_gateup_act.
 */
int moe_gemm_down(const uint16_t* act, const int32_t* offsets, int E_phys, int N, int H, int I,
                  const uint16_t* w_down, float* y, gbmoe_stream_t stream);

/*
 * moe_expert_mlp — both grouped GEMMs of the routed experts ("Stage 4":
 * grouped matmul gate/up -> SwiGLU -> grouped matmul down), exactly the
 * results of moe_gemm_gateup_act followed by moe_gemm_down, and the way
 * moe_forward runs them.
 *   x_rows, row_to_token, T: the token operand.  row_to_token NULL: x_rows is
 *     x_perm [N, H] (T ignored).  Otherwise x_rows is the unpermuted x [T, H]
 *     and row r of the operand is x[row_to_token[r]] (row_to_token [N] as
 *     written by moe_permute), gathered inside the GEMM: no x_perm is needed.
 *     An entry outside [0, T) is read as row 0 and reported as
 *     GBMOE_ERR_DEVICE through the device status.
 *   offsets, w_gate, w_up, w_down, activation, act, y as for the two calls
 *   above (act is
 *   written and then read back: it must not alias the token operand or y);
 *   ready: [E_phys] int32 device scratch, overwritten.  When
 *   gbmoe_expert_mlp_fused(E_phys, N, H) is 1 and ready is non-NULL the two
 *   GEMMs run as one launch: the down tiles of an expert start as soon as all
 *   of that expert's activation tiles are written (NULL: two launches).
 * Errors as for the two calls; a fused launch whose wait runs out records
 * GBMOE_ERR_TIMEOUT in the device status (gbmoe_check_device_status).
 */
int moe_expert_mlp(const uint16_t* x_rows, const int32_t* row_to_token, int T,
                   const int32_t* offsets, int E_phys, int N, int H, int I,
                   const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                   int activation, uint16_t* act, float* y, int32_t* ready,
                   gbmoe_stream_t stream);

/* 1 if moe_expert_mlp (and moe_forward) runs the two GEMMs as one launch for
 * this shape (groups averaging fewer than 96 rows, H a multiple of 256). */
int gbmoe_expert_mlp_fused(int E_phys, int N, int H);

/*
 * moe_combine — restore token order and apply the routing probabilities
 * ("Stage 4" table, AllGather combine), plus the shared expert's output
 * ("Forward Skeleton": shared experts).
 *   out[t] = bf16( sum_{j=0..k-1} weights[t,j] * y[flat_to_row[t*k+j]] + shared_y[t] )
 * in fp32, summed in the fixed order j = 0..k-1, then the shared term.
 *   y [T*k, H] fp32; flat_to_row [T*k]; weights [T, k] fp32;
 *   shared_y [T, H] fp32 or NULL; out [T, H] bf16.  H multiple of 8.
 * A flat_to_row entry outside [0, T*k) (moe_permute writes -1 for a skipped
 * id) contributes nothing and sets GBMOE_ERR_DEVICE in the device status.
 */
int moe_combine(const float* y, const int32_t* flat_to_row, const float* weights,
                const float* shared_y, int T, int k, int H, uint16_t* out,
                gbmoe_stream_t stream);

/*
 * moe_gemm_gateup_act_fp8 / moe_gemm_down_fp8 — the grouped GEMMs with FP8
 * (E4M3) operands on the tensor cores (tcgen05 kind::f8f6f4), one fp32 scale
 * per weight row and per token / routed row (reading of "Stage 4" W8A8FP):
 *   g = (sum_h xq[t,h] wgq[p,i,h]) * sx[t] * sg[p,i], u likewise with wuq, su;
 *   act[r, i] = bf16(f(g, u)), t = row_to_token[r] (row_to_token NULL: t = r,
 *   xq holds the N permuted rows);
 *   y[r, h] = (sum_i aq[r,i] wdq[p,h,i]) * sa[r] * sd[p,h]  (fp32).
 *   xq [T or N, H] codes, sx [T or N]; wgq, wuq [E_phys, I, H] codes, sg, su
 *   [E_phys, I]; aq [N, I] codes, sa [N]; wdq [E_phys, H, I] codes, sd
 *   [E_phys, H].  H % 256 == 0 and I % 128 == 0 (else UNSUPPORTED); code
 *   arrays 16-byte aligned.  Codes and scales come from moe_quantize_fp8_rows.
 */
int moe_gemm_gateup_act_fp8(const uint8_t* xq, const float* sx, const int32_t* row_to_token,
                            int T, const int32_t* offsets, int E_phys, int N, int H, int I,
                            const uint8_t* wgq, const float* sg, const uint8_t* wuq,
                            const float* su, int activation, uint16_t* act,
                            gbmoe_stream_t stream);
int moe_gemm_down_fp8(const uint8_t* aq, const float* sa, const int32_t* offsets, int E_phys,
                      int N, int H, int I, const uint8_t* wdq, const float* sd, float* y,
                      gbmoe_stream_t stream);

/*
 * moe_quantize_fp8_rows — FP8 (OCP E4M3) quantization of bf16 rows for the
 * FP8 expert path ("Stage 4" quantized paths, W8A8FP): per row r
 *   scales[r] = amax_k |x[r, k]| / 448  (1 for an all-zero row),
 *   q[r, k] = e4m3(x[r, k] / scales[r])  (IEEE division, round to nearest
 *   even, saturation to +-448).
 *   x [n, K] bf16, K a multiple of 8 (else GBMOE_ERR_UNSUPPORTED), 16-byte
 *   aligned; q [n, K] uint8 codes, 8-byte aligned; scales [n] fp32.  Used for
 *   weights (one scale per output channel) and for hidden states (per token).
 */
int moe_quantize_fp8_rows(const uint16_t* x, int64_t n, int K, uint8_t* q, float* scales,
                          gbmoe_stream_t stream);

/*
 * MX element formats (OCP Microscaling): E4M3 (one byte per element) or E2M1
 * (FP4: sign, 2 exponent bits with bias 1, 1 mantissa bit; magnitudes 0, 0.5,
 * 1, 1.5, 2, 3, 4, 6; two per byte, the even element in the low nibble).
 */
enum { GBMOE_MX_E4M3 = 0, GBMOE_MX_E2M1 = 1 };

/*
 * moe_quantize_mx_rows — MX block quantization of bf16 rows (reading of the
 * "Stage 4" quantized paths MXFP / W4A8): every row is cut into blocks of 32
 * consecutive elements; block b of row r gets the scale 2^e,
 *   e = floor(log2(amax of the block)) - emax  (emax = 8 for E4M3, 2 for E2M1),
 *   clamped to [-127, 127] (e = 0 for an all-zero block), stored as the byte
 *   scales[r, b] = e + 127 (UE8M0), and each element x becomes the code of
 *   x * 2^-e rounded to nearest even with saturation (448 / 6).
 *   x [n, K] bf16, 16-byte aligned, K a multiple of 32 (else UNSUPPORTED);
 *   q [n, K] (E4M3) or [n, K/2] (E2M1) uint8, 16-byte aligned; scales
 *   [n, K/32] uint8.  fmt: GBMOE_MX_E4M3 or GBMOE_MX_E2M1.
 */
int moe_quantize_mx_rows(const uint16_t* x, int64_t n, int K, int fmt, uint8_t* q,
                         uint8_t* scales, gbmoe_stream_t stream);

/*
 * moe_mx_tile_scales — rearranges MX weight scale bytes from the row-major
 * layout of moe_quantize_mx_rows ([rows, K/32]) into the tiled layout that
 * the MX grouped GEMMs read for their weights (the weight scale arguments of
 * moe_gemm_gateup_act_mx / moe_gemm_down_mx and gbmoe_layer's sf_gate, sf_up,
 * sf_down): for each block of 128 rows rb and K stage ks of 128 elements,
 * 512 contiguous bytes at offset (rb * (K/128) + ks) * 512 whose byte
 * r*16 + j*4 + b is the scale of row rb*128 + 32*j + r for the K block
 * 4*ks + b (r < 32, j < 4, b < 4) -- the order of the tensor-memory columns
 * the block-scaled MMA reads them from, so that a GEMM stage's weight scales
 * arrive as one 512-byte copy per 128-row block.  The output has the size of
 * the input.  A layer's weight scales are converted once, when it is loaded.
 *   sf_rows [rows, K/32] uint8, 4-byte aligned; sf_tiled the same number of
 *   bytes, 16-byte aligned, not overlapping sf_rows.  rows and K multiples of
 *   128 (else UNSUPPORTED).
 */
int moe_mx_tile_scales(const uint8_t* sf_rows, int64_t rows, int K, uint8_t* sf_tiled,
                       gbmoe_stream_t stream);

/*
 * moe_gemm_gateup_act_mx / moe_gemm_down_mx — the grouped GEMMs with MX
 * block-scaled operands on the tensor cores (tcgen05 kind::mxf8f6f4 with
 * block scales): weights in format w_fmt (E4M3: MXFP8; E2M1: W4A8), tokens
 * and activations in MX E4M3.  With dequantized values (code * 2^e of its
 * block):
 *   g = sum_h x[t,h] wg[p,i,h], u likewise (fp32 accumulation),
 *   act = bf16(f(g, u)) quantized to MX E4M3 along I: act_q [N, I] codes and
 *   act_s [N, I/32] scale bytes, the same definition as moe_quantize_mx_rows
 *   (the quantization is fused into the GEMM's epilogue);
 *   y[r, h] = sum_i a[r,i] wd[p,h,i]  (fp32).
 *   xq [T or N, H] codes + xs [T or N, H/32] (t = row_to_token[r], or r with
 *   row_to_token NULL); wgq / wuq [E_phys, I, H or H/2] + sg / su, the
 *   [E_phys, I, H/32] scale bytes in the tiled layout of moe_mx_tile_scales
 *   (rows = E_phys * I, K = H); aq [N, I] + as [N, I/32] (row-major); wdq
 *   [E_phys, H, I or I/2] + sd, [E_phys, H, I/32] tiled (rows = E_phys * H,
 *   K = I).  H % 256 == 0, I % 128 == 0 (else UNSUPPORTED);
 *   code arrays 16-byte aligned (E2M1 weights 32-byte aligned); weight scale
 *   arrays 16-byte aligned, token / activation scale arrays 4-byte aligned.
 */
int moe_gemm_gateup_act_mx(const uint8_t* xq, const uint8_t* xs, const int32_t* row_to_token,
                           int T, const int32_t* offsets, int E_phys, int N, int H, int I,
                           int w_fmt, const uint8_t* wgq, const uint8_t* sg, const uint8_t* wuq,
                           const uint8_t* su, int activation, uint8_t* act_q, uint8_t* act_s,
                           gbmoe_stream_t stream);
int moe_gemm_down_mx(const uint8_t* aq, const uint8_t* as, const int32_t* offsets, int E_phys,
                     int N, int H, int I, int w_fmt, const uint8_t* wdq, const uint8_t* sd,
                     float* y, gbmoe_stream_t stream);

/*
 * moe_latent_tail — the post-MoE tail of a latent MoE on one GPU (the NVIDIA
 * LatentMoERunner page, tier-1 tail "_overlap_allreduce_tail": reduce the
 * routed latent output, RMSNorm, up-project to the hidden size with the
 * replicated weight, add the shared-expert output; with one rank the
 * reductions are identities):
 *   z[t] = bf16(rmsnorm(latent[t]))  (fp32: r = 1/sqrt(sum_l v_l^2 / L + eps),
 *          z_l = bf16((v_l * r) * norm_w[l]); norm_w NULL: z = latent)
 *   out[t, h] = bf16(sum_l z[t, l] * up_proj[h, l] + shared[t, h])  (fp32 accumulate)
 *   latent [T, L] bf16; norm_w [L] bf16 or NULL; eps >= 0; up_proj [Hm, L]
 *   bf16 (row h = output channel); shared [T, Hm] bf16 or NULL; out [T, Hm]
 *   bf16.  L and Hm multiples of 128 (else GBMOE_ERR_UNSUPPORTED); 16-byte
 *   aligned pointers.  ws: device scratch of
 *   gbmoe_latent_tail_workspace_size(T, L, Hm) bytes (GBMOE_ERR_WORKSPACE if
 *   smaller).
 */
size_t gbmoe_latent_tail_workspace_size(int T, int L, int Hm);
int moe_latent_tail(const uint16_t* latent, int T, int L, const uint16_t* norm_w, float eps,
                    const uint16_t* up_proj, int Hm, const uint16_t* shared, uint16_t* out,
                    void* ws, size_t ws_bytes, gbmoe_stream_t stream);

/* Scratch bytes moe_forward needs for any T <= T_max (sized from capacity,
 * not from the runtime token count). */
size_t gbmoe_forward_workspace_size(const gbmoe_layer* L, int T_max);

/*
 * moe_forward — the whole routed layer: route -> permute -> gate/up GEMM +
 * SwiGLU -> down GEMM -> (shared expert) -> combine, all on `stream`.
 *   x [T, H] bf16; input_ids [T] (hash routing) or NULL; out [T, H] bf16.
 *   ids_log, ids_phys [T, top_k] int32, weights [T, top_k] fp32 and
 *   counts [E_phys] int32 are optional outputs (NULL: kept in the workspace).
 *   ws: device scratch of ws_bytes >= gbmoe_forward_workspace_size(L, T).
 */
int moe_forward(const gbmoe_layer* L, const uint16_t* x, int T, const int32_t* input_ids,
                uint16_t* out, int32_t* ids_log, int32_t* ids_phys, float* weights,
                int32_t* counts, void* ws, size_t ws_bytes, gbmoe_stream_t stream);

/* Scratch bytes moe_forward_host needs (moe_forward's plus staging). */
size_t gbmoe_forward_host_workspace_size(const gbmoe_layer* L, int T_max);

/*
 * moe_forward_host — moe_forward with HOST activations: copies x_host [T, H]
 * bf16 (and input_ids_host [T], when hash routing) to the device, runs the
 * layer, and copies out_host [T, H] (and ids_log_host [T, top_k] when not
 * NULL) back, all enqueued on `stream`.  Host buffers should be pinned
 * (cudaHostAlloc) for the copies to overlap; the caller synchronises
 * `stream` before reading the outputs.  Weights stay in device memory.
 */
int moe_forward_host(const gbmoe_layer* L, const uint16_t* x_host, int T,
                     const int32_t* input_ids_host, uint16_t* out_host, int32_t* ids_log_host,
                     void* ws, size_t ws_bytes, gbmoe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GBMOE_H */
