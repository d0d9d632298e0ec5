/*
 * CPU oracle for the routed mixture-of-experts layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously-correct
 * statement of what the GPU library computes.  Only the test-suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the product path
 * never does.  It shares no code, header, table or constant generator with
 * the CUDA library.
 *
 * Source of the method: the vLLM-Ascend "Kimi K3 MoE Forward Insight" page:
 *   - Runner Initialization: routing settings are grouped top-k,
 *     renormalisation, scoring function, correction bias, routed scaling;
 *     expert ids are two-level (logical -> physical through log2phy).
 *   - Stage 2 (Select Experts): softmax / sigmoid / sqrtsoftplus scoring,
 *     hash routing through tid2eid indexed by input_ids, then grouped top-k,
 *     correction bias, top-k, renormalisation, routed scaling.
 *   - Stage 4 (Dispatch, MLP, Combine): map topk_ids through log2phy, sort
 *     tokens by expert and return expert token counts (AllGather mode), grouped
 *     gate/up matmul -> SwiGLU -> grouped down matmul, then restore token order
 *     and apply the routing probabilities.
 *   - Stage 6 (Dynamic EPLB): per-expert token counts accumulated into moe_load.
 *   - Forward Skeleton / shared experts: the always-on shared expert's output is
 *     added to the routed output.
 *
 * Readings where the page is silent (each also listed in the design notes):
 *   R1 router logit l[t,e] = sum_h x[t,h]*Wr[e,h] in fp32 with a pinned order:
 *      32 partial sums, partial j accumulates the h with floor((h mod 64)/2)
 *      = j (h = 2j, 2j+1, 64+2j, 65+2j, ...) ascending with a fused
 *      multiply-add, then the pairwise tree s = 16,8,4,2,1
 *      (p[i] += p[i+s], i < s); an optional router bias is added last.
 *   R2 scores use this file's own elementary functions: exp by Cody-Waite
 *      reduction (ln2 split hi/lo) and the degree-7 Taylor polynomial;
 *      log1p(y) = 2 atanh(y/(2+y)) by its odd power series; sigmoid =
 *      1/(1+exp(-l)); sqrtsoftplus = sqrt(max(l,0) + log1p(exp(-|l|)));
 *      softmax normalises by a sum over experts taken as 32 partials
 *      (partial j takes e = j, j+32, ... ascending) and the same tree.
 *      Division and sqrt are IEEE correctly rounded.
 *   R3 selection score = score + correction bias (when given); the bias never
 *      enters the routing weights.
 *   R4 grouped top-k: E experts in n_group contiguous groups; group score = max
 *      of the group's selection scores, or the sum of its two largest; the
 *      topk_group best groups are kept, the others' experts are excluded.
 *   R5 ties: the lower expert (group) index wins; slots are filled in pick
 *      order (descending selection score).
 *   R6 weights: w_j = (s_j / sum_j s_j) * routed_scaling with the sum taken in
 *      slot order (renormalise on), else s_j * routed_scaling.
 *   R7 hash: ids = tid2eid[input_ids[t]][0..k-1]; weights from the scoring
 *      function at those experts.
 *   R8 replica of logical e for token t: log2phy[e][t mod replica_cnt[e]].
 *   R9 permutation: stable counting sort of the flat index f = t*k + j by
 *      physical expert; row r = offsets[p] + rank of f among equal p.
 *   R17 FP8 experts (W8A8FP): OCP E4M3 codes with one fp32 scale per row
 *      (weights per output channel, activations per token / routed row); see
 *      orc_f32_to_e4m3 and orc_ffn_row_fp8.
 *   R18 MX block-scaled experts (MXFP8 = W8A8 with E4M3 elements, and W4A8
 *      read as E2M1 weights with E4M3 activations): OCP Microscaling blocks
 *      of 32 consecutive elements along the reduction axis, one power-of-two
 *      scale per block; see orc_mx_block_exp and orc_ffn_row_mx.
 *   R16 latent-MoE tail with one rank (NVIDIA LatentMoERunner page, tier 1):
 *      out = bf16(rmsnorm(latent) . up_proj^T + shared); see oracle_latent_tail.
 *   R15 activation branches (named, not defined, by the page): SwiGLU,
 *      clipped SwiGLU-OAI, GeGLU (erf), GeGLU (tanh); see orc_act_value.
 *   R10 rounding points: only the activation is rounded to bf16 inside the
 *      layer (it is the input of the down matmul): act = bf16(silu(g) * u)
 *      with g, u held in fp32; the expert outputs y = act . Wd and the shared
 *      expert's ys stay fp32; out = bf16(sum_j w_j y_j + ys).  Dot products
 *      of the expert MLP accumulate in double (exact products).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread
 * (-ffp-contract=off keeps every a*b+c below as two rounded operations unless
 * written as fmaf).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */
static inline float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static inline uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

uint16_t orc_f32_to_bf16(float f) { return f32_to_bf16(f); }

/* -------------------------------------------------- elementary functions */
/* ln 2 split so that n*LN2_HI is exact for |n| <= 256: LN2_HI is ln 2 rounded
 * to 16 significant bits (45426 / 2^16), LN2_LO = fp32(ln 2 - LN2_HI). */
#define ORC_LN2_HI 0.693145751953125f
#define ORC_LN2_LO 1.428606820309417e-06f
#define ORC_LOG2E 1.44269502162933349609375f /* fp32(1 / ln 2) */

static inline float pow2i(int n) { /* 2^n for -126 <= n <= 127 */
    uint32_t u = (uint32_t)(n + 127) << 23;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* exp(x): Cody-Waite range reduction x = n ln2 + r, |r| <~ ln2/2, then the
 * Taylor polynomial of e^r to degree 7 by Horner's rule, then 2^n applied as
 * two exact power-of-two scalings.  Results below 2^-126 flush to zero. */
float orc_exp(float x) {
    if (x != x) return x;
    if (x > 88.72283935546875f) return INFINITY;
    if (x < -87.33654022216797f) return 0.0f;
    float nf = rintf(x * ORC_LOG2E);
    int n = (int)nf;
    float r = fmaf(-nf, ORC_LN2_HI, x);
    r = fmaf(-nf, ORC_LN2_LO, r);
    float p = 1.0f / 5040.0f;          /* 1/7! */
    p = fmaf(p, r, 1.0f / 720.0f);     /* 1/6! */
    p = fmaf(p, r, 1.0f / 120.0f);     /* 1/5! */
    p = fmaf(p, r, 1.0f / 24.0f);      /* 1/4! */
    p = fmaf(p, r, 1.0f / 6.0f);       /* 1/3! */
    p = fmaf(p, r, 0.5f);              /* 1/2! */
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int n1 = n / 2;
    int n2 = n - n1;
    return (p * pow2i(n1)) * pow2i(n2);
}

/* log(1+y) for 0 <= y <= 1: 2 atanh(z), z = y/(2+y) <= 1/3, with the series
 * z + z^3/3 + ... + z^17/17 (next term below 2e-10 relative). */
float orc_log1p(float y) {
    float z = y / (2.0f + y);
    float w = z * z;
    float q = 1.0f / 17.0f;
    q = fmaf(q, w, 1.0f / 15.0f);
    q = fmaf(q, w, 1.0f / 13.0f);
    q = fmaf(q, w, 1.0f / 11.0f);
    q = fmaf(q, w, 1.0f / 9.0f);
    q = fmaf(q, w, 1.0f / 7.0f);
    q = fmaf(q, w, 1.0f / 5.0f);
    q = fmaf(q, w, 1.0f / 3.0f);
    float zw = z * w;
    float a = fmaf(zw, q, z);
    return 2.0f * a;
}

float orc_sigmoid(float l) {
    float e = orc_exp(-l);
    float d = 1.0f + e;
    return 1.0f / d;
}

float orc_sqrtsoftplus(float l) {
    float a = fabsf(l);
    float sp = fmaxf(l, 0.0f) + orc_log1p(orc_exp(-a));
    return sqrtf(sp);
}

/* ------------------------------------------------------------- routing */
enum { ORC_SOFTMAX = 0, ORC_SIGMOID = 1, ORC_SQRTSOFTPLUS = 2 };
enum { ORC_GROUP_MAX = 0, ORC_GROUP_TOP2SUM = 1 };

typedef struct {
    int E;            /* logical experts */
    int P;            /* physical slots */
    int k;            /* experts per token */
    int n_group;
    int topk_group;
    int scoring;      /* ORC_SOFTMAX / ORC_SIGMOID / ORC_SQRTSOFTPLUS */
    int group_score;  /* ORC_GROUP_MAX / ORC_GROUP_TOP2SUM */
    int renormalize;
    float routed_scaling;
    int use_hash;
} orc_route_cfg;

/* R1: one router logit in the pinned order: 32 partial sums, partial j takes
 * the h with floor((h mod 64) / 2) = j (the pairs 2j, 2j+1 of every 64) in
 * ascending order with fma; then the pairwise tree s = 16, 8, 4, 2, 1. */
float orc_router_logit(const uint16_t* x, const float* w, int H) {
    float p[32];
    for (int j = 0; j < 32; ++j) p[j] = 0.0f;
    for (int h = 0; h < H; ++h) {
        const int j = (h >> 1) & 31;
        p[j] = fmaf(bf16_to_f32(x[h]), w[h], p[j]);
    }
    for (int s = 16; s >= 1; s >>= 1)
        for (int i = 0; i < s; ++i) p[i] = p[i] + p[i + s];
    return p[0];
}

/* a tiny static-striped parallel-for */
typedef struct {
    void (*fn)(void*, int64_t);
    void* ctx;
    int64_t n;
    int tid, nth;
} orc_job;

static void* orc_job_run(void* a) {
    orc_job* j = (orc_job*)a;
    for (int64_t i = j->tid; i < j->n; i += j->nth) j->fn(j->ctx, i);
    return NULL;
}

static void orc_parallel_for(int64_t n, int nthreads, void (*fn)(void*, int64_t), void* ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads == 1 || n < 2) {
        for (int64_t i = 0; i < n; ++i) fn(ctx, i);
        return;
    }
    pthread_t th[256];
    orc_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (orc_job){fn, ctx, n, t, nthreads};
        pthread_create(&th[t], NULL, orc_job_run, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

typedef struct {
    const uint16_t* x;
    const float *w, *bias;
    int H, E;
    float* logits;
} orc_logit_ctx;

static void orc_logit_task(void* c_, int64_t t) {
    orc_logit_ctx* c = (orc_logit_ctx*)c_;
    for (int e = 0; e < c->E; ++e) {
        float l = orc_router_logit(c->x + (size_t)t * c->H, c->w + (size_t)e * c->H, c->H);
        if (c->bias) l = l + c->bias[e];
        c->logits[(size_t)t * c->E + e] = l;
    }
}

/* logits [T, E]; router_bias may be NULL; tokens are independent (threads
 * split them; each logit keeps the R1 order). */
void oracle_router_logits(const uint16_t* x, int T, int H, const float* w_router, int E,
                          const float* router_bias, float* logits, int nthreads) {
    orc_logit_ctx c = {x, w_router, router_bias, H, E, logits};
    orc_parallel_for(T, nthreads, orc_logit_task, &c);
}

/* R2: scores of all E experts of one token. */
void orc_scores(const float* l, int E, int scoring, float* score) {
    if (scoring == ORC_SOFTMAX) {
        float m = l[0];
        for (int e = 1; e < E; ++e) m = fmaxf(m, l[e]);
        float q[32];
        for (int j = 0; j < 32; ++j) q[j] = 0.0f;
        for (int e = 0; e < E; ++e) {
            score[e] = orc_exp(l[e] - m);
            q[e & 31] = q[e & 31] + score[e];
        }
        for (int s = 16; s >= 1; s >>= 1)
            for (int i = 0; i < s; ++i) q[i] = q[i] + q[i + s];
        for (int e = 0; e < E; ++e) score[e] = score[e] / q[0];
    } else if (scoring == ORC_SIGMOID) {
        for (int e = 0; e < E; ++e) score[e] = orc_sigmoid(l[e]);
    } else {
        for (int e = 0; e < E; ++e) score[e] = orc_sqrtsoftplus(l[e]);
    }
}

/* R3-R5: the k chosen logical experts of one token, in pick order. */
int orc_select(const orc_route_cfg* c, const float* score, const float* corr_bias,
               int32_t* chosen) {
    const int E = c->E;
    float* sel = (float*)malloc(sizeof(float) * E);
    unsigned char* allowed = (unsigned char*)malloc(E);
    if (!sel || !allowed) { free(sel); free(allowed); return -1; }
    for (int e = 0; e < E; ++e) {
        sel[e] = corr_bias ? score[e] + corr_bias[e] : score[e];
        allowed[e] = 1;
    }
    if (c->n_group > 1) {
        const int G = c->n_group, gs = E / G;
        float gscore[1024];
        unsigned char gkeep[1024];
        for (int g = 0; g < G; ++g) {
            float best = -INFINITY, second = -INFINITY;
            for (int e = g * gs; e < (g + 1) * gs; ++e) {
                if (sel[e] > best) { second = best; best = sel[e]; }
                else if (sel[e] > second) second = sel[e];
            }
            gscore[g] = (c->group_score == ORC_GROUP_TOP2SUM && gs > 1) ? best + second : best;
            gkeep[g] = 0;
        }
        for (int r = 0; r < c->topk_group; ++r) {
            int bg = -1;
            for (int g = 0; g < G; ++g)
                if (!gkeep[g] && (bg < 0 || gscore[g] > gscore[bg])) bg = g;
            gkeep[bg] = 1;
        }
        for (int e = 0; e < E; ++e) allowed[e] = gkeep[e / gs];
    }
    for (int j = 0; j < c->k; ++j) {
        int be = -1;
        for (int e = 0; e < E; ++e)
            if (allowed[e] && (be < 0 || sel[e] > sel[be])) be = e;
        chosen[j] = be;
        allowed[be] = 0;
    }
    free(sel);
    free(allowed);
    return 0;
}

/*
 * Routing of T tokens from their logits [T, E].
 * corr_bias [E] or NULL; input_ids [T] + tid2eid [V, k] when c->use_hash;
 * log2phy [E, R] + replica_cnt [E] or NULL (identity placement).
 * Outputs ids_log / ids_phys int32 [T, k], weights fp32 [T, k].
 * Returns 0, or -2 for an out-of-range token id, -3 for an out-of-range
 * table entry, -4 for a bad placement table.
 */
int oracle_route(const orc_route_cfg* c, const float* logits, int T,
                 const float* corr_bias, const int32_t* input_ids, const int32_t* tid2eid,
                 int64_t V, const int32_t* log2phy, const int32_t* replica_cnt, int R,
                 int32_t* ids_log, int32_t* ids_phys, float* weights) {
    const int E = c->E, k = c->k;
    float* score = (float*)malloc(sizeof(float) * E);
    if (!score) return -1;
    int rc = 0;
    for (int t = 0; t < T && rc == 0; ++t) {
        const float* l = logits + (size_t)t * E;
        orc_scores(l, E, c->scoring, score);
        int32_t* ch = ids_log + (size_t)t * k;
        if (c->use_hash) {
            int64_t v = input_ids[t];
            if (v < 0 || v >= V) { rc = -2; break; }
            for (int j = 0; j < k; ++j) {
                int32_t e = tid2eid[v * k + j];
                if (e < 0 || e >= E) { rc = -3; break; }
                ch[j] = e;
            }
            if (rc) break;
        } else {
            if (orc_select(c, score, corr_bias, ch)) { rc = -1; break; }
        }
        float* w = weights + (size_t)t * k;
        if (c->renormalize) {
            float sum = 0.0f;
            for (int j = 0; j < k; ++j) sum = sum + score[ch[j]];
            for (int j = 0; j < k; ++j) w[j] = (score[ch[j]] / sum) * c->routed_scaling;
        } else {
            for (int j = 0; j < k; ++j) w[j] = score[ch[j]] * c->routed_scaling;
        }
        for (int j = 0; j < k; ++j) {
            int32_t e = ch[j], p = e;
            if (log2phy) {
                int32_t n = replica_cnt[e];
                if (n < 1 || n > R) { rc = -4; break; }
                p = log2phy[(size_t)e * R + (t % n)];
                if (p < 0 || p >= c->P) { rc = -4; break; }
            }
            ids_phys[(size_t)t * k + j] = p;
        }
    }
    free(score);
    return rc;
}

/* -------------------------------------------------- counts, permutation */
void oracle_expert_counts(const int32_t* ids_phys, int T, int k, int P, int32_t* counts,
                          int accumulate) {
    if (!accumulate)
        for (int p = 0; p < P; ++p) counts[p] = 0;
    for (int64_t f = 0; f < (int64_t)T * k; ++f) counts[ids_phys[f]] += 1;
}

/* R9: stable counting sort; offsets has P+1 entries. */
void oracle_permute(const int32_t* ids_phys, int T, int k, int P, int32_t* counts,
                    int32_t* offsets, int32_t* row_to_token, int32_t* flat_to_row) {
    const int64_t N = (int64_t)T * k;
    oracle_expert_counts(ids_phys, T, k, P, counts, 0);
    offsets[0] = 0;
    for (int p = 0; p < P; ++p) offsets[p + 1] = offsets[p] + counts[p];
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (P > 0 ? P : 1));
    for (int p = 0; p < P; ++p) cursor[p] = offsets[p];
    for (int64_t f = 0; f < N; ++f) {
        int32_t r = cursor[ids_phys[f]]++;
        row_to_token[r] = (int32_t)(f / k);
        flat_to_row[f] = r;
    }
    free(cursor);
}

/* ----------------------------------------------------------- expert MLP */
/* R15: the gated activations of the gate/up output ("Stage 4" activation
 * branches; the pages name them, the formulas are the usual definitions):
 *   0 SwiGLU:             silu(g) * u,  silu(g) = g / (1 + e^-g)
 *   1 clipped SwiGLU-OAI: g' = min(g, 7), u' = clamp(u, -7, 7),
 *                         g' * sigmoid(1.702 g') * (u' + 1)
 *   2 GeGLU (erf):        0.5 g (1 + erf(g / sqrt 2)) * u
 *   3 GeGLU (tanh):       0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) * u
 * in double on the fp32 values of g and u. */
double orc_act_value(int act, double g, double u) {
    switch (act) {
        case 1: {
            const double gc = g < 7.0 ? g : 7.0;
            const double uc = u < -7.0 ? -7.0 : (u > 7.0 ? 7.0 : u);
            return gc / (1.0 + exp(-1.702 * gc)) * (uc + 1.0);
        }
        case 2:
            return 0.5 * g * (1.0 + erf(g / sqrt(2.0))) * u;
        case 3: {
            const double c = sqrt(2.0 / 3.14159265358979323846);
            return 0.5 * g * (1.0 + tanh(c * (g + 0.044715 * g * g * g))) * u;
        }
        default:
            return g / (1.0 + exp(-g)) * u;
    }
}

/* One row through one gated expert MLP (R10, R15).
 * wg, wu: [I, H]; wd: [H, I]; act_out [I] as bf16 bits, y_out [H] fp32. */
void orc_ffn_row(const uint16_t* x, const uint16_t* wg, const uint16_t* wu,
                 const uint16_t* wd, int H, int I, int act, uint16_t* act_out, float* y_out) {
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        const uint16_t* rg = wg + (size_t)i * H;
        const uint16_t* ru = wu + (size_t)i * H;
        for (int h = 0; h < H; ++h) {
            double xv = bf16_to_f32(x[h]);
            g += xv * bf16_to_f32(rg[h]);
            u += xv * bf16_to_f32(ru[h]);
        }
        double gf = (float)g, uf = (float)u;
        act_out[i] = f32_to_bf16((float)orc_act_value(act, gf, uf));
    }
    for (int h = 0; h < H; ++h) {
        double acc = 0.0;
        const uint16_t* rd = wd + (size_t)h * I;
        for (int i = 0; i < I; ++i) acc += (double)bf16_to_f32(act_out[i]) * bf16_to_f32(rd[i]);
        y_out[h] = (float)acc;
    }
}

typedef struct {
    const uint16_t *x, *wg, *wu, *wd;
    const int32_t *row_to_token, *row_expert;
    int H, I, act_kind;
    uint16_t* act;
    float* y;
} orc_ffn_ctx;

static void orc_ffn_task(void* c_, int64_t r) {
    orc_ffn_ctx* c = (orc_ffn_ctx*)c_;
    int64_t t = c->row_to_token ? c->row_to_token[r] : r;
    int64_t p = c->row_expert ? c->row_expert[r] : 0;
    const size_t HI = (size_t)c->H * c->I;
    orc_ffn_row(c->x + (size_t)t * c->H, c->wg + p * HI, c->wu + p * HI, c->wd + p * HI, c->H,
                c->I, c->act_kind, c->act + (size_t)r * c->I, c->y + (size_t)r * c->H);
}

/* Rows of n inputs through one expert: act [n, I] bf16, y [n, H] fp32. */
void oracle_expert_ffn_rows(const uint16_t* x, int64_t n, int H, int I, const uint16_t* wg,
                            const uint16_t* wu, const uint16_t* wd, int act_kind, uint16_t* act,
                            float* y, int nthreads) {
    orc_ffn_ctx c = {x, wg, wu, wd, NULL, NULL, H, I, act_kind, act, y};
    orc_parallel_for(n, nthreads, orc_ffn_task, &c);
}

/* Grouped MLP over the permuted rows: row r belongs to the expert p with
 * offsets[p] <= r < offsets[p+1] and carries token row_to_token[r].
 * wg/wu [P, I, H], wd [P, H, I]; act [N, I] bf16, y [N, H] fp32. */
void oracle_ffn_grouped(const uint16_t* x, const int32_t* row_to_token, const int32_t* offsets,
                        int P, int H, int I, const uint16_t* wg, const uint16_t* wu,
                        const uint16_t* wd, int act_kind, uint16_t* act, float* y, int nthreads) {
    int64_t N = offsets[P];
    int32_t* row_expert = (int32_t*)malloc(sizeof(int32_t) * (N > 0 ? N : 1));
    for (int p = 0; p < P; ++p)
        for (int32_t r = offsets[p]; r < offsets[p + 1]; ++r) row_expert[r] = p;
    orc_ffn_ctx c = {x, wg, wu, wd, row_to_token, row_expert, H, I, act_kind, act, y};
    orc_parallel_for(N, nthreads, orc_ffn_task, &c);
    free(row_expert);
}

/* Restore token order and apply the routing weights (R10):
 * out[t,h] = bf16(sum_j w[t,j] * y[flat_to_row[t*k+j], h] + ys[t,h]); y, ys fp32. */
void oracle_combine(const float* y, const int32_t* flat_to_row, const float* weights,
                    const float* ys, int T, int k, int H, uint16_t* out) {
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                int64_t r = flat_to_row[(int64_t)t * k + j];
                acc += (double)weights[(int64_t)t * k + j] * (double)y[r * H + h];
            }
            if (ys) acc += (double)ys[(size_t)t * H + h];
            out[(size_t)t * H + h] = f32_to_bf16((float)acc);
        }
}

/*
 * The whole layer, stage by stage.  Weights are physical-slot stacks
 * (wg/wu [P, I, H], wd [P, H, I]); shared-expert weights may be NULL.
 * logits [T, E] are computed here when w_router is given, else taken as input.
 * Scratch outputs: offsets [P+1], row_to_token / flat_to_row [T*k],
 * act [T*k, I] bf16, y [T*k, H] fp32; ys [T, H] fp32 when a shared expert is
 * present.
 */
int oracle_moe_forward(const orc_route_cfg* c, const uint16_t* x, int T, int H, int I,
                       const float* w_router, const float* router_bias, float* logits,
                       const float* corr_bias, const int32_t* input_ids,
                       const int32_t* tid2eid, int64_t V, const int32_t* log2phy,
                       const int32_t* replica_cnt, int R, const uint16_t* wg,
                       const uint16_t* wu, const uint16_t* wd, int act_kind, int I_shared,
                       const uint16_t* wg_s, const uint16_t* wu_s, const uint16_t* wd_s,
                       int32_t* ids_log, int32_t* ids_phys, float* weights, int32_t* counts,
                       int32_t* offsets, int32_t* row_to_token, int32_t* flat_to_row,
                       uint16_t* act, float* y, uint16_t* act_s, float* ys,
                       uint16_t* out, int nthreads) {
    if (w_router) oracle_router_logits(x, T, H, w_router, c->E, router_bias, logits, nthreads);
    int rc = oracle_route(c, logits, T, corr_bias, input_ids, tid2eid, V, log2phy, replica_cnt,
                          R, ids_log, ids_phys, weights);
    if (rc) return rc;
    oracle_permute(ids_phys, T, c->k, c->P, counts, offsets, row_to_token, flat_to_row);
    oracle_ffn_grouped(x, row_to_token, offsets, c->P, H, I, wg, wu, wd, act_kind, act, y,
                       nthreads);
    const float* ysp = NULL;
    if (wg_s) {
        oracle_expert_ffn_rows(x, T, H, I_shared, wg_s, wu_s, wd_s, act_kind, act_s, ys,
                               nthreads);
        ysp = ys;
    }
    oracle_combine(y, flat_to_row, weights, ysp, T, c->k, H, out);
    return 0;
}

/* ------------------------------------------------------- latent MoE tail */
/*
 * R16: the post-MoE tail of a latent MoE on one GPU (the NVIDIA LatentMoERunner
 * page, tier 1 "_overlap_allreduce_tail" with tensor parallelism 1, where the
 * all-reduces are identities): out = bf16(norm(latent) . up_proj^T + shared).
 * norm is the standard RMSNorm with weight w and epsilon eps, taken in fp32 in
 * a pinned order and rounded to bf16 (the bf16 input of the up-projection):
 *   s = sum over l of v_l^2 as 32 partial sums (partial j takes l = j, j+32,
 *       ... ascending with fma) and the pairwise tree s = 16, 8, 4, 2, 1;
 *   r = 1 / sqrt(s / L + eps)   (IEEE division and square root);
 *   z_l = bf16((v_l * r) * w_l).
 * Without a norm weight z = latent.  The up-projection accumulates in double;
 * shared may be NULL.
 */
void oracle_rmsnorm_row(const uint16_t* v, int L, const uint16_t* w, float eps, uint16_t* z) {
    float p[32];
    for (int j = 0; j < 32; ++j) p[j] = 0.0f;
    for (int l = 0; l < L; ++l) {
        const float x = bf16_to_f32(v[l]);
        p[l & 31] = fmaf(x, x, p[l & 31]);
    }
    for (int s = 16; s >= 1; s >>= 1)
        for (int i = 0; i < s; ++i) p[i] = p[i] + p[i + s];
    const float r = 1.0f / sqrtf(p[0] / (float)L + eps);
    for (int l = 0; l < L; ++l) z[l] = f32_to_bf16((bf16_to_f32(v[l]) * r) * bf16_to_f32(w[l]));
}

typedef struct {
    const uint16_t *latent, *w, *up, *shared;
    int L, Hm;
    float eps;
    uint16_t* out;
} orc_tail_ctx;

static void orc_tail_task(void* c_, int64_t t) {
    orc_tail_ctx* c = (orc_tail_ctx*)c_;
    const uint16_t* v = c->latent + (size_t)t * c->L;
    uint16_t* z = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)c->L);
    if (!z) return;
    if (c->w)
        oracle_rmsnorm_row(v, c->L, c->w, c->eps, z);
    else
        memcpy(z, v, sizeof(uint16_t) * (size_t)c->L);
    for (int h = 0; h < c->Hm; ++h) {
        double acc = 0.0;
        const uint16_t* u = c->up + (size_t)h * c->L;
        for (int l = 0; l < c->L; ++l) acc += (double)bf16_to_f32(z[l]) * bf16_to_f32(u[l]);
        const float yf = (float)acc;
        const float sh = c->shared ? bf16_to_f32(c->shared[(size_t)t * c->Hm + h]) : 0.0f;
        c->out[(size_t)t * c->Hm + h] = f32_to_bf16(yf + sh);
    }
    free(z);
}

/* latent [T, L], w [L] or NULL, up [Hm, L], shared [T, Hm] or NULL -> out [T, Hm]. */
void oracle_latent_tail(const uint16_t* latent, int T, int L, const uint16_t* w, float eps,
                        const uint16_t* up, int Hm, const uint16_t* shared, uint16_t* out,
                        int nthreads) {
    orc_tail_ctx c = {latent, w, up, shared, L, Hm, eps, out};
    orc_parallel_for(T, nthreads, orc_tail_task, &c);
}

/* ------------------------------------------------------------ FP8 experts */
/*
 * R17: FP8 experts ("Stage 4": quantized paths include W8A8FP; the page gives
 * no scale layout).  OCP FP8 E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa
 * bits, no infinities, largest finite 448, subnormals down to 2^-9.  A row is
 * quantized with one fp32 scale s = amax / 448 (s = 1 for an all-zero row):
 * q = e4m3(x / s) with IEEE division, round to nearest even and saturation
 * to +-448.  Weights: one scale per output channel (row); activations: one
 * scale per token / routed row, computed when they are produced.
 */
static double orc_ldexp(double m, int e) { return ldexp(m, e); }

/* fp32 -> E4M3 code, round to nearest even, saturating to +-448 (NaN -> 0x7f). */
uint8_t orc_f32_to_e4m3(float xf) {
    const double x = (double)xf;
    if (x != x) return 0x7f;
    const uint8_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7e);      /* saturate: 1.75 * 2^8 */
    /* the representable magnitudes: subnormal k * 2^-9 (k < 8), normal
     * (8 + m) * 2^(e-10) for e = 1..15, m = 0..7; round a to the nearest
     * multiple of the spacing of its binade, ties to even */
    int e;
    frexp(a, &e);                                          /* a = f * 2^e, 0.5 <= f < 1 */
    int be = e - 1 + 7;                                    /* biased exponent of a */
    if (be < 1) be = 1;                                    /* subnormal binade: spacing 2^-9 */
    const double spacing = orc_ldexp(1.0, be - 7 - 3);
    double k = a / spacing;                                /* exact (power-of-two division) */
    double kr = floor(k);
    const double rem = k - kr;
    if (rem > 0.5 || (rem == 0.5 && fmod(kr, 2.0) == 1.0)) kr += 1.0;
    /* kr * spacing is the rounded magnitude; re-encode (may carry into the next binade) */
    const double r = kr * spacing;
    if (r >= 448.0) return (uint8_t)(sign | 0x7e);
    if (r == 0.0) return sign;
    int e2;
    frexp(r, &e2);
    int bexp = e2 - 1 + 7;
    if (bexp < 1) {                                        /* subnormal: r = mant * 2^-9 */
        const int mant = (int)(r / orc_ldexp(1.0, -9));
        return (uint8_t)(sign | mant);
    }
    const int mant = (int)(r / orc_ldexp(1.0, bexp - 7 - 3)) - 8;
    return (uint8_t)(sign | (bexp << 3) | mant);
}

/* E4M3 code -> value (exact in fp32). */
float orc_e4m3_to_f32(uint8_t c) {
    const int s = c >> 7, be = (c >> 3) & 15, m = c & 7;
    if (be == 15 && m == 7) return NAN;
    const double v = be == 0 ? m * orc_ldexp(1.0, -9) : (8 + m) * orc_ldexp(1.0, be - 10);
    return (float)(s ? -v : v);
}

/* One row of n values (bf16 bits, or fp32 when xf != NULL) -> codes + scale. */
float oracle_quantize_row(const uint16_t* xb, const float* xf, int n, uint8_t* q) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        const float v = fabsf(xf ? xf[i] : bf16_to_f32(xb[i]));
        if (v > amax) amax = v;
    }
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int i = 0; i < n; ++i) q[i] = orc_f32_to_e4m3((xf ? xf[i] : bf16_to_f32(xb[i])) / s);
    return s;
}

/* rows [n, K] bf16 -> codes [n, K] + scales [n] */
void oracle_quantize_rows(const uint16_t* x, int64_t n, int K, uint8_t* q, float* s) {
    for (int64_t r = 0; r < n; ++r) s[r] = oracle_quantize_row(x + r * K, NULL, K, q + r * K);
}

/*
 * One routed row through one FP8 expert: xq [H] codes with scale sx; wgq, wuq
 * [I, H] codes with per-row scales sg, su [I]; wdq [H, I] codes with sd [H].
 * g = (sum q_x q_g) sx sg, u likewise (double), act = bf16(f(g, u)) (R15);
 * act is quantized per row (aq, sa) and y = (sum q_a q_d) sa sd in fp32.
 */
void orc_ffn_row_fp8(const uint8_t* xq, float sx, const uint8_t* wgq, const float* sg,
                     const uint8_t* wuq, const float* su, const uint8_t* wdq, const float* sd,
                     int H, int I, int act, uint16_t* act_out, float* y_out) {
    float* actf = (float*)malloc(sizeof(float) * (size_t)I);
    uint8_t* aq = (uint8_t*)malloc((size_t)I);
    if (!actf || !aq) { free(actf); free(aq); return; }
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        const uint8_t* rg = wgq + (size_t)i * H;
        const uint8_t* ru = wuq + (size_t)i * H;
        for (int h = 0; h < H; ++h) {
            const double xv = orc_e4m3_to_f32(xq[h]);
            g += xv * orc_e4m3_to_f32(rg[h]);
            u += xv * orc_e4m3_to_f32(ru[h]);
        }
        const double gf = (float)((float)g * sx * sg[i]), uf = (float)((float)u * sx * su[i]);
        act_out[i] = f32_to_bf16((float)orc_act_value(act, gf, uf));
        actf[i] = bf16_to_f32(act_out[i]);
    }
    const float sa = oracle_quantize_row(NULL, actf, I, aq);
    for (int h = 0; h < H; ++h) {
        double acc = 0.0;
        const uint8_t* rd = wdq + (size_t)h * I;
        for (int i = 0; i < I; ++i) acc += (double)orc_e4m3_to_f32(aq[i]) * orc_e4m3_to_f32(rd[i]);
        y_out[h] = (float)acc * sa * sd[h];
    }
    free(actf);
    free(aq);
}

typedef struct {
    const uint8_t* xq;
    const float* sx;
    const uint8_t *wg, *wu, *wd;
    const float *sg, *su, *sd;
    const int32_t *row_to_token, *row_expert;
    int H, I, act_kind;
    uint16_t* act;
    float* y;
} orc_ffn8_ctx;

static void orc_ffn8_task(void* c_, int64_t r) {
    orc_ffn8_ctx* c = (orc_ffn8_ctx*)c_;
    const int64_t t = c->row_to_token[r];
    const int64_t p = c->row_expert[r];
    const size_t HI = (size_t)c->H * c->I;
    orc_ffn_row_fp8(c->xq + (size_t)t * c->H, c->sx[t], c->wg + p * HI, c->sg + p * c->I,
                    c->wu + p * HI, c->su + p * c->I, c->wd + p * HI, c->sd + p * c->H, c->H,
                    c->I, c->act_kind, c->act + (size_t)r * c->I, c->y + (size_t)r * c->H);
}

/* Grouped FP8 MLP over the permuted rows (x quantized per token: xq [T, H], sx [T]);
 * weight codes [P, I, H] / [P, H, I] with per-row scales [P, I] / [P, H]. */
void oracle_ffn_grouped_fp8(const uint8_t* xq, const float* sx, const int32_t* row_to_token,
                            const int32_t* offsets, int P, int H, int I, const uint8_t* wg,
                            const float* sg, const uint8_t* wu, const float* su,
                            const uint8_t* wd, const float* sd, int act_kind, uint16_t* act,
                            float* y, int nthreads) {
    int64_t N = offsets[P];
    int32_t* row_expert = (int32_t*)malloc(sizeof(int32_t) * (N > 0 ? N : 1));
    for (int p = 0; p < P; ++p)
        for (int32_t r = offsets[p]; r < offsets[p + 1]; ++r) row_expert[r] = p;
    orc_ffn8_ctx c = {xq, sx, wg, wu, wd, sg, su, sd, row_to_token, row_expert, H, I, act_kind,
                      act, y};
    orc_parallel_for(N, nthreads, orc_ffn8_task, &c);
    free(row_expert);
}

/* ------------------------------------------------------ MX block scales */
/*
 * R18: MX experts ("Stage 4": quantized paths include MXFP variants and W4A8;
 * the page gives no formats).  Read as the OCP Microscaling (MX) format:
 * every row is cut into blocks of 32 consecutive elements along the
 * reduction axis (H for x, W_gate, W_up; I for the activations and W_down);
 * a block shares one scale X = 2^e stored as an unsigned exponent byte
 * (UE8M0, byte = e + 127); e = floor(log2(amax)) - emax, emax being the
 * exponent of the element format's largest binade (8 for E4M3, 2 for E2M1),
 * clamped to [-127, 127]; an all-zero block takes byte 127.  Each element is
 * v / X rounded to nearest even in the element format, saturating to its
 * largest magnitude (448, 6).  E2M1 (FP4): sign, 2 exponent bits (bias 1),
 * 1 mantissa bit, magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; two codes per byte,
 * the even element in the low nibble.  MXFP8 = E4M3 weights and
 * activations; W4A8 = E2M1 weights and E4M3 activations.
 */
#define ORC_MX_BLOCK 32
#define ORC_FMT_E4M3 0
#define ORC_FMT_E2M1 1

static const double orc_e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* fp32 -> E2M1 code: nearest representable magnitude, ties to the even code
 * (mantissa bit 0), saturating to 6. */
uint8_t orc_f32_to_e2m1(float xf) {
    const double x = (double)xf;
    const uint8_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x8 : 0x0;
    const double a = fabs(x);
    if (!(a < 6.0)) return (uint8_t)(sign | 7);     /* also NaN: no NaN code */
    int k = 0;
    while (k < 7 && orc_e2m1_mag[k + 1] <= a) ++k;   /* mag[k] <= a < mag[k+1] */
    if (a > orc_e2m1_mag[k]) {
        const double mid = 0.5 * (orc_e2m1_mag[k] + orc_e2m1_mag[k + 1]);
        if (a > mid || (a == mid && (k & 1))) ++k;
    }
    return (uint8_t)(sign | k);
}

float orc_e2m1_to_f32(uint8_t c) {
    const double v = orc_e2m1_mag[c & 7];
    return (float)((c & 8) ? -v : v);
}

/* the block exponent e of a block with largest magnitude amax */
int orc_mx_block_exp(float amax, int fmt) {
    if (!(amax > 0.0f)) return 0;
    int e2;
    frexp((double)amax, &e2);                        /* amax = f 2^e2, 0.5 <= f < 1 */
    int e = (e2 - 1) - (fmt == ORC_FMT_E2M1 ? 2 : 8);
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* element k of an MX row as a double: codes (bytes, or packed nibbles) and
 * block scale bytes */
static double orc_mx_value(const uint8_t* q, const uint8_t* sc, int k, int fmt) {
    const double x = orc_ldexp(1.0, (int)sc[k / ORC_MX_BLOCK] - 127);
    if (fmt == ORC_FMT_E2M1) return orc_e2m1_to_f32((uint8_t)((q[k / 2] >> (4 * (k & 1))) & 15)) * x;
    return orc_e4m3_to_f32(q[k]) * x;
}

/* one row of K values (bf16 bits, or fp32 when xf != NULL) -> MX codes + block scales */
void oracle_mx_quantize_row(const uint16_t* xb, const float* xf, int K, int fmt, uint8_t* q,
                            uint8_t* sc) {
    if (fmt == ORC_FMT_E2M1) memset(q, 0, (size_t)K / 2);
    for (int b = 0; b < K / ORC_MX_BLOCK; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < ORC_MX_BLOCK; ++i) {
            const int k = b * ORC_MX_BLOCK + i;
            const float v = fabsf(xf ? xf[k] : bf16_to_f32(xb[k]));
            if (v > amax) amax = v;
        }
        const int e = orc_mx_block_exp(amax, fmt);
        sc[b] = (uint8_t)(e + 127);
        for (int i = 0; i < ORC_MX_BLOCK; ++i) {
            const int k = b * ORC_MX_BLOCK + i;
            const double v = (double)(xf ? xf[k] : bf16_to_f32(xb[k]));
            const float r = (float)orc_ldexp(v, -e);     /* exact: a power-of-two scaling */
            if (fmt == ORC_FMT_E2M1)
                q[k / 2] |= (uint8_t)(orc_f32_to_e2m1(r) << (4 * (k & 1)));
            else
                q[k] = orc_f32_to_e4m3(r);
        }
    }
}

/* rows [n, K] bf16 -> codes [n, K] (E4M3) or [n, K/2] (E2M1) + scales [n, K/32] */
void oracle_mx_quantize_rows(const uint16_t* x, int64_t n, int K, int fmt, uint8_t* q,
                             uint8_t* sc) {
    const size_t qrow = fmt == ORC_FMT_E2M1 ? (size_t)K / 2 : (size_t)K;
    for (int64_t r = 0; r < n; ++r)
        oracle_mx_quantize_row(x + r * K, NULL, K, fmt, q + r * qrow, sc + r * (K / ORC_MX_BLOCK));
}

/*
 * One routed row through one MX expert: x codes (E4M3) [H] with block scales
 * [H/32]; W_gate / W_up [I, H] and W_down [H, I] in format wfmt with their
 * block scales.  g = sum_h x_h w_h over the dequantized values (each
 * product exact in double), rounded once to fp32; act = bf16(f(g, u)) (R15);
 * the activation row is quantized to MX E4M3 (aq, as) and y = sum_i a_i d_i
 * over the dequantized values, rounded once to fp32.
 */
void orc_ffn_row_mx(const uint8_t* xq, const uint8_t* xs, const uint8_t* wgq, const uint8_t* sg,
                    const uint8_t* wuq, const uint8_t* su, const uint8_t* wdq, const uint8_t* sd,
                    int wfmt, int H, int I, int act, uint16_t* act_out, uint8_t* aq,
                    uint8_t* as, float* y_out) {
    const size_t wrow_h = wfmt == ORC_FMT_E2M1 ? (size_t)H / 2 : (size_t)H;
    const size_t wrow_i = wfmt == ORC_FMT_E2M1 ? (size_t)I / 2 : (size_t)I;
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    float* actf = (float*)malloc(sizeof(float) * (size_t)I);
    if (!xv || !actf) { free(xv); free(actf); return; }
    for (int h = 0; h < H; ++h) xv[h] = orc_mx_value(xq, xs, h, ORC_FMT_E4M3);
    for (int i = 0; i < I; ++i) {
        const uint8_t *rg = wgq + (size_t)i * wrow_h, *ru = wuq + (size_t)i * wrow_h;
        const uint8_t *rsg = sg + (size_t)i * (H / ORC_MX_BLOCK), *rsu = su + (size_t)i * (H / ORC_MX_BLOCK);
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            g += xv[h] * orc_mx_value(rg, rsg, h, wfmt);
            u += xv[h] * orc_mx_value(ru, rsu, h, wfmt);
        }
        act_out[i] = f32_to_bf16((float)orc_act_value(act, (float)g, (float)u));
        actf[i] = bf16_to_f32(act_out[i]);
    }
    oracle_mx_quantize_row(NULL, actf, I, ORC_FMT_E4M3, aq, as);
    for (int h = 0; h < H; ++h) {
        const uint8_t* rd = wdq + (size_t)h * wrow_i;
        const uint8_t* rsd = sd + (size_t)h * (I / ORC_MX_BLOCK);
        double acc = 0.0;
        for (int i = 0; i < I; ++i)
            acc += orc_mx_value(aq, as, i, ORC_FMT_E4M3) * orc_mx_value(rd, rsd, i, wfmt);
        y_out[h] = (float)acc;
    }
    free(xv);
    free(actf);
}

typedef struct {
    const uint8_t *xq, *xs, *wg, *sg, *wu, *su, *wd, *sd;
    const int32_t *row_to_token, *row_expert;
    int wfmt, H, I, act_kind;
    uint16_t* act;
    uint8_t *aq, *as;
    float* y;
} orc_ffnmx_ctx;

static void orc_ffnmx_task(void* c_, int64_t r) {
    orc_ffnmx_ctx* c = (orc_ffnmx_ctx*)c_;
    const int64_t t = c->row_to_token[r];
    const int64_t p = c->row_expert[r];
    const int H = c->H, I = c->I;
    const size_t wq = (size_t)H * I / (c->wfmt == ORC_FMT_E2M1 ? 2 : 1);
    const size_t ws = (size_t)H * I / ORC_MX_BLOCK;
    orc_ffn_row_mx(c->xq + (size_t)t * H, c->xs + (size_t)t * (H / ORC_MX_BLOCK), c->wg + p * wq,
                   c->sg + p * ws, c->wu + p * wq, c->su + p * ws, c->wd + p * wq, c->sd + p * ws,
                   c->wfmt, H, I, c->act_kind, c->act + (size_t)r * I, c->aq + (size_t)r * I,
                   c->as + (size_t)r * (I / ORC_MX_BLOCK), c->y + (size_t)r * H);
}

/* Grouped MX MLP over the permuted rows: x codes [T, H] E4M3 + scales
 * [T, H/32]; weights in format wfmt: codes [P, I, H(/2)] / [P, H, I(/2)],
 * scales [P, I, H/32] / [P, H, I/32].  Outputs act bf16 [N, I], its MX E4M3
 * codes [N, I] and scales [N, I/32], and y fp32 [N, H]. */
void oracle_ffn_grouped_mx(const uint8_t* xq, const uint8_t* xs, const int32_t* row_to_token,
                           const int32_t* offsets, int P, int H, int I, int wfmt,
                           const uint8_t* wg, const uint8_t* sg, const uint8_t* wu,
                           const uint8_t* su, const uint8_t* wd, const uint8_t* sd, int act_kind,
                           uint16_t* act, uint8_t* aq, uint8_t* as, float* y, int nthreads) {
    int64_t N = offsets[P];
    int32_t* row_expert = (int32_t*)malloc(sizeof(int32_t) * (N > 0 ? N : 1));
    for (int p = 0; p < P; ++p)
        for (int32_t r = offsets[p]; r < offsets[p + 1]; ++r) row_expert[r] = p;
    orc_ffnmx_ctx c = {xq, xs, wg, sg, wu, su, wd, sd, row_to_token, row_expert, wfmt, H, I,
                       act_kind, act, aq, as, y};
    orc_parallel_for(N, nthreads, orc_ffnmx_task, &c);
    free(row_expert);
}
