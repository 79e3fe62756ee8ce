/*
 * oracle.c -- plain, slow CPU oracle for the MoE routing front-end.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file; only the tests, the package smoke check and the CPU-baseline leg
 * of the benchmark do. It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Every step is the plain definition, evaluated in fp64, in the order the
 * pages give it:
 *
 *  1. gate GEMM: z[t,e] = sum_h x[t,h] * W[e,h] (+ bias[e]), summed in double.
 *     "[AMD] One-launch small-M MoE router for Qwen3.5 on gfx950",
 *     Modifications (one launch computes the 513 gate rows: 512 routed plus
 *     the shared-expert gate, read in place) and Accuracy Tests (the
 *     fp64-then-bf16 reference).
 *  2. the routed logits are rounded to bf16 (round to nearest even) straight
 *     from the double, with no intermediate fp32 rounding. Same page,
 *     Modifications (the routed logits, and only those, go through a bf16
 *     rounding before the selection) and Accuracy Tests.
 *  3. top-k over the rounded logits; equal values go to the lowest expert id,
 *     and slots are ordered by (value desc, id asc), the order k successive
 *     argmax passes produce. Same page, Motivation and Modifications.
 *  4. softmax over the E experts followed by renormalising the k selected
 *     weights, which equals a softmax over the selected logits (the full
 *     denominator cancels). Same page, Motivation.
 *  5. shared slot k = (E, scale * sigmoid(shared logit)); the shared logit is
 *     the unrounded fp64 dot (only the routed logits are rounded). Same page,
 *     Modifications; expert id E = 512 as the shared expert also in the
 *     vLLM "--monokernel decode" pull request (#60833), Details (Launches).
 *  6. moe_align_block_size: per-expert counts over all slots, padded prefix
 *     sum off[e+1] = off[e] + ceil(cnt[e]/A)*A, num_tokens_post_padded =
 *     off[E_al], stable scatter of flat slot indices, sentinel padding and one
 *     expert id per block. "[ROCm][Kernel] W4A16 MoE prefill: M-aware
 *     moe_align block size", Purpose.
 *  7. M-aware tier: A = 64 while num_tokens*topk/E is below one full
 *     128-row block per expert, else 128. Same page, Purpose (commit 2) and
 *     Scope and safety (2048+ tokens keep the large tier).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ---------------------------------------------------------------- bf16 --- */

/* bf16: 1 sign bit, 8 exponent bits (bias 127), 7 stored fraction bits.
 * Normal numbers carry 8 significant bits; below 2^-126 the spacing is fixed
 * at 2^-133 (subnormals). The largest finite value is (2 - 2^-7) * 2^127. */
ORACLE_API uint16_t oracle_bf16_from_double(double v)
{
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e2;
    frexp(a, &e2);                 /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                /* a in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;        /* subnormal range: fixed spacing */
    double q = ldexp(1.0, e - 7);  /* spacing of bf16 values near a */
    double n = nearbyint(a / q);   /* a/q is exact; default mode is RNE */
    double r = n * q;
    if (r >= ldexp(2.0, 127)) return (uint16_t)(sign | 0x7F80);  /* overflow */
    float f = (float)r;            /* exact: r has <= 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return (uint16_t)(sign | ((bits >> 16) & 0x7FFF));
}

ORACLE_API double oracle_bf16_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* out[i] = in[i] rounded to bf16 (as above), as a double. */
ORACLE_API void oracle_bf16_round_array(int64_t n, const double *in, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_to_double(oracle_bf16_from_double(in[i]));
}

/* ---------------------------------------------------------------- e4m3 --- */

/* E4M3 (the FP8 format of "Netra Kernel ...", Fusing the activation/
 * quantization boundary): 1 sign bit, 4 exponent bits (bias 7), 3 stored
 * fraction bits, no infinities; code 0x7F / 0xFF is NaN. Normal numbers carry
 * 4 significant bits; below 2^-6 the spacing is fixed at 2^-9 (subnormals).
 * The largest finite value is 1.75 * 2^8 = 448. Rounds to nearest even and
 * saturates: magnitudes beyond 448 give +-448. */
ORACLE_API uint8_t oracle_e4m3_from_double(double v)
{
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);
    int e = e2 - 1;                /* a in [2^e, 2^(e+1)) */
    if (e < -6) e = -6;            /* subnormal range: fixed spacing 2^-9 */
    double step = ldexp(1.0, e - 3);  /* spacing of e4m3 values near a */
    double m = nearbyint(a / step);     /* exact quotient; default mode is RNE */
    double r = m * step;
    if (r > 448.0) r = 448.0;      /* cannot happen below 448 (448 is a code) */
    /* encode r: exponent field and fraction */
    if (r < ldexp(1.0, -6)) return (uint8_t)(sign | (int)(r / ldexp(1.0, -9)));  /* subnormal */
    int re2;
    double f = frexp(r, &re2);     /* r = f * 2^re2, f in [0.5, 1) */
    int exp_field = re2 - 1 + 7;
    int frac = (int)((f * 2.0 - 1.0) * 8.0);
    return (uint8_t)(sign | (exp_field << 3) | frac);
}

ORACLE_API double oracle_e4m3_to_double(uint8_t c)
{
    int sign = c & 0x80, ef = (c >> 3) & 0xF, fr = c & 7;
    if ((c & 0x7F) == 0x7F) return NAN;
    double mag = ef == 0 ? ldexp((double)fr, -9) : ldexp(1.0 + fr / 8.0, ef - 7);
    return sign ? -mag : mag;
}

/* Hidden states quantised once for the expert GEMMs ("Netra Kernel ...",
 * Fusing the activation/quantization boundary: each contiguous 128-element
 * block to E4M3 with its block scale). Reading taken: per row t and block b
 * of 128 elements, amax = max |x|, scale[t][b] = amax / 448 and the codes are
 * e4m3(x * (448 / amax)), each division and the product rounded to fp32 (the
 * precision the kernel decides the codes in: fp32 operands and results);
 * a block of zeros has scale 0 and zero codes. H must be a multiple of 128.
 * q [M][H] codes, scales [M][H/128]. */
ORACLE_API void oracle_quant_fp8(int M, int H, const uint16_t *x, int64_t ld_x, uint8_t *q, float *scales)
{
    for (int t = 0; t < M; ++t) {
        for (int b = 0; b < H / 128; ++b) {
            const uint16_t *xb = x + (int64_t)t * ld_x + (int64_t)b * 128;
            double amax = 0.0;
            for (int i = 0; i < 128; ++i) {
                double a = fabs(oracle_bf16_to_double(xb[i]));
                if (a > amax) amax = a;
            }
            uint8_t *qb = q + (int64_t)t * H + (int64_t)b * 128;
            if (amax == 0.0) {
                scales[(int64_t)t * (H / 128) + b] = 0.0f;
                for (int i = 0; i < 128; ++i) qb[i] = 0;
                continue;
            }
            float scale = (float)(amax / 448.0);
            float inv = (float)(448.0 / amax);
            scales[(int64_t)t * (H / 128) + b] = scale;
            for (int i = 0; i < 128; ++i) {
                float v = (float)(oracle_bf16_to_double(xb[i]) * (double)inv);
                qb[i] = oracle_e4m3_from_double((double)v);
            }
        }
    }
}

/* --------------------------------------------------------- gate GEMM --- */

/* z[t*E + e] = sum_h x[t,h]*W[e,h] + bias[e] in double; absdot (optional)
 * gets sum_h |x[t,h]*W[e,h]| + |bias[e]|, the scale of the rounding error a
 * finite-precision accumulation of the same sum can make. */
ORACLE_API void oracle_gate_logits(int M, int H, int E, const uint16_t *x, int64_t ld_x,
                                   const uint16_t *W, const float *bias,
                                   double *z, double *absdot)
{
    for (int t = 0; t < M; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0, aacc = 0.0;
            for (int h = 0; h < H; ++h) {
                double p = oracle_bf16_to_double(x[(int64_t)t * ld_x + h]) *
                           oracle_bf16_to_double(W[(int64_t)e * H + h]);
                acc += p;
                aacc += fabs(p);
            }
            if (bias) {
                acc += (double)bias[e];
                aacc += fabs((double)bias[e]);
            }
            z[(int64_t)t * E + e] = acc;
            if (absdot) absdot[(int64_t)t * E + e] = aacc;
        }
    }
}

/* ------------------------------------------------- top-k and softmax --- */

typedef struct { double v; int id; } scored;

/* (value desc, id asc); -0 and +0 compare equal as values. */
static int by_value_then_id(const void *pa, const void *pb)
{
    const scored *a = (const scored *)pa, *b = (const scored *)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->id < b->id) ? -1 : (a->id > b->id);
}

/* One token row: zhat[E] are the bf16-rounded logits (as doubles). Writes
 * ids[k] (slot order: value desc, id asc) and w[k], computed in double and
 * rounded once to fp32:
 *   renormalize = 1: the softmax over the E experts renormalised over the k
 *     selected, i.e. a softmax over the selected logits (the full
 *     denominator cancels);
 *   renormalize = 0: the softmax over the E experts itself, read at the k
 *     selected ids (weights sum to less than 1 when k < E) -- the
 *     "unnormalized top-k weights" a guard of vLLM #60833 ("--monokernel
 *     decode", Details, Refusals) refuses, and the renormalize flag of the
 *     _router_triton_kernel of sglang #41133 (Motivation) turned off. */
ORACLE_API void oracle_select(int E, int k, int renormalize, const double *zhat, int32_t *ids, float *w)
{
    scored *s = (scored *)malloc(sizeof(scored) * (size_t)E);
    for (int e = 0; e < E; ++e) { s[e].v = zhat[e]; s[e].id = e; }
    qsort(s, (size_t)E, sizeof(scored), by_value_then_id);
    double zmax = s[0].v;
    double denom = 0.0;
    int nden = renormalize ? k : E;
    for (int i = 0; i < nden; ++i) denom += exp(s[i].v - zmax);
    for (int i = 0; i < k; ++i) {
        ids[i] = s[i].id;
        w[i] = (float)(exp(s[i].v - zmax) / denom);
    }
    free(s);
}

/* Shared slot weight: scale * sigmoid(s), s the unrounded shared logit. */
ORACLE_API float oracle_shared_weight(double s, float scale)
{
    return (float)((double)scale * (1.0 / (1.0 + exp(-s))));
}

/* Full route for M rows. Outputs ids/w are [M, k+S] row-major. Optional:
 * zhat_out [M,E] (rounded logits as doubles), z_out [M,E] (unrounded),
 * absdot_out [M,E], s_out [M] (shared logit, unrounded). renormalize: see
 * oracle_select. shared_bf16 = 1 rounds the shared logit to bf16 before the
 * sigmoid (the shared gate as a bf16 dot product, "Netra Kernel ...",
 * Reusing routing work instead of recomputing it); 0 keeps it unrounded
 * (only the routed logits are rounded, sglang #41133, Modifications). */
ORACLE_API void oracle_route(int M, int H, int E, int k, int has_shared, float scale,
                             int renormalize, int shared_bf16,
                             const uint16_t *x, int64_t ld_x, const uint16_t *W,
                             const uint16_t *Ws, const float *bias,
                             int32_t *ids, float *w,
                             double *zhat_out, double *z_out, double *absdot_out,
                             double *s_out)
{
    int width = k + (has_shared ? 1 : 0);
    double *z = (double *)malloc(sizeof(double) * (size_t)E);
    double *zh = (double *)malloc(sizeof(double) * (size_t)E);
    double *ad = absdot_out ? (double *)malloc(sizeof(double) * (size_t)E) : NULL;
    for (int t = 0; t < M; ++t) {
        const uint16_t *xt = x + (int64_t)t * ld_x;
        oracle_gate_logits(1, H, E, xt, ld_x, W, bias, z, ad);
        for (int e = 0; e < E; ++e)
            zh[e] = oracle_bf16_to_double(oracle_bf16_from_double(z[e]));
        oracle_select(E, k, renormalize, zh, ids + (int64_t)t * width, w + (int64_t)t * width);
        if (has_shared) {
            double s;
            oracle_gate_logits(1, H, 1, xt, ld_x, Ws, NULL, &s, NULL);
            double sr = shared_bf16 ? oracle_bf16_to_double(oracle_bf16_from_double(s)) : s;
            ids[(int64_t)t * width + k] = E;
            w[(int64_t)t * width + k] = oracle_shared_weight(sr, scale);
            if (s_out) s_out[t] = s;
        }
        if (zhat_out) memcpy(zhat_out + (int64_t)t * E, zh, sizeof(double) * (size_t)E);
        if (z_out) memcpy(z_out + (int64_t)t * E, z, sizeof(double) * (size_t)E);
        if (absdot_out) memcpy(absdot_out + (int64_t)t * E, ad, sizeof(double) * (size_t)E);
    }
    free(z);
    free(zh);
    free(ad);
}

/* The same route with the token rows split into nthreads contiguous blocks,
 * one thread each. Every row is computed by oracle_route exactly as in a
 * single call (rows are independent), so the results are identical; the
 * threads only shorten the wall time. Returns 0, or -1 if a thread could
 * not be started (its rows are then computed on the calling thread). */
typedef struct {
    int M, H, E, k, has_shared;
    float scale;
    int renormalize, shared_bf16;
    const uint16_t *x;
    int64_t ld_x;
    const uint16_t *W, *Ws;
    const float *bias;
    int32_t *ids;
    float *w;
    double *zhat_out, *z_out, *absdot_out, *s_out;
} route_job;

static void *route_job_run(void *arg)
{
    route_job *j = (route_job *)arg;
    oracle_route(j->M, j->H, j->E, j->k, j->has_shared, j->scale, j->renormalize, j->shared_bf16,
                 j->x, j->ld_x, j->W, j->Ws,
                 j->bias, j->ids, j->w, j->zhat_out, j->z_out, j->absdot_out, j->s_out);
    return NULL;
}

ORACLE_API int oracle_route_threads(int nthreads, int M, int H, int E, int k, int has_shared,
                                    float scale, int renormalize, int shared_bf16,
                                    const uint16_t *x, int64_t ld_x,
                                    const uint16_t *W, const uint16_t *Ws, const float *bias,
                                    int32_t *ids, float *w, double *zhat_out, double *z_out,
                                    double *absdot_out, double *s_out)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = M > 0 ? M : 1;
    int width = k + (has_shared ? 1 : 0);
    route_job *jobs = (route_job *)calloc((size_t)nthreads, sizeof(route_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    int *started = (int *)calloc((size_t)nthreads, sizeof(int));
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        int r0 = (int)((int64_t)M * i / nthreads), r1 = (int)((int64_t)M * (i + 1) / nthreads);
        route_job *j = &jobs[i];
        j->M = r1 - r0; j->H = H; j->E = E; j->k = k; j->has_shared = has_shared; j->scale = scale;
        j->renormalize = renormalize; j->shared_bf16 = shared_bf16;
        j->x = x + (int64_t)r0 * ld_x; j->ld_x = ld_x; j->W = W; j->Ws = Ws; j->bias = bias;
        j->ids = ids + (int64_t)r0 * width; j->w = w + (int64_t)r0 * width;
        j->zhat_out = zhat_out ? zhat_out + (int64_t)r0 * E : NULL;
        j->z_out = z_out ? z_out + (int64_t)r0 * E : NULL;
        j->absdot_out = absdot_out ? absdot_out + (int64_t)r0 * E : NULL;
        j->s_out = s_out ? s_out + r0 : NULL;
        started[i] = pthread_create(&th[i], NULL, route_job_run, j) == 0;
        if (!started[i]) rc = -1;
    }
    for (int i = 0; i < nthreads; ++i) {
        if (started[i]) pthread_join(th[i], NULL);
        else route_job_run(&jobs[i]);
    }
    free(jobs);
    free(th);
    free(started);
    return rc;
}

/* ------------------------------------------------------------- align --- */

/* M-aware alignment tier: 64 below one full 128-row block of routed rows per
 * expert (num_tokens*topk/E < 128), 128 at or above it. */
ORACLE_API int oracle_select_block_size(int num_tokens, int topk, int num_experts)
{
    return ((int64_t)num_tokens * topk < (int64_t)128 * num_experts) ? 64 : 128;
}

/* Worst-case num_tokens_post_padded: every slot plus A-1 padding rows per
 * expert (the workspace num_slots of the alignment page). */
ORACLE_API int64_t oracle_align_capacity(int64_t numel, int num_experts, int A)
{
    return numel + (int64_t)num_experts * (A - 1);
}

/* Sequential moe_align_block_size. ids[numel] hold expert ids in
 * [0, num_experts); the flat slot index i = t*width + s is the value stored.
 * sorted[0, npp) and expert_ids[0, npp/A) are written; padding = numel.
 * Returns 0, or -1 if an id is out of range or a capacity is too small. */
ORACLE_API int oracle_align(const int32_t *ids, int64_t numel, int num_experts, int A,
                            int32_t *sorted, int64_t sorted_cap,
                            int32_t *expert_ids, int64_t expert_cap, int32_t *npp_out)
{
    int64_t *cnt = (int64_t *)calloc((size_t)num_experts, sizeof(int64_t));
    int64_t *off = (int64_t *)calloc((size_t)num_experts + 1, sizeof(int64_t));
    int64_t *cur = (int64_t *)calloc((size_t)num_experts, sizeof(int64_t));
    int rc = 0;
    /* per-expert counts */
    for (int64_t i = 0; i < numel; ++i) {
        if (ids[i] < 0 || ids[i] >= num_experts) { rc = -1; goto done; }
        cnt[ids[i]] += 1;
    }
    /* padded prefix sum */
    for (int e = 0; e < num_experts; ++e)
        off[e + 1] = off[e] + (cnt[e] + A - 1) / A * A;
    if (off[num_experts] > sorted_cap || off[num_experts] / A > expert_cap) { rc = -1; goto done; }
    /* stable scatter in ascending flat index */
    for (int e = 0; e < num_experts; ++e) cur[e] = off[e];
    for (int64_t i = 0; i < numel; ++i) sorted[cur[ids[i]]++] = (int32_t)i;
    /* padding rows and per-block expert ids */
    for (int e = 0; e < num_experts; ++e) {
        for (int64_t p = off[e] + cnt[e]; p < off[e + 1]; ++p) sorted[p] = (int32_t)numel;
        for (int64_t b = off[e] / A; b < off[e + 1] / A; ++b) expert_ids[b] = e;
    }
    *npp_out = (int32_t)off[num_experts];
done:
    free(cnt);
    free(off);
    free(cur);
    return rc;
}

/* moe_align_block_size behind an expert-parallel load-balancing (EPLB)
 * logical->physical remap, which the pages' guards refuse (sglang #41133,
 * Modifications: "no EPLB remap"; vLLM #60833, Details, Refusals) and do not
 * define; the reading taken here: logical expert e is held by count[e]
 * physical replicas, listed in map[e * max_replicas + r], r < count[e]; the
 * slot (t, s) of token t = i / width goes to replica r = t mod count[e], so a
 * token's slots of one expert meet on one replica and consecutive tokens
 * take its replicas in turn. The physical ids are then aligned exactly as
 * above over num_physical experts (ids, padding and block owners are
 * physical; the flat slot indices stored are unchanged). Returns 0, or -1 on
 * an id, count or physical id out of range or a capacity too small. */
ORACLE_API int oracle_align_eplb(const int32_t *ids, int64_t numel, int width, int num_experts,
                                 const int32_t *map, const int32_t *count, int max_replicas,
                                 int num_physical, int A, int32_t *sorted, int64_t sorted_cap,
                                 int32_t *expert_ids, int64_t expert_cap, int32_t *npp_out)
{
    int32_t *phys = (int32_t *)malloc(sizeof(int32_t) * (size_t)(numel > 0 ? numel : 1));
    int rc = 0;
    for (int64_t i = 0; i < numel; ++i) {
        int e = ids[i];
        if (e < 0 || e >= num_experts || count[e] < 1 || count[e] > max_replicas) { rc = -1; break; }
        int64_t t = i / width;
        int p = map[(int64_t)e * max_replicas + (int)(t % count[e])];
        if (p < 0 || p >= num_physical) { rc = -1; break; }
        phys[i] = p;
    }
    if (rc == 0)
        rc = oracle_align(phys, numel, num_physical, A, sorted, sorted_cap, expert_ids, expert_cap,
                          npp_out);
    free(phys);
    return rc;
}

/* ------------------------------------------------- consumer expert GEMM --- */

/* The expert GEMM that consumes the align's output ("[ROCm][Kernel] W4A16
 * MoE prefill: M-aware moe_align block size", Purpose: each block of A rows
 * of sorted_token_ids runs the full K contraction against the weights of
 * expert_ids[block]; blocks at or past num_tokens_post_padded return early),
 * here with bf16 expert weights. Whatever the blocking, every routed slot
 * i = t * width + s gets out[i][n] = sum_h x[t][h] * W[ids[i]][n][h], so the
 * oracle is that plain definition per slot, in double, with absdot (optional)
 * the sum of |x * W|. W is [num_experts][N][H]. */
ORACLE_API void oracle_expert_gemm(int64_t numel, int H, int N, int width, const int32_t *ids,
                                   const uint16_t *x, int64_t ld_x, const uint16_t *W, double *out,
                                   double *absdot)
{
    for (int64_t i = 0; i < numel; ++i) {
        const uint16_t *xt = x + (i / width) * ld_x;
        const uint16_t *we = W + (int64_t)ids[i] * N * H;
        for (int n = 0; n < N; ++n) {
            double acc = 0.0, aacc = 0.0;
            for (int h = 0; h < H; ++h) {
                double p = oracle_bf16_to_double(xt[h]) * oracle_bf16_to_double(we[(int64_t)n * H + h]);
                acc += p;
                aacc += fabs(p);
            }
            out[i * N + n] = acc;
            if (absdot) absdot[i * N + n] = aacc;
        }
    }
}

