/*
 * bimoe_oracle.c -- plain, slow, single-threaded fp64 CPU oracle for the
 * batch-invariant MoE hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
 * its Python binding) may link, load or call this file; only the test-suite,
 * the smoke check and the CPU-baseline leg of the benchmark use it.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * Every routine is the textbook definition written out as loops, in double
 * precision, with no blocking, fusion or reordering.  Inputs arrive in the
 * storage formats the CUDA path consumes (fp32, and bf16 as raw uint16 bit
 * patterns); each fp32/bf16 value converts to double exactly, so the only
 * rounding here is fp64 summation.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off (no -ffast-math, no FMA
 * contraction) so that x86-64 and aarch64 hosts produce identical doubles.
 *
 * Sources (page title, section):
 *  - "[BI][DSv4] Batch-invariant GateLinear router with fp32 persistent
 *    matmul", section "What": the router is an fp32 linear layer y = x W^T + b
 *    whose scores must stay fp32; bias is preserved.
 *  - "Batch-invariance generation with vLLM fused-MoE backend ...", section
 *    "What's included" and the strict-review summary: gated SwiGLU with the
 *    routing probability applied at the activation, gate|up half split, and a
 *    top-k reduction with unit weights in a fixed slot order.
 *  - "[BI][DSv4] Pin sparse-MLA decode and prefill scheduling ...", commit
 *    "deterministic per-row top-k": score descending, exact ties by ascending
 *    index, -0.0 canonicalised to +0.0, ranking on a monotone int32 key; and
 *    for the windowed (indexer) top-k the same commit plus the masked-lane,
 *    sentinel and validity-first ranking commits that follow it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

static double bf16_to_double(uint16_t v) {
    uint32_t u = ((uint32_t)v) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------- router --
 * r[m,n] = sum_{k=0}^{K-1} x[m,k] * w[n,k]  (+ b[n])
 * x is [M,K] row-major, w is [N,K] row-major (nn.Linear layout, used as W^T),
 * b is [N] or NULL, r is [M,N] row-major fp64.  The sum runs in increasing k
 * in fp64; the bias is added last.  (GateLinear page, "What".) */
ORACLE_API void oracle_router(const float *x, const float *w, const float *b,
                              int64_t M, int64_t K, int64_t N, double *r) {
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += (double)x[m * K + k] * (double)w[n * K + k];
            if (b) s += (double)b[n];
            r[m * N + n] = s;
        }
    }
}

/* Logistic sigmoid 1 / (1 + e^-v) in fp64; the scoring function of the
 * router (sigmoid scoring of the DSv4-style router). */
ORACLE_API double oracle_sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

ORACLE_API void oracle_sigmoid_vec(const float *y, int64_t n, double *p) {
    for (int64_t i = 0; i < n; ++i) p[i] = oracle_sigmoid((double)y[i]);
}

/* Monotone int32 key of an fp32 value ("deterministic per-row top-k" commit):
 * -0.0 is canonicalised to +0.0, then negative values have their low 31 bits
 * flipped so that signed-integer order equals numeric order.  +NaN sorts above
 * +inf and -NaN below -inf; two distinct NaN patterns keep distinct keys. */
ORACLE_API int32_t oracle_score_key(float v) {
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    if (u == 0x80000000u) u = 0u;
    if (u & 0x80000000u) u ^= 0x7fffffffu;
    return (int32_t)u;
}

/* ------------------------------------------------------------------ top-k --
 * For each row of scores[M,E] (fp32 router outputs) choose top_k experts in
 * rank order: larger key first, and among equal keys the lower expert index
 * first.  Done as top_k rounds of "scan every untaken expert in ascending
 * index, keep the first strictly better one".  ids[m,t] is the rank-t expert,
 * wts[m,t] = sigmoid(scores[m, ids[m,t]]) in fp64.  Slot t is rank t. */
ORACLE_API void oracle_topk(const float *scores, int64_t M, int64_t E,
                            int32_t top_k, int32_t *ids, double *wts) {
    unsigned char *taken = (unsigned char *)malloc((size_t)(E > 0 ? E : 1));
    for (int64_t m = 0; m < M; ++m) {
        const float *row = scores + m * E;
        memset(taken, 0, (size_t)(E > 0 ? E : 1));
        for (int32_t t = 0; t < top_k; ++t) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || oracle_score_key(row[e]) > oracle_score_key(row[best]))
                    best = e;
            }
            taken[best] = 1;
            ids[m * top_k + t] = (int32_t)best;
            wts[m * top_k + t] = oracle_sigmoid((double)row[best]);
        }
    }
    free(taken);
}

/* --------------------------------------------------------- windowed top-k --
 * The sparse-MLA indexer's per-row top-k ("[BI][DSv4] Pin sparse-MLA decode
 * and prefill scheduling under batch invariance", commit log: the
 * deterministic per-row top-k commit, then the masked-lane, sentinel and
 * validity-first ranking commits).  Row i of scores (row stride ld, num_cols
 * columns) has the window [rs, re) with rs = clamp(row_start[i], 0,
 * num_cols) and re = clamp(row_end[i], 0, num_cols) (empty when re <= rs);
 * row_start / row_end NULL means the whole row.  Only columns inside the
 * window can be chosen (validity ranks before any score, so no key value is
 * reserved as a sentinel).  Inside the window columns are ranked by the
 * monotone key descending, equal keys by ascending column; the first
 * min(k, window size) are chosen.  out[i, 0..] holds the chosen columns in
 * ascending column order as window-relative indices (column - rs), then -1
 * up to k.  Written as: collect the window, sort by rank, keep k, sort the
 * kept columns. */
typedef struct { int32_t key; int64_t col; } oracle_kc;

static int by_rank(const void *a, const void *b) {
    const oracle_kc *x = (const oracle_kc *)a, *y = (const oracle_kc *)b;
    if (x->key != y->key) return x->key > y->key ? -1 : 1;
    return x->col < y->col ? -1 : (x->col > y->col ? 1 : 0);
}
static int by_col(const void *a, const void *b) {
    const int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return x < y ? -1 : (x > y ? 1 : 0);
}
static int64_t clamp64(int64_t v, int64_t lo, int64_t hi) {
    return v < lo ? lo : (v > hi ? hi : v);
}

ORACLE_API void oracle_topk_window(const float *scores, int64_t ld, const int64_t *row_start,
                                   const int64_t *row_end, int64_t n_rows, int64_t num_cols,
                                   int32_t k, int32_t *out) {
    oracle_kc *cand = (oracle_kc *)malloc(sizeof(oracle_kc) * (size_t)(num_cols > 0 ? num_cols : 1));
    int64_t *kept = (int64_t *)malloc(sizeof(int64_t) * (size_t)(k > 0 ? k : 1));
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t rs = row_start ? clamp64(row_start[i], 0, num_cols) : 0;
        const int64_t re = row_end ? clamp64(row_end[i], 0, num_cols) : num_cols;
        int64_t n = 0;
        for (int64_t c = rs; c < re; ++c) {
            cand[n].key = oracle_score_key(scores[i * ld + c]);
            cand[n].col = c;
            ++n;
        }
        qsort(cand, (size_t)n, sizeof(oracle_kc), by_rank);
        const int64_t m = n < k ? n : k;
        for (int64_t j = 0; j < m; ++j) kept[j] = cand[j].col;
        qsort(kept, (size_t)m, sizeof(int64_t), by_col);
        for (int64_t j = 0; j < k; ++j)
            out[i * k + j] = j < m ? (int32_t)(kept[j] - rs) : -1;
    }
    free(kept);
    free(cand);
}

/* ---------------------------------------------------------------- permute --
 * Stable grouping of the M*top_k (token, slot) pairs by expert: pairs of
 * expert 0 first, then expert 1, ...; inside an expert by ascending token,
 * then slot.  perm[p] = m*top_k + t of the p-th pair; offsets[e] is the first
 * position of expert e and offsets[E] = M*top_k.  Returns 0, or -1 if an id is
 * outside [0,E).  Written as one pass over the pairs per expert. */
ORACLE_API int oracle_permute(const int32_t *ids, int64_t M, int64_t E,
                              int32_t top_k, int32_t *offsets, int32_t *perm) {
    for (int64_t i = 0; i < M * top_k; ++i)
        if (ids[i] < 0 || ids[i] >= E) return -1;
    int64_t pos = 0;
    for (int64_t e = 0; e < E; ++e) {
        offsets[e] = (int32_t)pos;
        for (int64_t m = 0; m < M; ++m)
            for (int32_t t = 0; t < top_k; ++t)
                if (ids[m * top_k + t] == e) perm[pos++] = (int32_t)(m * top_k + t);
    }
    offsets[E] = (int32_t)pos;
    return 0;
}

/* SwiGLU with the routing probability applied at the activation (fused-MoE
 * page, "What's included"): silu(g) * u * p with silu(g) = g * sigmoid(g). */
static double swiglu_prob(double g, double u, double p) {
    return g * oracle_sigmoid(g) * u * p;
}

/* Gate and up projections of one token row for expert e.  W13 is
 * [E, 2I, H]: rows [0,I) of an expert are the gate half, rows [I,2I) the up
 * half (half-split convention). */
static void gate_up_row(const uint16_t *xrow, const uint16_t *w13, int64_t e,
                        int64_t H, int64_t I, double p, double *act) {
    const uint16_t *we = w13 + e * 2 * I * H;
    for (int64_t j = 0; j < I; ++j) {
        double g = 0.0, u = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            double xv = bf16_to_double(xrow[h]);
            g += xv * bf16_to_double(we[j * H + h]);
            u += xv * bf16_to_double(we[(I + j) * H + h]);
        }
        act[j] = swiglu_prob(g, u, p);
    }
}

/* ------------------------------------------------------- full MoE layer --
 * out[m,h] = sum_{t=0}^{top_k-1} sum_{j<I} a_{m,t}[j] * W2[e,h,j],
 *   e = ids[m,t], p = wts[m,t],
 *   a_{m,t}[j] = silu(g_j) * u_j * p,  g_j = x[m,:].W13[e,j,:],
 *                                    u_j = x[m,:].W13[e,I+j,:].
 * x [M,H] bf16, W13 [E,2I,H] bf16, W2 [E,H,I] bf16, out [M,H] fp64.  All in
 * fp64 with no intermediate rounding; slots summed in slot order t=0..k-1. */
ORACLE_API void oracle_moe(const uint16_t *x, const int32_t *ids, const float *wts,
                           const uint16_t *w13, const uint16_t *w2, int64_t M,
                           int64_t H, int64_t E, int32_t top_k, int64_t I,
                           double *out) {
    (void)E;
    double *act = (double *)malloc((size_t)(I > 0 ? I : 1) * sizeof(double));
    for (int64_t m = 0; m < M; ++m) {
        double *orow = out + m * H;
        for (int64_t h = 0; h < H; ++h) orow[h] = 0.0;
        for (int32_t t = 0; t < top_k; ++t) {
            int64_t e = ids[m * top_k + t];
            gate_up_row(x + m * H, w13, e, H, I, (double)wts[m * top_k + t], act);
            const uint16_t *w2e = w2 + e * H * I;
            for (int64_t h = 0; h < H; ++h) {
                double c = 0.0;
                for (int64_t j = 0; j < I; ++j) c += act[j] * bf16_to_double(w2e[h * I + j]);
                orow[h] += c;
            }
        }
    }
    free(act);
}

/* Expert that owns permuted position p: the e with offsets[e] <= p < offsets[e+1]. */
static int64_t expert_of(const int32_t *offsets, int64_t E, int64_t p) {
    for (int64_t e = 0; e < E; ++e)
        if (p >= offsets[e] && p < offsets[e + 1]) return e;
    return -1;
}

/* ------------------------------------------------------------ stage: gate/up
 * For every permuted position p (pair = perm[p], token m = pair / top_k):
 * act[p,j] = silu(g_j) * u_j * wts[pair] with g, u the gate/up projections
 * of x[m,:] by the owning expert.  act is [P, I] fp64, P = offsets[E]. */
ORACLE_API void oracle_gate_up(const uint16_t *x, const int32_t *offsets,
                               const int32_t *perm, const float *wts,
                               const uint16_t *w13, int64_t H, int64_t E,
                               int32_t top_k, int64_t I, double *act) {
    int64_t P = offsets[E];
    for (int64_t p = 0; p < P; ++p) {
        int64_t e = expert_of(offsets, E, p);
        int64_t pair = perm[p];
        gate_up_row(x + (pair / top_k) * H, w13, e, H, I, (double)wts[pair], act + p * I);
    }
}

/* -------------------------------------------------------------- stage: down
 * contrib[pair,h] = sum_{j<I} act[p,j] * W2[e,h,j] for pair = perm[p], e the
 * owning expert of position p.  act [P,I] bf16, contrib [M*top_k, H] fp64
 * (row = token*top_k + slot). */
ORACLE_API void oracle_down(const uint16_t *act, const int32_t *offsets,
                            const int32_t *perm, const uint16_t *w2, int64_t H,
                            int64_t E, int64_t I, double *contrib) {
    int64_t P = offsets[E];
    for (int64_t p = 0; p < P; ++p) {
        int64_t e = expert_of(offsets, E, p);
        const uint16_t *w2e = w2 + e * H * I;
        double *crow = contrib + (int64_t)perm[p] * H;
        for (int64_t h = 0; h < H; ++h) {
            double c = 0.0;
            for (int64_t j = 0; j < I; ++j)
                c += bf16_to_double(act[p * I + j]) * bf16_to_double(w2e[h * I + j]);
            crow[h] = c;
        }
    }
}

/* ----------------------------------------------------------- stage: combine
 * out[m,h] = sum_{t=0}^{top_k-1} contrib[m,t,h] with unit weights (the
 * probabilities were applied at the activation), in slot order. */
ORACLE_API void oracle_combine(const float *contrib, int64_t M, int64_t H,
                               int32_t top_k, double *out) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t h = 0; h < H; ++h) {
            double s = 0.0;
            for (int32_t t = 0; t < top_k; ++t)
                s += (double)contrib[(m * top_k + t) * H + h];
            out[m * H + h] = s;
        }
}
