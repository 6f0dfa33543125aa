/*
 * moe_oracle.c -- CPU oracle for the forward pass of a top-k gated
 * Mixture-of-Experts FFN layer: route -> dispatch (permute) -> per-expert
 * SwiGLU FFN -> gate-weighted combine.
 *
 * TEST INFRASTRUCTURE. This is the plain, slow, checkable statement of what
 * the layer computes. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it; the CUDA library never does, and the two
 * share no code, header, table or helper. If the CUDA library is missing the
 * product path fails; it never falls back to this file.
 *
 * Where the method comes from.
 *   - The parts of the layer (top-k routing, "dispatch" of tokens to experts,
 *     "combine" of the expert outputs) are named in the DisagMoE summary
 *     (gist.science, "Resumo Tecnico: DisagMoE", section 2.2 AF-Pipe,
 *     "Alinhamento de Estagios").
 *   - The two expert GEMMs, split along the token dimension M for the first
 *     ("Layer 0") and along the hidden dimension N for the second ("Layer 1"),
 *     are named on the COMET page (nav.superapi.store/en/comet, "COMET's
 *     Technical Principles", "Tensor Decomposition").
 *   - The pages give no formula for the gate, the activation or the
 *     summation order. This file takes these readings (each one listed in the
 *     design notes of the repository):
 *       R1 logits are an fp32 dot product in one fixed "canonical" order
 *          (below), so that the selected expert ids are well defined bit for
 *          bit; the optional per-expert bias is added with one fp32 add;
 *       R2 top-k is taken on the logits, in descending order, ties going to
 *          the lower expert id; the rank of a selection is its position;
 *       R3 gate weights are the softmax of the k selected logits (equal to a
 *          softmax over all E experts renormalised over the selected k);
 *       R4 the expert FFN is SwiGLU: y = (silu(x W1) * (x W3)) W2 with
 *          silu(a) = a / (1 + exp(-a)); W1 is under the silu;
 *       R5 the combine sums w_j * y_j over ranks j = 0..k-1 in rank order,
 *          then adds the always-on shared expert (weight 1) when present.
 *     Two gating variants (readings too; the pages have neither):
 *       R3' no renormalisation: w_j is the softmax of logit j over all E
 *          experts, so the k weights sum to less than 1 (unless k = E);
 *       R5' sigmoid-gated shared expert: the shared expert's output is
 *          scaled by s(x) = 1 / (1 + exp(-x . wsg)) for a gate vector wsg[H]
 *          (x . wsg in fp64) instead of 1.
 *
 * Precision. Every input is bf16 and is widened to float exactly. The
 * logits (which decide integers: the expert ids) are computed in fp32 in the
 * canonical order, the same precision the GPU router uses. Everything
 * downstream of the ids (gate weights, the FFN, the combine) is computed in
 * fp64, the gate weights rounded once to fp32 because they are an fp32
 * output of the router.
 *
 * Canonical logit order (reading R1). For one token and one expert e, the
 * H products x[h] * Wg[h,e] (exact in fp32, since bf16 x bf16 fits in 24
 * bits) are split into 8-element chunks: chunk c holds h = 8c .. 8c+7. Chunk
 * c belongs to lane c mod 32. Each of the 32 lanes starts from +0.0f and
 * accumulates, chunk by chunk in increasing c and element by element in
 * increasing h, acc = fma(x[h], Wg[h,e], acc). The 32 lane partials are then
 * reduced by an xor butterfly: for s = 16, 8, 4, 2, 1 in turn, every lane i
 * takes a[i] + a[i ^ s]. All lanes end equal; that value, plus bias[e] if a
 * bias is given, is the logit.
 *
 * Build: cc -O2 -std=c11 -fopenmp -ffp-contract=off -fPIC -shared.
 * Portable C: no intrinsics, no architecture flags.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_NO_MEMORY (-2)

/* bf16 -> float is exact: the bf16 bits are the high half of the float. */
static float bf16_to_float(uint16_t v)
{
    uint32_t u = (uint32_t)v << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- route -- */

/* One logit, in the canonical order described in the header. */
static float canonical_logit(int32_t H, int32_t E, const uint16_t* xrow,
                             const uint16_t* Wg, int32_t e)
{
    float lane[32];
    for (int L = 0; L < 32; ++L) lane[L] = 0.0f;
    int32_t n_chunks = (H + 7) / 8;
    for (int32_t c = 0; c < n_chunks; ++c) {
        int L = c % 32;
        for (int32_t h = 8 * c; h < 8 * c + 8 && h < H; ++h) {
            float xv = bf16_to_float(xrow[h]);
            float wv = bf16_to_float(Wg[(int64_t)h * E + e]);
            lane[L] = fmaf(xv, wv, lane[L]);
        }
    }
    for (int s = 16; s >= 1; s /= 2) {
        float next[32];
        for (int i = 0; i < 32; ++i) next[i] = lane[i] + lane[i ^ s];
        for (int i = 0; i < 32; ++i) lane[i] = next[i];
    }
    return lane[0];
}

/* logits[t,e] for t < T. bias may be NULL. */
int oracle_logits(int64_t T, int32_t H, int32_t E, const uint16_t* x,
                  const uint16_t* Wg, const float* bias, float* logits)
{
    if (T < 0 || H <= 0 || E <= 0 || (T > 0 && (!x || !Wg || !logits)))
        return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t* xrow = x + t * (int64_t)H;
        for (int32_t e = 0; e < E; ++e) {
            float l = canonical_logit(H, E, xrow, Wg, e);
            if (bias) l = l + bias[e];
            logits[t * E + e] = l;
        }
    }
    return ORACLE_OK;
}

/* Top-k selection (reading R2) and gate weights (reading R3) from logits. */
int oracle_topk(int64_t T, int32_t E, int32_t k, const float* logits,
                int32_t* topk_idx, float* topk_w)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E || (T > 0 && (!logits || !topk_idx || !topk_w)))
        return ORACLE_BAD_ARG;
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        char* taken = (char*)calloc((size_t)E, 1);
        if (!taken) return ORACLE_NO_MEMORY;
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                /* strict '>' while scanning upwards: a tie keeps the lower id */
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            topk_idx[t * k + j] = best;
        }
        free(taken);
        /* softmax over the k selected logits, shifted by the largest (rank 0) */
        double m = (double)l[topk_idx[t * k]];
        double den = 0.0;
        for (int32_t j = 0; j < k; ++j) den += exp((double)l[topk_idx[t * k + j]] - m);
        for (int32_t j = 0; j < k; ++j)
            topk_w[t * k + j] = (float)(exp((double)l[topk_idx[t * k + j]] - m) / den);
    }
    return ORACLE_OK;
}

int oracle_route(int64_t T, int32_t H, int32_t E, int32_t k, const uint16_t* x,
                 const uint16_t* Wg, const float* bias, float* logits,
                 int32_t* topk_idx, float* topk_w)
{
    int rc = oracle_logits(T, H, E, x, Wg, bias, logits);
    if (rc != ORACLE_OK) return rc;
    return oracle_topk(T, E, k, logits, topk_idx, topk_w);
}

/* Reading R3': gate weights without renormalisation, from the logits and the
 * selected ids: w_j = exp(l_j - m) / sum over all E experts of exp(l_e - m),
 * m the largest logit (rank 0's), in fp64, rounded once to fp32. */
int oracle_gate_weights_full(int64_t T, int32_t E, int32_t k, const float* logits,
                             const int32_t* topk_idx, float* topk_w)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E || (T > 0 && (!logits || !topk_idx || !topk_w)))
        return ORACLE_BAD_ARG;
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        double m = (double)l[topk_idx[t * k]];
        double den_all = 0.0;
        for (int32_t e = 0; e < E; ++e) den_all += exp((double)l[e] - m);
        for (int32_t j = 0; j < k; ++j)
            topk_w[t * k + j] = (float)(exp((double)l[topk_idx[t * k + j]] - m) / den_all);
    }
    return ORACLE_OK;
}

/* Reading R5': the shared expert's scale s[t] = 1 / (1 + exp(-x[t] . wsg)),
 * the dot product in fp64 in increasing h. */
int oracle_shared_gate(int64_t T, int32_t H, const uint16_t* x, const uint16_t* wsg, double* scale)
{
    if (T < 0 || H <= 0 || (T > 0 && (!x || !wsg || !scale))) return ORACLE_BAD_ARG;
    for (int64_t t = 0; t < T; ++t) {
        double d = 0.0;
        for (int32_t h = 0; h < H; ++h)
            d += (double)bf16_to_float(x[t * H + h]) * (double)bf16_to_float(wsg[h]);
        scale[t] = 1.0 / (1.0 + exp(-d));
    }
    return ORACLE_OK;
}

/* -------------------------------------------------------------- permute -- */

/*
 * Dispatch: a stable counting sort of the R = T*k flat assignments
 * f = t*k + j by expert id topk_idx[f].
 *   counts[e]  = number of f with topk_idx[f] == e
 *   offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]
 *   src_row[p] = f for the p-th entry of the sorted order (within one expert,
 *                f increasing)
 *   inv_pos[f] = p with src_row[p] == f
 * Returns ORACLE_BAD_ARG if an id is outside [0, E).
 */
int oracle_permute(int64_t R, int32_t E, const int32_t* topk_idx, int32_t* counts,
                   int32_t* offsets, int32_t* src_row, int32_t* inv_pos)
{
    if (R < 0 || E <= 0 || !counts || !offsets || (R > 0 && (!topk_idx || !src_row || !inv_pos)))
        return ORACLE_BAD_ARG;
    for (int64_t f = 0; f < R; ++f)
        if (topk_idx[f] < 0 || topk_idx[f] >= E) return ORACLE_BAD_ARG;
    for (int32_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t f = 0; f < R; ++f) counts[topk_idx[f]] += 1;
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    if (!fill) return ORACLE_NO_MEMORY;
    for (int32_t e = 0; e < E; ++e) fill[e] = offsets[e];
    for (int64_t f = 0; f < R; ++f) {
        int32_t p = fill[topk_idx[f]]++;
        src_row[p] = (int32_t)f;
        inv_pos[f] = p;
    }
    free(fill);
    return ORACLE_OK;
}

/* ----------------------------------------------------------- expert FFN -- */

/*
 * One SwiGLU expert on one token row (reading R4), in fp64:
 *   a[f] = sum_h x[h] W1[h,f],  b[f] = sum_h x[h] W3[h,f]   (h increasing)
 *   g[f] = silu(a[f]) * b[f],   silu(a) = a / (1 + exp(-a))
 *   y[n] = sum_f g[f] W2[f,n]                              (f increasing)
 * W1, W3 are [H,F] and W2 is [F,H], row-major. scratch holds 3*F doubles.
 */
static void swiglu_row(int32_t H, int32_t F, const uint16_t* xrow, const uint16_t* W1,
                       const uint16_t* W3, const uint16_t* W2, double* scratch, double* y)
{
    double* a = scratch;
    double* b = scratch + F;
    double* g = scratch + 2 * (int64_t)F;
    for (int32_t f = 0; f < F; ++f) { a[f] = 0.0; b[f] = 0.0; }
    for (int32_t h = 0; h < H; ++h) {
        double xv = (double)bf16_to_float(xrow[h]);
        const uint16_t* w1 = W1 + (int64_t)h * F;
        const uint16_t* w3 = W3 + (int64_t)h * F;
        for (int32_t f = 0; f < F; ++f) {
            a[f] += xv * (double)bf16_to_float(w1[f]);
            b[f] += xv * (double)bf16_to_float(w3[f]);
        }
    }
    for (int32_t f = 0; f < F; ++f) g[f] = a[f] / (1.0 + exp(-a[f])) * b[f];
    for (int32_t n = 0; n < H; ++n) y[n] = 0.0;
    for (int32_t f = 0; f < F; ++f) {
        const uint16_t* w2 = W2 + (int64_t)f * H;
        double gv = g[f];
        for (int32_t n = 0; n < H; ++n) y[n] += gv * (double)bf16_to_float(w2[n]);
    }
}

/* y[H] = the SwiGLU expert e applied to one row (exposed for the tests). */
int oracle_expert_row(int32_t H, int32_t F, const uint16_t* xrow, const uint16_t* W1e,
                      const uint16_t* W3e, const uint16_t* W2e, double* y)
{
    if (H <= 0 || F <= 0 || !xrow || !W1e || !W3e || !W2e || !y) return ORACLE_BAD_ARG;
    double* scratch = (double*)malloc(sizeof(double) * 3 * (size_t)F);
    if (!scratch) return ORACLE_NO_MEMORY;
    swiglu_row(H, F, xrow, W1e, W3e, W2e, scratch, y);
    free(scratch);
    return ORACLE_OK;
}

/*
 * Layer output for a list of tokens (reading R5; R5' when shared_scale, [T],
 * is given):
 *   out[i,:] = sum_{j=0..k-1} topk_w[t,j] * FFN_{topk_idx[t,j]}(x[t])
 *              (+ FFN_shared(x[t]) when Fs > 0),  t = tokens[i]
 * summed in rank order j = 0..k-1, the shared expert last.
 * The rows are independent (a token's output depends on that token only),
 * so any subset of tokens gives the exact same rows as the whole batch.
 * The (token, expert) FFNs run in parallel; the sums run in the order above.
 * W1, W3 are [E,H,F], W2 is [E,F,H]; W1s, W3s are [H,Fs], W2s is [Fs,H].
 */
int oracle_layer_rows_gated(int64_t T, int32_t H, int32_t F, int32_t E, int32_t k, int32_t Fs,
                            const int64_t* tokens, int64_t n_tok, const int32_t* topk_idx,
                            const float* topk_w, const uint16_t* x, const uint16_t* W1,
                            const uint16_t* W3, const uint16_t* W2, const uint16_t* W1s,
                            const uint16_t* W3s, const uint16_t* W2s, const double* shared_scale,
                            double* out)
{
    if (T < 0 || H <= 0 || F <= 0 || E <= 0 || k <= 0 || k > E || Fs < 0 || n_tok < 0)
        return ORACLE_BAD_ARG;
    if (n_tok == 0) return ORACLE_OK;
    if (!tokens || !topk_idx || !topk_w || !x || !W1 || !W3 || !W2 || !out) return ORACLE_BAD_ARG;
    if (Fs > 0 && (!W1s || !W3s || !W2s)) return ORACLE_BAD_ARG;
    for (int64_t i = 0; i < n_tok; ++i) {
        if (tokens[i] < 0 || tokens[i] >= T) return ORACLE_BAD_ARG;
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = topk_idx[tokens[i] * k + j];
            if (e < 0 || e >= E) return ORACLE_BAD_ARG;
        }
    }
    int32_t per_tok = k + (Fs > 0 ? 1 : 0);
    int64_t n_jobs = n_tok * per_tok;
    int32_t Fmax = Fs > F ? Fs : F;
    double* ys = (double*)malloc(sizeof(double) * (size_t)n_jobs * (size_t)H);
    if (!ys) return ORACLE_NO_MEMORY;
    int failed = 0;
#pragma omp parallel
    {
        double* scratch = (double*)malloc(sizeof(double) * 3 * (size_t)Fmax);
        if (!scratch) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t job = 0; job < n_jobs; ++job) {
                int64_t t = tokens[job / per_tok];
                int32_t j = (int32_t)(job % per_tok);
                const uint16_t* xrow = x + t * (int64_t)H;
                double* y = ys + job * (int64_t)H;
                if (j < k) {
                    int64_t e = topk_idx[t * k + j];
                    swiglu_row(H, F, xrow, W1 + e * H * (int64_t)F, W3 + e * H * (int64_t)F,
                               W2 + e * F * (int64_t)H, scratch, y);
                } else {
                    swiglu_row(H, Fs, xrow, W1s, W3s, W2s, scratch, y);
                }
            }
            free(scratch);
        }
    }
    if (failed) { free(ys); return ORACLE_NO_MEMORY; }
    for (int64_t i = 0; i < n_tok; ++i) {
        int64_t t = tokens[i];
        double* o = out + i * (int64_t)H;
        for (int32_t n = 0; n < H; ++n) o[n] = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            double w = (double)topk_w[t * k + j];
            const double* y = ys + (i * per_tok + j) * (int64_t)H;
            for (int32_t n = 0; n < H; ++n) o[n] += w * y[n];
        }
        if (Fs > 0) {
            const double* y = ys + (i * per_tok + k) * (int64_t)H;
            if (!shared_scale) {
                for (int32_t n = 0; n < H; ++n) o[n] += y[n];
            } else {
                double sc = shared_scale[t];   /* reading R5' */
                for (int32_t n = 0; n < H; ++n) o[n] += sc * y[n];
            }
        }
    }
    free(ys);
    return ORACLE_OK;
}

/* The layer rows with the always-on shared expert at weight 1 (reading R5). */
int oracle_layer_rows(int64_t T, int32_t H, int32_t F, int32_t E, int32_t k, int32_t Fs,
                      const int64_t* tokens, int64_t n_tok, const int32_t* topk_idx,
                      const float* topk_w, const uint16_t* x, const uint16_t* W1,
                      const uint16_t* W3, const uint16_t* W2, const uint16_t* W1s,
                      const uint16_t* W3s, const uint16_t* W2s, double* out)
{
    return oracle_layer_rows_gated(T, H, F, E, k, Fs, tokens, n_tok, topk_idx, topk_w, x, W1, W3,
                                   W2, W1s, W3s, W2s, NULL, out);
}
