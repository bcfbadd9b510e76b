/*
 * gr_oracle.c -- fp64 CPU oracle for large-beam decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes is the plain definition of the three-stage attention the
 * pages describe, written out without any blocking or fusion:
 *
 *   - GR-Inference blog, "system design": ContextKV is one long KV per
 *     request shared by every beam; BeamKV holds only the short K/V each beam
 *     adds per decode step; BeamPath records forks and reorders by index.
 *   - GR-Inference blog, "kernel design" / SID-GR README section 3 ("Core
 *     implementation points": BeamPath records logical parent-child
 *     relations): the decode attention reads ContextKV, follows BeamPath into
 *     BeamKV, and merges the two parts by log-sum-exp.
 *   - xGR review, "xAttention" (three-stage computation): shared stage,
 *     unshared stage, merging stage.  Merging two exact partial softmaxes by
 *     log-sum-exp gives the softmax over the union of their key sets, so the
 *     oracle computes that union directly.
 *
 * For request r, active beam b < W_s at step s, query head h (kv head
 * g = h / G, G = Hq / Hkv):
 *   1. ancestors: a_s = b, a_{t-1} = BeamPath[r, t, a_t] for t = s .. 1
 *   2. keys   = ctx_k[r, g, 0 .. len_r-1] ++ beam_k[r, t, a_t, g] (t = 0 .. s)
 *      values = ctx_v[r, g, 0 .. len_r-1] ++ beam_v[r, t, a_t, g] (t = 0 .. s)
 *   3. x_j = scale * <q[r, b, h], key_j>            (fp64)
 *   4. lse = max_j x_j + ln sum_j exp(x_j - max)    (natural log)
 *   5. out = sum_j exp(x_j - lse) * value_j
 *
 * Readings where the pages are silent: BeamPath entries are parent slots in
 * the previous step (step 0 expands from the single prefill row, so its
 * entries are never followed); the chain includes the current step's token;
 * query heads g*G .. g*G+G-1 share kv head g; the scale is the caller's fp32
 * value widened to fp64.
 *
 * Compile-time switch ORACLE_MUTANT=k plants one deliberate mistake (used by
 * the test that shows the pins catch mistakes); 0 (the default) is the
 * oracle itself.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_PATH (-2)
#define ORACLE_NO_MEMORY (-3)

/* bf16 is the top half of an IEEE binary32; widening to double is exact. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }

/* Step 1: walk BeamPath from slot b at step `step` back to step 0.
 * anc_row[t] receives a_t.  Returns ORACLE_BAD_PATH on a parent outside
 * [0, W_{t-1}). */
static int walk_path(int32_t S_max, int32_t W_max, const int32_t *beam_path,
                     const int32_t *widths, int32_t step, int32_t r, int32_t b,
                     int32_t *anc_row)
{
    int32_t a = b;
    anc_row[step] = a;
    for (int32_t t = step; t >= 1; --t) {
#if ORACLE_MUTANT == 2
        /* mistake: reads the parent from the wrong step row */
        int32_t p = beam_path[((int64_t)r * S_max + (t - 1)) * W_max + a];
#else
        int32_t p = beam_path[((int64_t)r * S_max + t) * W_max + a];
#endif
        if (p < 0 || p >= widths[t - 1])
            return ORACLE_BAD_PATH;
#if ORACLE_MUTANT == 5
        /* mistake: ignores BeamPath and keeps the beam's own slot */
        p = (b < widths[t - 1]) ? b : 0;
#endif
        a = p;
        anc_row[t - 1] = a;
    }
    return ORACLE_OK;
}

int oracle_ancestors(int32_t R, int32_t S_max, int32_t W_max,
                     const int32_t *beam_path, const int32_t *widths, int32_t step,
                     const int32_t *sel_r, const int32_t *sel_b, int64_t n_sel,
                     int32_t *anc)
{
    if (!beam_path || !widths || !sel_r || !sel_b || !anc || step < 0 || step >= S_max)
        return ORACLE_BAD_ARG;
    for (int64_t i = 0; i < n_sel; ++i) {
        if (sel_r[i] < 0 || sel_r[i] >= R || sel_b[i] < 0 || sel_b[i] >= widths[step])
            return ORACLE_BAD_ARG;
        int rc = walk_path(S_max, W_max, beam_path, widths, step, sel_r[i], sel_b[i],
                           anc + i * (int64_t)(step + 1));
        if (rc)
            return rc;
    }
    return ORACLE_OK;
}

/*
 * Full attention for the selected rows (sel_r[i], sel_b[i]), all Hq heads.
 * The key set is ctx positions [lo, hi) clipped to [0, len_r) (hi < 0 means
 * len_r), plus the beam chain when include_beam != 0.  With an empty key
 * set the row's lse is -inf and its output 0.
 *   q      : bf16 [R, W_s, Hq, D]
 *   ctx_k/v: bf16 [R, Hkv, Lc_max, D]
 *   beam_k/v: bf16 [R, S_max, W_max, Hkv, D]
 *   out    : f64 [n_sel, Hq, D];  lse: f64 [n_sel, Hq];  anc: i32 [n_sel, step+1] or NULL
 */
int oracle_decode_attn(int32_t R, int32_t Hq, int32_t Hkv, int32_t D,
                       int32_t Lc_max, int32_t S_max, int32_t W_max, float softmax_scale,
                       const uint16_t *q, const uint16_t *ctx_k, const uint16_t *ctx_v,
                       const int32_t *ctx_len, const uint16_t *beam_k, const uint16_t *beam_v,
                       const int32_t *beam_path, const int32_t *widths, int32_t step,
                       const int32_t *sel_r, const int32_t *sel_b, int64_t n_sel,
                       int32_t ctx_lo, int32_t ctx_hi, int32_t include_beam,
                       double *out, double *lse, int32_t *anc, int32_t num_threads)
{
    if (R <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || S_max <= 0 ||
        W_max <= 0 || Lc_max < 0 || step < 0 || step >= S_max)
        return ORACLE_BAD_ARG;
    if (!q || !ctx_len || !beam_k || !beam_v || !beam_path || !widths || !sel_r ||
        !sel_b || !out || !lse)
        return ORACLE_BAD_ARG;
    if (Lc_max > 0 && (!ctx_k || !ctx_v))
        return ORACLE_BAD_ARG;
    for (int32_t t = 0; t <= step; ++t)
        if (widths[t] < 1 || widths[t] > W_max)
            return ORACLE_BAD_ARG;
    for (int32_t r = 0; r < R; ++r)
        if (ctx_len[r] < 0 || ctx_len[r] > Lc_max)
            return ORACLE_BAD_ARG;
    for (int64_t i = 0; i < n_sel; ++i)
        if (sel_r[i] < 0 || sel_r[i] >= R || sel_b[i] < 0 || sel_b[i] >= widths[step])
            return ORACLE_BAD_ARG;

    const int32_t G = Hq / Hkv;
    const int32_t W_s = widths[step];
    const int32_t n_max = Lc_max + step + 1;
    const double scale = (double)softmax_scale;
    int status = ORACLE_OK;

#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif

#pragma omp parallel
    {
        /* per-thread scratch: the materialised key/value sequence of one
         * (request, beam, kv head), its scores, and the ancestor chain */
        double *kseq = (double *)malloc(sizeof(double) * (size_t)n_max * (size_t)D);
        double *vseq = (double *)malloc(sizeof(double) * (size_t)n_max * (size_t)D);
        double *x = (double *)malloc(sizeof(double) * (size_t)n_max);
        int32_t *chain = (int32_t *)malloc(sizeof(int32_t) * (size_t)(step + 1));
        if (!kseq || !vseq || !x || !chain) {
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < n_sel; ++i) {
                const int32_t r = sel_r[i], b = sel_b[i];
                if (walk_path(S_max, W_max, beam_path, widths, step, r, b, chain)) {
#pragma omp atomic write
                    status = ORACLE_BAD_PATH;
                    continue;
                }
                if (anc)
                    memcpy(anc + i * (int64_t)(step + 1), chain, sizeof(int32_t) * (size_t)(step + 1));

                int32_t lo = ctx_lo < 0 ? 0 : ctx_lo;
                int32_t hi = (ctx_hi < 0 || ctx_hi > ctx_len[r]) ? ctx_len[r] : ctx_hi;
                if (lo > hi)
                    lo = hi;

                for (int32_t g = 0; g < Hkv; ++g) {
                    /* step 2: materialise keys and values for kv head g */
                    int32_t n = 0;
                    for (int32_t j = lo; j < hi; ++j, ++n) {
                        const int64_t base = (((int64_t)r * Hkv + g) * Lc_max + j) * D;
                        for (int32_t d = 0; d < D; ++d) {
                            kseq[(int64_t)n * D + d] = bf16_to_double(ctx_k[base + d]);
                            vseq[(int64_t)n * D + d] = bf16_to_double(ctx_v[base + d]);
                        }
                    }
#if ORACLE_MUTANT == 1
                    /* mistake: drops the per-beam (unshared) stage */
                    if (0)
#else
                    if (include_beam)
#endif
                    {
#if ORACLE_MUTANT == 8
                        /* mistake: leaves out the current step's own token */
                        const int32_t t_end = step - 1;
#else
                        const int32_t t_end = step;
#endif
                        for (int32_t t = 0; t <= t_end; ++t, ++n) {
                            const int64_t base =
                                ((((int64_t)r * S_max + t) * W_max + chain[t]) * Hkv + g) * D;
                            for (int32_t d = 0; d < D; ++d) {
                                kseq[(int64_t)n * D + d] = bf16_to_double(beam_k[base + d]);
                                vseq[(int64_t)n * D + d] = bf16_to_double(beam_v[base + d]);
                            }
                        }
                    }

                    for (int32_t hh = 0; hh < G; ++hh) {
#if ORACLE_MUTANT == 3
                        /* mistake: interleaved instead of contiguous head groups */
                        const int32_t h = hh * Hkv + g;
#else
                        const int32_t h = g * G + hh;
#endif
                        const uint16_t *qrow = q + (((int64_t)r * W_s + b) * Hq + h) * D;
                        double *orow = out + (i * Hq + h) * (int64_t)D;
                        if (n == 0) {
                            lse[i * Hq + h] = -INFINITY;
                            for (int32_t d = 0; d < D; ++d)
                                orow[d] = 0.0;
                            continue;
                        }
                        /* step 3: scores */
                        double m = -INFINITY;
                        for (int32_t j = 0; j < n; ++j) {
                            double acc = 0.0;
                            for (int32_t d = 0; d < D; ++d)
                                acc += bf16_to_double(qrow[d]) * kseq[(int64_t)j * D + d];
#if ORACLE_MUTANT == 4
                            x[j] = acc; /* mistake: scale left out */
#else
                            x[j] = scale * acc;
#endif
                            if (x[j] > m)
                                m = x[j];
                        }
                        /* step 4: log-sum-exp */
                        double sum = 0.0;
                        for (int32_t j = 0; j < n; ++j)
                            sum += exp(x[j] - m);
#if ORACLE_MUTANT == 6
                        const double L = m + log2(sum); /* mistake: base-2 log */
#else
                        const double L = m + log(sum);
#endif
                        lse[i * Hq + h] = L;
                        /* step 5: weighted sum of values */
                        for (int32_t d = 0; d < D; ++d)
                            orow[d] = 0.0;
                        for (int32_t j = 0; j < n; ++j) {
#if ORACLE_MUTANT == 7
                            const double p = exp(x[j] - m); /* mistake: not normalised */
#else
                            const double p = exp(x[j] - L);
#endif
                            for (int32_t d = 0; d < D; ++d)
                                orow[d] += p * vseq[(int64_t)j * D + d];
                        }
                    }
                }
            }
        }
        free(kseq);
        free(vseq);
        free(x);
        free(chain);
    }
    return status;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
