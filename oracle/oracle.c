/*
 * oracle.c -- plain, slow, obviously-correct fp64 CPU oracle for the
 * attention hot path of a bounded-generation SLM inference engine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path calls, links or
 * loads this file; only tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * Source of the method: "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化"
 * (163.com), abstract and section 1.2 (input/state bounds):
 *   - Packed Prefill: every sequence keeps its valid length and only valid
 *     tokens are computed (no padding).
 *   - Beam Search: all beams of one request share one prompt K/V and each
 *     beam keeps its own short suffix K/V (section 1.2); candidates, scores
 *     and the beam *parent index* come from the model (section 1.1).
 * The pages give no formula for attention itself; the plain definition used
 * here is scaled dot-product softmax attention:
 *     o = sum_j softmax_j(scale * q.k_j) v_j
 * with causal masking for prefill (query position p sees keys 0..p of its
 * own sequence, diagonal included) and no mask for decode (the query is the
 * newest position, it sees the whole prompt and its beam's suffix).
 * Readings where the pages are silent (all listed in the design notes):
 *   - grouped-query attention: q-head h reads kv-head floor(h / (Hq/Hkv));
 *   - scale is a parameter (1/sqrt(head_dim) in every workload);
 *   - inputs are bf16 bit patterns, widened exactly to double; everything
 *     after that is computed in double.
 *
 * Parity pins for these functions live in tests/test_oracle_pins.py
 * (closed forms, invariants, brute force on tiny inputs, cross-formulations).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bits -> double, exact (bf16 is the top half of an IEEE binary32). */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Softmax attention of one query row over n >= 1 keys, all in double.
 *   qrow      : head_dim bf16 values
 *   key(j)    : pointer to head_dim bf16 values of key j
 *   val(j)    : pointer to head_dim bf16 values of value j
 * Writes out[0..head_dim) and *lse = log(sum_j exp(scale q.k_j)).
 * z (scratch) holds n doubles.
 */
static void attend_row(const uint16_t *qrow, const uint16_t *const *keys,
                       const uint16_t *const *vals, int64_t n, int32_t d,
                       double scale, double *z, double *out, double *lse)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int32_t c = 0; c < d; ++c)
            dot += bf16_to_double(qrow[c]) * bf16_to_double(keys[j][c]);
        z[j] = scale * dot;
        if (z[j] > m) m = z[j];
    }
    double den = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        z[j] = exp(z[j] - m);           /* z now holds unnormalised weights */
        den += z[j];
    }
    for (int32_t c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int64_t j = 0; j < n; ++j)
            acc += z[j] * bf16_to_double(vals[j][c]);
        out[c] = acc / den;
    }
    if (lse) *lse = m + log(den);
}

/*
 * Packed variable-length causal GQA prefill attention (abstract: Packed
 * Prefill; section 1.2: only valid tokens are processed).
 *
 *   q   : bf16 [T, Hq, d]      k, v : bf16 [T, Hkv, d]
 *   cu  : int32 [B+1], cu[0] = 0, non-decreasing, cu[B] = T
 *   out : double [T, Hq, d]     lse : double [T, Hq] or NULL
 * Sequence i occupies packed rows cu[i] .. cu[i+1]-1.  Query row p of
 * sequence i, head h attends keys 0..p of the same sequence through kv-head
 * h / (Hq/Hkv).  Returns 0, or -1 on an invalid argument.
 */
int oracle_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const int32_t *cu, int32_t B, int32_t Hq, int32_t Hkv,
                   int32_t d, double scale, double *out, double *lse)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return -1;
    if (B > 0 && cu[0] != 0) return -1;
    int64_t maxlen = 0;
    for (int32_t i = 0; i < B; ++i) {
        if (cu[i + 1] < cu[i]) return -1;
        if (cu[i + 1] - cu[i] > maxlen) maxlen = cu[i + 1] - cu[i];
    }
    const int32_t g = Hq / Hkv;
    const int64_t pairs = (int64_t)B * Hq;
    int err = 0;

#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
        const uint16_t **keys = (const uint16_t **)malloc(sizeof(void *) * (size_t)(maxlen > 0 ? maxlen : 1));
        const uint16_t **vals = (const uint16_t **)malloc(sizeof(void *) * (size_t)(maxlen > 0 ? maxlen : 1));
        if (!z || !keys || !vals) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t w = 0; w < pairs; ++w) {
                const int32_t i = (int32_t)(w / Hq);
                const int32_t h = (int32_t)(w % Hq);
                const int32_t kh = h / g;
                const int64_t s0 = cu[i];
                const int64_t L = (int64_t)cu[i + 1] - s0;
                for (int64_t j = 0; j < L; ++j) {
                    keys[j] = k + ((s0 + j) * Hkv + kh) * d;
                    vals[j] = v + ((s0 + j) * Hkv + kh) * d;
                }
                for (int64_t p = 0; p < L; ++p) {
                    const int64_t row = s0 + p;
                    attend_row(q + (row * Hq + h) * d, keys, vals, p + 1, d, scale, z,
                               out + (row * Hq + h) * d, lse ? lse + row * Hq + h : NULL);
                }
            }
        }
        free(z);
        free((void *)keys);
        free((void *)vals);
    }
    return err ? -2 : 0;
}

/*
 * Attention of each sequence's last valid token only (abstract and section
 * 1.1: a Prefill-Only request needs the next-token logits at the last valid
 * position of each sequence, so the last layer's attention is needed for that
 * one row): for sequence i of length L >= 1 and query head h,
 *   out[i, h] = softmax(scale q[i, h] . k_j) v_j  over the sequence's L keys,
 * i.e. row L-1 of the causal prefill.  Zero-length sequences write nothing.
 *
 *   q   : bf16 [B, Hq, d]   the last row of each sequence
 *   k, v: bf16 [T, Hkv, d]  packed by cu (int32 [B+1], cu[0] = 0, non-decreasing)
 *   out : double [B, Hq, d]  lse : double [B, Hq] or NULL
 */
int oracle_last_token(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const int32_t *cu, int32_t B, int32_t Hq, int32_t Hkv,
                      int32_t d, double scale, double *out, double *lse)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return -1;
    if (B > 0 && cu[0] != 0) return -1;
    int64_t maxlen = 0;
    for (int32_t i = 0; i < B; ++i) {
        if (cu[i + 1] < cu[i]) return -1;
        if (cu[i + 1] - cu[i] > maxlen) maxlen = cu[i + 1] - cu[i];
    }
    const int32_t g = Hq / Hkv;
    const int64_t pairs = (int64_t)B * Hq;
    int err = 0;

#pragma omp parallel
    {
        const size_t n = (size_t)(maxlen > 0 ? maxlen : 1);
        double *z = (double *)malloc(sizeof(double) * n);
        const uint16_t **keys = (const uint16_t **)malloc(sizeof(void *) * n);
        const uint16_t **vals = (const uint16_t **)malloc(sizeof(void *) * n);
        if (!z || !keys || !vals) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t w = 0; w < pairs; ++w) {
                const int32_t i = (int32_t)(w / Hq);
                const int32_t h = (int32_t)(w % Hq);
                const int32_t kh = h / g;
                const int64_t s0 = cu[i];
                const int64_t L = (int64_t)cu[i + 1] - s0;
                if (L == 0) continue;
                for (int64_t j = 0; j < L; ++j) {
                    keys[j] = k + ((s0 + j) * Hkv + kh) * d;
                    vals[j] = v + ((s0 + j) * Hkv + kh) * d;
                }
                attend_row(q + ((int64_t)i * Hq + h) * d, keys, vals, L, d, scale, z,
                           out + ((int64_t)i * Hq + h) * d, lse ? lse + (int64_t)i * Hq + h : NULL);
            }
        }
        free(z);
        free((void *)keys);
        free((void *)vals);
    }
    return err ? -2 : 0;
}

/*
 * Beam-search decode attention over a shared prompt K/V and per-beam
 * suffixes (section 1.2: the beams of one request share a single prompt
 * K/V, each beam keeps its own short suffix K/V).
 *
 *   q          : bf16 [R, W, Hq, d]      query of the newest position
 *   pk, pv     : bf16 [sum_r P_r, Hkv, d] prompt K/V, request r at rows
 *                cu_prompt[r] .. cu_prompt[r+1]-1
 *   hk, hv     : bf16 [R, W, t, Hkv, d]  the beam's own suffix history, in
 *                order (already the parent-gathered history of this beam)
 *   t          : suffix length (>= 0); P_r + t >= 1 for every request
 *   out        : double [R, W, Hq, d]
 * Keys of (r, b) are the concatenation [prompt_r ; suffix(r, b)]; no mask.
 */
int oracle_decode(const uint16_t *q, const uint16_t *pk, const uint16_t *pv,
                  const int32_t *cu_prompt, const uint16_t *hk, const uint16_t *hv,
                  int32_t t, int32_t R, int32_t W, int32_t Hq, int32_t Hkv, int32_t d,
                  double scale, double *out, double *lse)
{
    if (R < 0 || W <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || t < 0 || Hq % Hkv != 0) return -1;
    if (R > 0 && cu_prompt[0] != 0) return -1;
    int64_t maxp = 0;
    for (int32_t r = 0; r < R; ++r) {
        const int64_t P = (int64_t)cu_prompt[r + 1] - cu_prompt[r];
        if (P < 0) return -1;
        if (P + t < 1) return -1;          /* empty softmax is undefined */
        if (P > maxp) maxp = P;
    }
    const int32_t g = Hq / Hkv;
    const int64_t nmax = maxp + t;
    const int64_t units = (int64_t)R * W * Hq;
    int err = 0;

#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)(nmax > 0 ? nmax : 1));
        const uint16_t **keys = (const uint16_t **)malloc(sizeof(void *) * (size_t)(nmax > 0 ? nmax : 1));
        const uint16_t **vals = (const uint16_t **)malloc(sizeof(void *) * (size_t)(nmax > 0 ? nmax : 1));
        if (!z || !keys || !vals) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t u = 0; u < units; ++u) {
                const int32_t h = (int32_t)(u % Hq);
                const int64_t rb = u / Hq;          /* r * W + b */
                const int32_t r = (int32_t)(rb / W);
                const int32_t kh = h / g;
                const int64_t p0 = cu_prompt[r];
                const int64_t P = (int64_t)cu_prompt[r + 1] - p0;
                for (int64_t j = 0; j < P; ++j) {
                    keys[j] = pk + ((p0 + j) * Hkv + kh) * d;
                    vals[j] = pv + ((p0 + j) * Hkv + kh) * d;
                }
                for (int64_t s = 0; s < t; ++s) {
                    keys[P + s] = hk + ((rb * t + s) * Hkv + kh) * d;
                    vals[P + s] = hv + ((rb * t + s) * Hkv + kh) * d;
                }
                attend_row(q + (rb * Hq + h) * d, keys, vals, P + t, d, scale, z,
                           out + (rb * Hq + h) * d, lse ? lse + rb * Hq + h : NULL);
            }
        }
        free(z);
        free((void *)keys);
        free((void *)vals);
    }
    return err ? -2 : 0;
}

/* Number of threads the OpenMP runtime will use (reported with timings). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
