/*
 * CPU oracle for attention over a latent (MLA) cache -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, the smoke check and the benchmark's cpu_baseline / reference
 * arm may load this file's library.  It shares no code with the CUDA path.
 *
 * What it computes is the plain definition of absorbed-query attention over
 * one shared latent (issue #1313, "Step 2", the decode bullet: every head's
 * absorbed query is read against the same latent rows; issue #1142, "What
 * happens now": 512 latent values a row plus the rope part), over CONTIGUOUS
 * rows in token order, with no pages, no tiling, no splitting:
 *
 *   for query row r at position p = len - R + r and head h,
 *     s_j  = scale * ( sum_{d<512} q[d] * C[j][d] + sum_{e<64} q[512+e] * Kr[j][e] ),  j = 0..p
 *     w_j  = exp(s_j - max s) / sum_i exp(s_i - max s)
 *     o[d] = sum_j w_j * C[j][d]                     (the value is the latent itself)
 *     lse  = max s + log sum_j exp(s_j - max s)
 *
 * Causality (a row sees keys up to and including its own position) follows the
 * MTP reading of PR #1732 ("What this changes": a lookahead of 1, the draft row
 * reads the token after a mark) and the chunked-prefill note (section 1: a
 * chunk's T rows against the prefix L plus the rows before them in the chunk).
 *
 * Inputs are bf16 bit patterns widened exactly to double; every sum is a plain
 * left-to-right double sum.  Independent (row, head) items run on OpenMP
 * threads; each item is computed alone, so threading does not change a bit.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define LAT 512
#define ROPE 64
#define DK (LAT + ROPE)

static double widen(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * One stream.  q: [R][H][576] bf16 bits; lat: [len][512]; rope: [len][64]
 * (contiguous logical rows).  items: n_items indices r*H + h to evaluate.
 * out: [n_items][512] doubles; lse: [n_items] doubles.
 * Returns 0, or -1 on a bad argument (a row with no visible key, an item outside [0, R*H)).
 */
static int attend_core(int64_t len, int32_t R, int32_t H,
                       const uint16_t *q, const uint16_t *lat, const double *latd, const uint16_t *rope,
                       double scale, int32_t n_items, const int32_t *items,
                       double *out, double *lse, int32_t n_threads);

int oracle_mla_attend(int64_t len, int32_t R, int32_t H,
                      const uint16_t *q, const uint16_t *lat, const uint16_t *rope,
                      double scale, int32_t n_items, const int32_t *items,
                      double *out, double *lse, int32_t n_threads)
{
    return attend_core(len, R, H, q, lat, NULL, rope, scale, n_items, items, out, lse, n_threads);
}

/*
 * The same definition with the latent given as doubles [len][512] (the dequantized
 * values of FP8 rows: issue #1313, step 1.3, item 3); q and rope as above.
 */
int oracle_mla_attend_f64(int64_t len, int32_t R, int32_t H,
                          const uint16_t *q, const double *latd, const uint16_t *rope,
                          double scale, int32_t n_items, const int32_t *items,
                          double *out, double *lse, int32_t n_threads)
{
    return attend_core(len, R, H, q, NULL, latd, rope, scale, n_items, items, out, lse, n_threads);
}

#define LAT_AT(j, d) (latd ? latd[(j) * LAT + (d)] : widen(lat[(j) * LAT + (d)]))

static int attend_core(int64_t len, int32_t R, int32_t H,
                       const uint16_t *q, const uint16_t *lat, const double *latd, const uint16_t *rope,
                       double scale, int32_t n_items, const int32_t *items,
                       double *out, double *lse, int32_t n_threads)
{
    if (len < R || R < 1 || H < 1)
        return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads > 0 ? n_threads : 1) reduction(| : bad)
    for (int32_t it = 0; it < n_items; ++it) {
        if (items[it] < 0 || (int64_t)items[it] >= (int64_t)R * H) { bad = 1; continue; }
        int32_t r = items[it] / H, h = items[it] % H;
        int64_t p = len - R + r;               /* this row's position: keys 0..p are visible */
        int64_t nk = p + 1;
        double qd[DK];
        for (int d = 0; d < DK; ++d)
            qd[d] = widen(q[((int64_t)r * H + h) * DK + d]);
        double *s = (double *)malloc((size_t)nk * sizeof(double));
        if (!s) { bad = 1; continue; }
        double m = -INFINITY;
        for (int64_t j = 0; j < nk; ++j) {
            double dot = 0.0;
            for (int d = 0; d < LAT; ++d)
                dot += qd[d] * LAT_AT(j, d);
            for (int e = 0; e < ROPE; ++e)
                dot += qd[LAT + e] * widen(rope[j * ROPE + e]);
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
        }
        double sum = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
            s[j] = exp(s[j] - m);
            sum += s[j];
        }
        double acc[LAT];
        for (int d = 0; d < LAT; ++d) acc[d] = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
            double w = s[j] / sum;
            for (int d = 0; d < LAT; ++d)
                acc[d] += w * LAT_AT(j, d);
        }
        for (int d = 0; d < LAT; ++d)
            out[(int64_t)it * LAT + d] = acc[d];
        lse[it] = m + log(sum);
        free(s);
    }
    return bad ? -1 : 0;
}
