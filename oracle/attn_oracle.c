/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for exact attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes (per query row, written out from the definition):
 *
 *   s_j   = scale * sum_c q[i,c] * k[j,c]      for every key j the row may see
 *   M     = max_j s_j
 *   L     = sum_j exp(s_j - M)
 *   o[c]  = sum_j exp(s_j - M) * v[j,c] / L
 *   lse   = M + ln L
 *
 * This is softmax(Q K^T * scale [+ causal mask]) V, the fused operation the
 * IO-aware tiling pages describe ("FlashAttention-4 中的 IO 感知块分块策略",
 * opening section: tiling reaches the same result as the plain softmax with no
 * loss of exactness), so the oracle is that plain definition, materialising
 * one whole score row at a time in double precision.  Inputs are bf16 bit
 * patterns, widened to double exactly.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - causal alignment is bottom-right: key j is visible to row i iff
 *     j <= i + Sk - Sq (the last query sees every key; decode is Sq = 1);
 *   - a row that sees no key returns o = 0 and lse = -inf;
 *   - the grouped-query head map is contiguous: kv head = h / (Hq / Hkv);
 *   - layouts: BSHD = [B][S][H][d], BHSD = [B][H][S][d], dense.
 *
 * Also here, for the pins: the online-softmax recurrence over key tiles
 * (running max m and running sum l, m' = max(m, m_new),
 * l' = l * exp(m - m') + l_new, from the same IO-aware tiling page, section
 * "具体而言"), the log-sum-exp merge of key-range partials (the Flash-Decoding
 * style tail split of the MoonMath HIP kernel page), and paged-KV decode with
 * an int32 block table (the ROCm port page, "Vendor-Agnostic 多查询推理优化").
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <tgmath.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/*
 * The number type of the whole-row definition (attend_row, behind
 * oracle_attention and oracle_attention_rows).  Double unless built with
 * -DORACLE_REAL=float: the test suite builds that single-precision copy only
 * to check that the fp64 results sit far inside the parity tolerance of any
 * rounding of the same steps (an oracle whose numbers depended on the last
 * bits of its arithmetic could not judge a bf16 kernel).  <tgmath.h> makes
 * exp and log follow the argument's type.
 */
#ifndef ORACLE_REAL
#define ORACLE_REAL double
#endif
typedef ORACLE_REAL oreal;

#define ORACLE_OK 0
#define ORACLE_BAD_ARG -1
#define ORACLE_NO_MEMORY -2

/* bf16 is the top half of an IEEE binary32: widening is exact. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Element offset of (b, s, h, c) in a dense tensor of the given layout. */
static int64_t offset_of(int layout, int64_t b, int64_t s, int64_t h, int64_t c,
                         int64_t S, int64_t H, int64_t d) {
    if (layout == 0) return ((b * S + s) * H + h) * d + c;  /* BSHD */
    return ((b * H + h) * S + s) * d + c;                   /* BHSD */
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Last key index row i may see (inclusive); -1 when it sees none. */
static int64_t last_visible_key(int causal, int64_t i, int64_t Sq, int64_t Sk) {
    int64_t last = Sk - 1;
    if (causal) {
        int64_t lim = i + Sk - Sq;
        if (lim < last) last = lim;
    }
    return last < -1 ? -1 : last;
}

typedef struct {
    const uint16_t *q, *k, *v;
    int64_t B, Hq, Hkv, Sq, Sk, d;
    int layout, causal;
    double scale;
} problem_t;

static int check_problem(const problem_t *p) {
    if (!p->q || !p->k || !p->v) return ORACLE_BAD_ARG;
    if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->Sq < 1 || p->Sk < 1 || p->d < 1) return ORACLE_BAD_ARG;
    if (p->Hq % p->Hkv != 0) return ORACLE_BAD_ARG;
    if (p->layout != 0 && p->layout != 1) return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

/*
 * One query row over the keys [klo, khi) that it may see, straight from the
 * definition.  scores: scratch of at least Sk values; acc: scratch of d
 * values.  Writes d outputs and the row's log-sum-exp.  (bf16 inputs are
 * exact in either number type.)
 */
static void attend_row(const problem_t *p, int64_t b, int64_t h, int64_t i,
                       int64_t klo, int64_t khi, oreal *scores, oreal *acc,
                       double *o, double *lse) {
    const int64_t g = h / (p->Hq / p->Hkv);
    const int64_t d = p->d;
    int64_t last = last_visible_key(p->causal, i, p->Sq, p->Sk);
    if (khi > last + 1) khi = last + 1;
    if (klo < 0) klo = 0;
    for (int64_t c = 0; c < d; ++c) acc[c] = 0.0;
    if (khi <= klo) {
        for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    oreal M = -INFINITY;
    for (int64_t j = klo; j < khi; ++j) {
        oreal dot = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            oreal qv = (oreal)bf16_to_double(p->q[offset_of(p->layout, b, i, h, c, p->Sq, p->Hq, d)]);
            oreal kv = (oreal)bf16_to_double(p->k[offset_of(p->layout, b, j, g, c, p->Sk, p->Hkv, d)]);
            dot += qv * kv;
        }
        scores[j] = (oreal)p->scale * dot;
        if (scores[j] > M) M = scores[j];
    }
    oreal L = 0.0;
    for (int64_t j = klo; j < khi; ++j) {
        oreal w = exp(scores[j] - M);
        L += w;
        for (int64_t c = 0; c < d; ++c)
            acc[c] += w * (oreal)bf16_to_double(p->v[offset_of(p->layout, b, j, g, c, p->Sk, p->Hkv, d)]);
    }
    for (int64_t c = 0; c < d; ++c) o[c] = acc[c] / L;
    *lse = M + log(L);
}

/*
 * Whole problem.  out: doubles in q's layout ([B,Sq,Hq,d] or [B,Hq,Sq,d]);
 * lse: [B,Hq,Sq] doubles (may be NULL).
 */
int oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t d,
                     int layout, int causal, double scale, double *out, double *lse) {
    problem_t p = {q, k, v, B, Hq, Hkv, Sq, Sk, d, layout, causal, scale};
    int rc = check_problem(&p);
    if (rc != ORACLE_OK || !out) return ORACLE_BAD_ARG;
    const int64_t nrows = B * Hq * Sq;
    int failed = 0;
#pragma omp parallel
    {
        oreal *scores = (oreal *)malloc(sizeof(oreal) * (size_t)Sk);
        oreal *acc = (oreal *)malloc(sizeof(oreal) * (size_t)d);
        double *orow = (double *)malloc(sizeof(double) * (size_t)d);
        if (!scores || !acc || !orow) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < nrows; ++r) {
                int64_t b = r / (Hq * Sq), h = (r / Sq) % Hq, i = r % Sq;
                double l;
                attend_row(&p, b, h, i, 0, Sk, scores, acc, orow, &l);
                for (int64_t c = 0; c < d; ++c) out[offset_of(layout, b, i, h, c, Sq, Hq, d)] = orow[c];
                if (lse) lse[(b * Hq + h) * Sq + i] = l;
            }
        }
        free(scores);
        free(acc);
        free(orow);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Selected rows only, each restricted to keys [klo, khi).  rows: n triples
 * (b, h, i).  out: [n, d]; lse: [n].  With klo = 0, khi = Sk this is the
 * full definition for those rows; a narrower range gives a key-range partial
 * (normalised within the range) for the split/merge pin.
 */
int oracle_attention_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t d,
                          int layout, int causal, double scale,
                          int64_t n, const int64_t *rows, int64_t klo, int64_t khi,
                          double *out, double *lse) {
    problem_t p = {q, k, v, B, Hq, Hkv, Sq, Sk, d, layout, causal, scale};
    int rc = check_problem(&p);
    if (rc != ORACLE_OK || !rows || !out || !lse || n < 0) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < n; ++r) {
        const int64_t *t = rows + 3 * r;
        if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= Hq || t[2] < 0 || t[2] >= Sq) return ORACLE_BAD_ARG;
    }
    int failed = 0;
#pragma omp parallel
    {
        oreal *scores = (oreal *)malloc(sizeof(oreal) * (size_t)Sk);
        oreal *acc = (oreal *)malloc(sizeof(oreal) * (size_t)d);
        if (!scores || !acc) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < n; ++r) {
                const int64_t *t = rows + 3 * r;
                attend_row(&p, t[0], t[1], t[2], klo, khi, scores, acc, out + r * d, lse + r);
            }
        }
        free(scores);
        free(acc);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * The softmax probabilities of one row (P_ij for every key j, zero where
 * masked), for the "rows of P sum to one" pin.
 */
int oracle_attention_probs_row(const uint16_t *q, const uint16_t *k,
                               int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t d,
                               int layout, int causal, double scale,
                               int64_t b, int64_t h, int64_t i, double *probs) {
    problem_t p = {q, k, q, B, Hq, Hkv, Sq, Sk, d, layout, causal, scale};
    if (check_problem(&p) != ORACLE_OK || !probs) return ORACLE_BAD_ARG;
    if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Sq) return ORACLE_BAD_ARG;
    const int64_t g = h / (Hq / Hkv);
    int64_t last = last_visible_key(causal, i, Sq, Sk);
    double M = -INFINITY;
    for (int64_t j = 0; j < Sk; ++j) {
        probs[j] = 0.0;
        if (j > last) continue;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c)
            dot += bf16_to_double(q[offset_of(layout, b, i, h, c, Sq, Hq, d)]) *
                   bf16_to_double(k[offset_of(layout, b, j, g, c, Sk, Hkv, d)]);
        probs[j] = scale * dot;
        if (probs[j] > M) M = probs[j];
    }
    double L = 0.0;
    for (int64_t j = 0; j <= last; ++j) L += exp(probs[j] - M);
    for (int64_t j = 0; j <= last; ++j) probs[j] = exp(probs[j] - M) / L;
    return ORACLE_OK;
}

/*
 * The online-softmax recurrence itself, in fp64, over key tiles of `tile`
 * keys: for each tile the scores are formed, the running max and running sum
 * are updated with m' = max(m, m_tile), l' = l * exp(m - m') + sum exp(s - m'),
 * and the output accumulator is rescaled by exp(m - m') before the tile's
 * contribution is added.  The final output is acc / l and lse = m + ln l.
 * Used only to pin that the recurrence equals the full softmax.
 */
int oracle_attention_tiled_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t d,
                                int layout, int causal, double scale, int64_t tile,
                                int64_t n, const int64_t *rows, double *out, double *lse) {
    problem_t p = {q, k, v, B, Hq, Hkv, Sq, Sk, d, layout, causal, scale};
    if (check_problem(&p) != ORACLE_OK || tile < 1 || !rows || !out || !lse || n < 0) return ORACLE_BAD_ARG;
    double *s = (double *)malloc(sizeof(double) * (size_t)tile);
    if (!s) return ORACLE_NO_MEMORY;
    for (int64_t r = 0; r < n; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Sq) { free(s); return ORACLE_BAD_ARG; }
        const int64_t g = h / (Hq / Hkv);
        const int64_t last = last_visible_key(causal, i, Sq, Sk);
        double *acc = out + r * d;
        for (int64_t c = 0; c < d; ++c) acc[c] = 0.0;
        double m = -INFINITY, l = 0.0;
        for (int64_t j0 = 0; j0 <= last; j0 += tile) {
            int64_t j1 = j0 + tile - 1;
            if (j1 > last) j1 = last;
            double m_tile = -INFINITY;
            for (int64_t j = j0; j <= j1; ++j) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += bf16_to_double(q[offset_of(layout, b, i, h, c, Sq, Hq, d)]) *
                           bf16_to_double(k[offset_of(layout, b, j, g, c, Sk, Hkv, d)]);
                s[j - j0] = scale * dot;
                if (s[j - j0] > m_tile) m_tile = s[j - j0];
            }
            double m_new = m > m_tile ? m : m_tile;
            double corr = (m == -INFINITY) ? 0.0 : exp(m - m_new);
            double l_tile = 0.0;
            for (int64_t c = 0; c < d; ++c) acc[c] *= corr;
            for (int64_t j = j0; j <= j1; ++j) {
                double w = exp(s[j - j0] - m_new);
                l_tile += w;
                for (int64_t c = 0; c < d; ++c)
                    acc[c] += w * bf16_to_double(v[offset_of(layout, b, j, g, c, Sk, Hkv, d)]);
            }
            l = l * corr + l_tile;
            m = m_new;
        }
        if (l > 0.0) {
            for (int64_t c = 0; c < d; ++c) acc[c] /= l;
            lse[r] = m + log(l);
        } else {
            lse[r] = -INFINITY;
        }
    }
    free(s);
    return ORACLE_OK;
}

/*
 * Log-sum-exp merge of `nsplit` key-range partials, each normalised within
 * its own range: lse = M + ln sum_s exp(lse_s - M) with M = max_s lse_s, and
 * o = sum_s exp(lse_s - lse) * o_s.  lse_s: [nsplit][n]; o_s: [nsplit][n][d];
 * out: [n][d]; lse: [n].  A partial with lse_s = -inf contributes nothing; if
 * every partial is empty the row is o = 0, lse = -inf.
 */
int oracle_lse_merge(int64_t nsplit, int64_t n, int64_t d, const double *lse_s,
                     const double *o_s, double *out, double *lse) {
    if (nsplit < 1 || n < 0 || d < 1 || !lse_s || !o_s || !out || !lse) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < n; ++r) {
        double M = -INFINITY;
        for (int64_t s = 0; s < nsplit; ++s)
            if (lse_s[s * n + r] > M) M = lse_s[s * n + r];
        for (int64_t c = 0; c < d; ++c) out[r * d + c] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int64_t s = 0; s < nsplit; ++s) sum += exp(lse_s[s * n + r] - M);
        double total = M + log(sum);
        for (int64_t s = 0; s < nsplit; ++s) {
            double w = exp(lse_s[s * n + r] - total);
            if (w == 0.0) continue;
            for (int64_t c = 0; c < d; ++c) out[r * d + c] += w * o_s[(s * n + r) * d + c];
        }
        lse[r] = total;
    }
    return ORACLE_OK;
}

/*
 * Paged-KV decode: one query per (sequence, head), keys 0 .. seqlen_b - 1 of
 * sequence b.  Key t of sequence b lives in physical page
 * block_table[b][t / page_size], slot t % page_size; the page pool is
 * [num_pages][page_size][Hkv][d] for K and V.  q: [B][Hq][d]; out: [B][Hq][d]
 * doubles; lse: [B][Hq].  Block-table entries past the sequence's last page
 * are never read.  Returns ORACLE_BAD_ARG if a needed entry is out of range.
 */
int oracle_decode_paged(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                        const int32_t *block_table, const int32_t *seqlens,
                        int64_t B, int64_t Hq, int64_t Hkv, int64_t d,
                        int64_t page_size, int64_t num_pages, int64_t max_blocks,
                        double scale, double *out, double *lse) {
    if (!q || !k_pages || !v_pages || !block_table || !seqlens || !out || !lse) return ORACLE_BAD_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || d < 1 || page_size < 1 || num_pages < 1 || max_blocks < 1) return ORACLE_BAD_ARG;
    if (Hq % Hkv != 0) return ORACLE_BAD_ARG;
    for (int64_t b = 0; b < B; ++b) {
        int64_t L = seqlens[b];
        if (L < 0 || L > page_size * max_blocks) return ORACLE_BAD_ARG;
        for (int64_t pg = 0; pg < (L + page_size - 1) / page_size; ++pg) {
            int32_t phys = block_table[b * max_blocks + pg];
            if (phys < 0 || phys >= num_pages) return ORACLE_BAD_ARG;
        }
    }
    const int64_t G = Hq / Hkv;
    int failed = 0;
#pragma omp parallel
    {
        int64_t cap = page_size * max_blocks;
        double *scores = (double *)malloc(sizeof(double) * (size_t)cap);
        if (!scores) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < B * Hq; ++r) {
                int64_t b = r / Hq, h = r % Hq, g = h / G;
                int64_t L = seqlens[b];
                double *o = out + r * d;
                for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
                if (L == 0) {
                    lse[r] = -INFINITY;
                    continue;
                }
                double M = -INFINITY;
                for (int64_t t = 0; t < L; ++t) {
                    int64_t phys = block_table[b * max_blocks + t / page_size];
                    int64_t base = ((phys * page_size + t % page_size) * Hkv + g) * d;
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c)
                        dot += bf16_to_double(q[r * d + c]) * bf16_to_double(k_pages[base + c]);
                    scores[t] = scale * dot;
                    if (scores[t] > M) M = scores[t];
                }
                double sum = 0.0;
                for (int64_t t = 0; t < L; ++t) {
                    int64_t phys = block_table[b * max_blocks + t / page_size];
                    int64_t base = ((phys * page_size + t % page_size) * Hkv + g) * d;
                    double w = exp(scores[t] - M);
                    sum += w;
                    for (int64_t c = 0; c < d; ++c) o[c] += w * bf16_to_double(v_pages[base + c]);
                }
                for (int64_t c = 0; c < d; ++c) o[c] /= sum;
                lse[r] = M + log(sum);
            }
        }
        free(scores);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Round a double to bf16 in one of the three output rounding modes the
 * MoonMath HIP kernel page lists for its bf16 output (benchmark and
 * limitations sections): 0 = RTNE (to nearest, ties to even), 1 = RTNA (to
 * nearest, ties away from zero), 2 = RTZ (toward zero).  Returns the bit
 * pattern.  Written from the definition of the format (8 exponent bits, 8
 * significant bits): the quantum at the value's binade is 2^(e-8) (never below
 * the subnormal quantum 2^-133); the magnitude divided by the quantum is
 * rounded to an integer by nearbyint (default mode: ties to even), round
 * (ties away from zero) or trunc; times the quantum again it is exactly
 * representable in binary32, whose top 16 bits are the bf16 pattern.  One
 * rounding step only, from the double itself.  NaN becomes the quiet NaN
 * 0x7fc0.  Past the largest finite bf16, the nearest modes give infinity and
 * RTZ gives the largest finite value; an infinite input stays infinite.
 */
uint16_t oracle_round_bf16(double x, int mode) {
    if (isnan(x)) return 0x7fc0u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double ax = fabs(x);
    double r = 0.0;
    if (isinf(ax)) {
        r = ax;
    } else if (ax > 0.0) {
        int e;
        frexp(ax, &e); /* ax = m * 2^e, m in [0.5, 1) */
        int qexp = e - 8;
        if (qexp < -133) qexp = -133;
        double units = ldexp(ax, -qexp);
        double n = mode == 1 ? round(units) : mode == 2 ? trunc(units) : nearbyint(units);
        r = ldexp(n, qexp);
        if (mode == 2 && r > 0x1.fep127) r = 0x1.fep127; /* RTZ never overflows */
    }
    float f = (float)r; /* exact, or +inf past the bf16 range */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

uint16_t oracle_round_bf16_rtne(double x) { return oracle_round_bf16(x, 0); }

/* Element-wise oracle_round_bf16 over n doubles. */
int oracle_round_bf16_array(const double *x, uint16_t *out, int64_t n, int mode) {
    if (mode < 0 || mode > 2) return ORACLE_BAD_ARG;
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(x[i], mode);
    return ORACLE_OK;
}
