/*
 * kv8_oracle.c -- CPU oracle for the fp8 e4m3 latent KV cache and absorbed MLA
 * decode attention.  TEST INFRASTRUCTURE ONLY (see kv8_oracle.h).
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -fPIC -shared (never -ffast-math:
 * the quantizer must round every f32 operation exactly once, and an f32 a*b+c
 * must not be fused).
 *
 * "The KV8 page" = the pull-request page "KV8=1: fp8 e4m3 latent KV cache
 * (CPU + CUDA) with .coli_kv v2".
 */
#include "kv8_oracle.h"

#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* e4m3 decode.  KV8 page, PR description, c/kv_fp8.h item: a decode table of
 * all 256 codes.  The table is filled from the closed form of the OCP e4m3fn format:
 *   sign s = bit 7, exponent e = bits 6..3 (bias 7), mantissa m = bits 2..0;
 *   e = 15, m = 7        -> NaN (codes 0x7F and 0xFF; there is no infinity);
 *   e = 0                -> (-1)^s * m * 2^-9           (subnormals, and +-0);
 *   otherwise            -> (-1)^s * 2^(e-7) * (1 + m/8).                       */
static float g_lut[256];
static int g_lut_ready = 0;

static float e4m3_closed_form(unsigned c) {
    unsigned s = (c >> 7) & 1u, e = (c >> 3) & 15u, m = c & 7u;
    float v;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u) v = ldexpf((float)m, -9);
    else v = ldexpf((float)(8u + m), (int)e - 10); /* (8+m)*2^(e-10) = 2^(e-7)(1+m/8) */
    return s ? -v : v;
}

static void lut_init(void) {
    if (g_lut_ready) return;
    for (unsigned c = 0; c < 256u; ++c) g_lut[c] = e4m3_closed_form(c);
    g_lut_ready = 1;
}

float orc_e4m3_decode(uint8_t code) {
    lut_init();
    return g_lut[code];
}

void orc_e4m3_decode_table(float out[256]) {
    lut_init();
    memcpy(out, g_lut, sizeof(g_lut));
}

/* ------------------------------------------------------------------------ */
/* e4m3 encode.  KV8 page, PR description, c/kv_fp8.h item: an encoder on the bit
 * pattern with round-to-nearest-even that saturates at +/-448, keeps the sign of
 * zero and stores NaN as the code 0.  Works on the f32 bit pattern with integer arithmetic only.                   */
uint8_t orc_e4m3_encode(float q) {
    uint32_t u;
    memcpy(&u, &q, sizeof u);
    const uint32_t sign = (u >> 24) & 0x80u;
    const uint32_t mag = u & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) return 0x00u;              /* NaN -> inert zero          */
    if (mag >= 0x43E00000u) return (uint8_t)(sign | 0x7Eu); /* |q| >= 448, incl. inf */
    const uint32_t E = mag >> 23, M = mag & 0x7FFFFFu;
    if (E >= 121u) {
        /* |q| >= 2^-6: a normal e4m3 target with exponent field E - 120 in [1, 15].
         * Keep the top 3 mantissa bits, round the 20 dropped bits to nearest even;
         * a carry out of the mantissa moves into the exponent by plain addition.  */
        uint32_t code = ((E - 120u) << 3) | (M >> 20);
        const uint32_t rest = M & 0xFFFFFu, half = 0x80000u;
        if (rest > half || (rest == half && (code & 1u))) code += 1u;
        return (uint8_t)(sign | code); /* |q| < 448 keeps code <= 0x7E */
    }
    /* |q| < 2^-6: target is k * 2^-9 with integer k in [0, 8] (k = 8 is the
     * smallest normal, 0x08).  |q| = sig * 2^(max(E,1) - 150), so
     * |q| * 2^9 = sig * 2^-(141 - max(E,1)).                                    */
    const uint32_t sig = E ? (M | 0x800000u) : M;
    const uint32_t shift = 141u - (E ? E : 1u); /* >= 21 */
    if (shift >= 26u) return (uint8_t)sign;     /* sig < 2^24 -> value < 2^-2 -> k = 0 */
    uint32_t k = sig >> shift;
    const uint32_t rest = sig & ((1u << shift) - 1u), half = 1u << (shift - 1u);
    if (rest > half || (rest == half && (k & 1u))) k += 1u;
    return (uint8_t)(sign | k);
}

/* Brute-force nearest encoder: scan every non-negative finite code and keep the
 * one nearest to |q|, ties to the code with an even mantissa LSB.  The
 * differences are formed in double; for the two codes that bracket |q| they are
 * exact (Sterbenz, or a subtraction of zero), which is all a tie decision needs. */
uint8_t orc_e4m3_encode_nearest(float q) {
    lut_init();
    if (isnan(q)) return 0x00u;
    const uint8_t sign = signbit(q) ? 0x80u : 0x00u;
    const double a = fabs((double)q);
    if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);
    unsigned best = 0;
    double best_d = INFINITY;
    for (unsigned c = 0; c <= 0x7Eu; ++c) {
        const double d = fabs(a - (double)g_lut[c]);
        if (d < best_d || (d == best_d && (c & 1u) == 0u)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* Bracket encoder: binary search for the pair of adjacent codes around |q| and
 * compare with their exact midpoint (5 significant bits: exact in f32). */
uint8_t orc_e4m3_encode_bracket(float q) {
    lut_init();
    if (isnan(q)) return 0x00u;
    const uint8_t sign = signbit(q) ? 0x80u : 0x00u;
    const float a = fabsf(q);
    if (a >= 448.0f) return (uint8_t)(sign | 0x7Eu);
    unsigned lo = 0, hi = 0x7Eu; /* g_lut[lo] <= a < g_lut[hi] */
    while (hi - lo > 1u) {
        const unsigned mid = (lo + hi) / 2u;
        if (g_lut[mid] <= a) lo = mid;
        else hi = mid;
    }
    const float midpoint = 0.5f * (g_lut[lo] + g_lut[hi]);
    unsigned c;
    if (a < midpoint) c = lo;
    else if (a > midpoint) c = hi;
    else c = (lo & 1u) ? hi : lo;
    return (uint8_t)(sign | c);
}

void orc_e4m3_encode_array(const float* x, int64_t n, uint8_t* out, int which) {
    lut_init();
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = which == 0 ? orc_e4m3_encode(x[i])
                 : which == 1 ? orc_e4m3_encode_nearest(x[i])
                              : orc_e4m3_encode_bracket(x[i]);
}

int64_t orc_e4m3_exhaustive_mismatches(uint64_t lo, uint64_t hi, uint32_t* first_bad) {
    lut_init();
    int64_t bad = 0;
    uint64_t first = UINT64_MAX;
#pragma omp parallel for schedule(static) reduction(+ : bad) reduction(min : first)
    for (int64_t i = (int64_t)lo; i < (int64_t)hi; ++i) {
        const uint32_t u = (uint32_t)i;
        float f;
        memcpy(&f, &u, sizeof f);
        if (orc_e4m3_encode(f) != orc_e4m3_encode_bracket(f)) {
            ++bad;
            if ((uint64_t)i < first) first = (uint64_t)i;
        }
    }
    if (first_bad) *first_bad = (first == UINT64_MAX) ? 0u : (uint32_t)first;
    return bad;
}

int64_t orc_e4m3_list_mismatches_nearest(const uint32_t* bits, int64_t n, uint32_t* first_bad) {
    lut_init();
    int64_t bad = 0;
    int64_t first = n;
#pragma omp parallel for schedule(static) reduction(+ : bad) reduction(min : first)
    for (int64_t i = 0; i < n; ++i) {
        float f;
        memcpy(&f, &bits[i], sizeof f);
        if (orc_e4m3_encode(f) != orc_e4m3_encode_nearest(f)) {
            ++bad;
            if (i < first) first = i;
        }
    }
    if (first_bad) *first_bad = (first < n) ? bits[first] : 0u;
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Per-row quantizer.  KV8 page, PR description and expanded summary: each of Lc
 * and Rc gets its own f32 scale amax/448; c/kv_fp8.h item: a guard for rows whose
 * amax is so small (subnormal) that 448/amax overflows to +inf.  Steps, for each segment (Lc: 512 values, Rc: 64 values):
 *   1. amax = max |x_i| over the non-NaN entries (0 if there are none);
 *   2. s = amax / 448 (f32, rounded once) is the stored scale;
 *   3. inv = 448 / amax (f32, rounded once);
 *   4. guard: if inv is not finite (amax = 0, or amax < 448/FLT_MAX, which
 *      includes every subnormal amax) every code is a signed zero (NaN -> 0x00);
 *      otherwise code_i = encode(x_i * inv), the product rounded once.           */
static void quantize_segment(const float* x, int n, uint8_t* codes, float* scale) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        const float a = fabsf(x[i]);
        if (!isnan(a) && a > amax) amax = a;
    }
    volatile float s = amax / 448.0f; /* volatile: keep each f32 op separately rounded */
    volatile float inv = 448.0f / amax;
    *scale = s;
    if (!isfinite(inv)) {
        for (int i = 0; i < n; ++i)
            codes[i] = (isnan(x[i]) || !signbit(x[i])) ? 0x00u : 0x80u;
        return;
    }
    for (int i = 0; i < n; ++i) {
        volatile float prod = x[i] * inv;
        codes[i] = orc_e4m3_encode(prod);
    }
}

void orc_quantize_row(const float* x, uint8_t* codes, float* scales) {
    quantize_segment(x, ORC_DL, codes, &scales[0]);
    quantize_segment(x + ORC_DL, ORC_DR, codes + ORC_DL, &scales[1]);
}

void orc_quantize_rows(const float* src, int64_t n_rows, int64_t src_row_stride,
                       const int64_t* dst_slot, uint8_t* codes, float* scales) {
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t slot = dst_slot ? dst_slot[r] : r;
        orc_quantize_row(src + r * src_row_stride, codes + slot * ORC_D, scales + slot * 2);
    }
}

/* ------------------------------------------------------------------------ */
/* Fused producer.  KV8 page, PR description, attention_rows item: the producer
 * quantizes the new row after its normalisation and rotation.  The page names the steps but not
 * their formulas; the readings (RMS norm with a weight over Lc, rotation of the
 * pairs (2j, 2j+1) of Rc by tabulated angles) and the fixed f32 order are in
 * kv8_oracle.h.  Each f32 operation goes through a volatile, so it is rounded
 * once, in the order written.                                                  */
void orc_rmsnorm_row(const float* x, const float* weight, float eps, float* y) {
    /* The sum of squares as written: each square is exact in double (a 24-bit
     * significand squared fits in 53 bits), the 512 squares are added in index
     * order in double, and the total is rounded to f32 once.  Away from f32
     * rounding boundaries this is the correctly rounded f32 of the exact sum,
     * whatever order any other implementation adds in. */
    double acc = 0.0;
    for (int i = 0; i < ORC_DL; ++i) {
        const double xi = (double)x[i];
        acc += xi * xi;
    }
    volatile float ss = (float)acc;
    volatile float ms = ss * (1.0f / 512.0f);     /* exact: a power of two */
    volatile float t = ms + eps;
    volatile float r = sqrtf(t);
    volatile float inv = 1.0f / r;
    for (int i = 0; i < ORC_DL; ++i) {
        volatile float a = x[i] * inv;
        volatile float b = a * weight[i];
        y[i] = b;
    }
}

void orc_rope_pairs(const float* x, const float* cos_row, const float* sin_row, float* y) {
    for (int j = 0; j < ORC_DR / 2; ++j) {
        const float x0 = x[2 * j], x1 = x[2 * j + 1], c = cos_row[j], s = sin_row[j];
        volatile float a = x0 * c, b = x1 * s, d = x0 * s, e = x1 * c;
        volatile float y0 = a - b, y1 = d + e;
        y[2 * j] = y0;
        y[2 * j + 1] = y1;
    }
}

void orc_produce_rows(const float* src, int64_t n_rows, int64_t src_row_stride,
                      const float* norm_weight, float eps, const int64_t* positions,
                      const float* rope_cos, const float* rope_sin, int64_t max_pos,
                      const int64_t* dst_slot, uint8_t* codes, float* scales) {
    float y[ORC_D];
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t pos = positions[r];
        if (pos < 0 || pos >= max_pos) continue;
        const float* x = src + r * src_row_stride;
        orc_rmsnorm_row(x, norm_weight, eps, y);
        orc_rope_pairs(x + ORC_DL, rope_cos + pos * (ORC_DR / 2), rope_sin + pos * (ORC_DR / 2),
                       y + ORC_DL);
        const int64_t slot = dst_slot ? dst_slot[r] : r;
        orc_quantize_row(y, codes + slot * ORC_D, scales + slot * 2);
    }
}

/* ------------------------------------------------------------------------ */
/* Absorbed decode attention.  KV8 page, PR description, opening paragraph: in the
 * absorbed attention the latent serves as key and as value; attention_rows item:
 * the score and context loops decode the codes as they go and apply the row scale
 * outside each dot product.  For one head with query (q_lat, q_rope):
 *   z_t = sm_scale * ( sLc_t * sum_i q_lat[i] dec(Lc_t[i])
 *                    + sRc_t * sum_j q_rope[j] dec(Rc_t[j]) )
 *   M = max_t z_t,  p_t = exp(z_t - M),  l = sum_t p_t
 *   out[i] = ( sum_t (p_t * sLc_t) * dec(Lc_t[i]) ) / l,   lse = M + log(l)
 * Dots and sums run in index order.  T = 0 gives out = 0 and lse = -inf (our
 * reading; the page does not treat an empty cache).                           */
static inline int64_t slot_of(const int64_t* map, int64_t t) { return map ? map[t] : t; }

static void attention_head_f32(const float* ql, const float* qr, const uint8_t* codes,
                               const float* scales, const int64_t* map, int64_t T,
                               float sm_scale, float* out, float* lse, float* z) {
    lut_init();
    for (int i = 0; i < ORC_DL; ++i) out[i] = 0.0f;
    if (T == 0) {
        if (lse) *lse = -INFINITY;
        return;
    }
    float M = -INFINITY;
    for (int64_t t = 0; t < T; ++t) {
        const uint8_t* row = codes + slot_of(map, t) * ORC_D;
        const float* sc = scales + slot_of(map, t) * 2;
        float dl = 0.0f, dr = 0.0f;
        for (int i = 0; i < ORC_DL; ++i) dl += ql[i] * g_lut[row[i]];
        for (int j = 0; j < ORC_DR; ++j) dr += qr[j] * g_lut[row[ORC_DL + j]];
        const float zl = sc[0] * dl;
        const float zr = sc[1] * dr;
        z[t] = sm_scale * (zl + zr);
        if (z[t] > M) M = z[t];
    }
    float l = 0.0f;
    for (int64_t t = 0; t < T; ++t) {
        const uint8_t* row = codes + slot_of(map, t) * ORC_D;
        const float p = expf(z[t] - M);
        l += p;
        const float w = p * scales[slot_of(map, t) * 2];
        for (int i = 0; i < ORC_DL; ++i) out[i] += w * g_lut[row[i]];
    }
    for (int i = 0; i < ORC_DL; ++i) out[i] /= l;
    if (lse) *lse = M + logf(l);
}

#include <stdlib.h>

void orc_attention_f32(const float* q_lat, const float* q_rope, const uint8_t* codes,
                       const float* scales, const int64_t* slot_of_token, int64_t T, int H,
                       float sm_scale, float* out, float* lse) {
    float* z = (float*)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1));
    for (int h = 0; h < H; ++h)
        attention_head_f32(q_lat + (int64_t)h * ORC_DL, q_rope + (int64_t)h * ORC_DR, codes,
                           scales, slot_of_token, T, sm_scale, out + (int64_t)h * ORC_DL,
                           lse ? lse + h : NULL, z);
    free(z);
}

/* f64 twin: the same steps with every product, sum, exp and log in double.  The
 * codes and the f32 scales are exact in double, so this is the attention of the
 * stored cache up to double rounding. */
static void partial_head_f64(const float* ql, const float* qr, const uint8_t* codes,
                             const float* scales, const int64_t* map, int64_t t0, int64_t t1,
                             double sm_scale, double* o, double* m_out, double* l_out,
                             double* z) {
    lut_init();
    for (int i = 0; i < ORC_DL; ++i) o[i] = 0.0;
    double M = -INFINITY;
    for (int64_t t = t0; t < t1; ++t) {
        const uint8_t* row = codes + slot_of(map, t) * ORC_D;
        const float* sc = scales + slot_of(map, t) * 2;
        double dl = 0.0, dr = 0.0;
        for (int i = 0; i < ORC_DL; ++i) dl += (double)ql[i] * (double)g_lut[row[i]];
        for (int j = 0; j < ORC_DR; ++j) dr += (double)qr[j] * (double)g_lut[row[ORC_DL + j]];
        z[t - t0] = sm_scale * ((double)sc[0] * dl + (double)sc[1] * dr);
        if (z[t - t0] > M) M = z[t - t0];
    }
    double l = 0.0;
    for (int64_t t = t0; t < t1; ++t) {
        const uint8_t* row = codes + slot_of(map, t) * ORC_D;
        const double p = exp(z[t - t0] - M);
        l += p;
        const double w = p * (double)scales[slot_of(map, t) * 2];
        for (int i = 0; i < ORC_DL; ++i) o[i] += w * (double)g_lut[row[i]];
    }
    *m_out = M;
    *l_out = l;
}

void orc_attention_partial_f64(const float* q_lat, const float* q_rope, const uint8_t* codes,
                               const float* scales, const int64_t* slot_of_token, int64_t t0,
                               int64_t t1, int H, double sm_scale, double* o, double* m,
                               double* l) {
    double* z = (double*)malloc(sizeof(double) * (size_t)(t1 > t0 ? t1 - t0 : 1));
    for (int h = 0; h < H; ++h) {
        if (t1 <= t0) {
            for (int i = 0; i < ORC_DL; ++i) o[(int64_t)h * ORC_DL + i] = 0.0;
            m[h] = -INFINITY;
            l[h] = 0.0;
            continue;
        }
        partial_head_f64(q_lat + (int64_t)h * ORC_DL, q_rope + (int64_t)h * ORC_DR, codes,
                         scales, slot_of_token, t0, t1, sm_scale, o + (int64_t)h * ORC_DL,
                         &m[h], &l[h], z);
    }
    free(z);
}

/* Split-T merge (flash-decoding): with M = max_s m_s and w_s = exp(m_s - M),
 * out = sum_s w_s o_s / sum_s w_s l_s and lse = M + log(sum_s w_s l_s).  The
 * KV8 page's closing note names split-T kernels for long caches; this is the
 * standard exact recombination of softmax partials. */
void orc_lse_merge_f64(int n_parts, int H, const double* o_parts, const double* m_parts,
                       const double* l_parts, double* out, double* lse) {
    for (int h = 0; h < H; ++h) {
        double M = -INFINITY;
        for (int s = 0; s < n_parts; ++s)
            if (m_parts[(int64_t)s * H + h] > M) M = m_parts[(int64_t)s * H + h];
        double L = 0.0;
        for (int i = 0; i < ORC_DL; ++i) out[(int64_t)h * ORC_DL + i] = 0.0;
        if (M == -INFINITY) {
            if (lse) lse[h] = -INFINITY;
            continue;
        }
        for (int s = 0; s < n_parts; ++s) {
            const double ms = m_parts[(int64_t)s * H + h];
            if (ms == -INFINITY) continue;
            const double w = exp(ms - M);
            L += w * l_parts[(int64_t)s * H + h];
            const double* os = o_parts + ((int64_t)s * H + h) * ORC_DL;
            for (int i = 0; i < ORC_DL; ++i) out[(int64_t)h * ORC_DL + i] += w * os[i];
        }
        for (int i = 0; i < ORC_DL; ++i) out[(int64_t)h * ORC_DL + i] /= L;
        if (lse) lse[h] = M + log(L);
    }
}

void orc_attention_heads_f64(const float* q_lat, const float* q_rope, const uint8_t* codes,
                             const float* scales, const int64_t* slot_of_token, int64_t T,
                             int H, int h0, int nh, double sm_scale, double* out, double* lse) {
    (void)H;
    double* z = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    for (int k = 0; k < nh; ++k) {
        const int h = h0 + k;
        double* o = out + (int64_t)k * ORC_DL;
        if (T == 0) {
            for (int i = 0; i < ORC_DL; ++i) o[i] = 0.0;
            if (lse) lse[k] = -INFINITY;
            continue;
        }
        double m, l;
        partial_head_f64(q_lat + (int64_t)h * ORC_DL, q_rope + (int64_t)h * ORC_DR, codes,
                         scales, slot_of_token, 0, T, sm_scale, o, &m, &l, z);
        for (int i = 0; i < ORC_DL; ++i) o[i] /= l;
        if (lse) lse[k] = m + log(l);
    }
    free(z);
}

void orc_attention_f64(const float* q_lat, const float* q_rope, const uint8_t* codes,
                       const float* scales, const int64_t* slot_of_token, int64_t T, int H,
                       double sm_scale, double* out, double* lse) {
    orc_attention_heads_f64(q_lat, q_rope, codes, scales, slot_of_token, T, H, 0, H, sm_scale,
                            out, lse);
}

/* ------------------------------------------------------------------------ */
/* Paged batch.  The KV8 page's batched CUDA entry point does not say what the
 * batch is; our reading is ragged sequences whose rows sit in fixed-size blocks
 * of one pool, listed per sequence in a block table. */
void orc_paged_slots(const int32_t* block_table, int max_blocks, int block_size, int b,
                     int64_t T, int64_t* slots) {
    for (int64_t t = 0; t < T; ++t)
        slots[t] = (int64_t)block_table[(int64_t)b * max_blocks + t / block_size] * block_size +
                   t % block_size;
}

void orc_attention_batch_f32(const float* q_lat, const float* q_rope, const uint8_t* codes,
                             const float* scales, const int32_t* block_table,
                             const int32_t* seq_lens, int B, int H, int max_blocks,
                             int block_size, float sm_scale, float* out, float* lse,
                             int n_threads) {
    int64_t Tmax = 1;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] > Tmax) Tmax = seq_lens[b];
    int64_t* slots = (int64_t*)malloc(sizeof(int64_t) * (size_t)B * (size_t)Tmax);
    for (int b = 0; b < B; ++b)
        orc_paged_slots(block_table, max_blocks, block_size, b, seq_lens[b], slots + b * Tmax);
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel
    {
        float* z = (float*)malloc(sizeof(float) * (size_t)Tmax);
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
            const int b = (int)(bh / H), h = (int)(bh % H);
            const int64_t qo = (int64_t)b * H + h;
            attention_head_f32(q_lat + qo * ORC_DL, q_rope + qo * ORC_DR, codes, scales,
                               slots + b * Tmax, seq_lens[b], sm_scale, out + qo * ORC_DL,
                               lse ? lse + qo : NULL, z);
        }
        free(z);
    }
    free(slots);
}

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
