/*
 * kv8_oracle.h -- plain, slow, obviously-correct CPU oracle for the fp8 e4m3
 * latent KV cache and absorbed MLA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code; only the test suite, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code with the CUDA library.
 *
 * Source of the method: the pull-request page "KV8=1: fp8 e4m3 latent KV cache
 * (CPU + CUDA) with .coli_kv v2" (called "the KV8 page" below).  Every function
 * cites the part of that page it follows.  Precision: the page fixes f32 for the
 * stored scales and for the quantizer arithmetic; attention is given in f32 (the
 * page's CPU loops) and in an f64 twin that serves as the tolerance reference.
 *
 * Row format (our reading of the page; it states no byte layout):
 *   codes[slot][0:512]   = Lc (kv_lora latent, key and value), e4m3 bytes
 *   codes[slot][512:576] = Rc (qk_rope key), e4m3 bytes
 *   scales[slot][0]      = sLc = amax(Lc)/448  (f32)
 *   scales[slot][1]      = sRc = amax(Rc)/448  (f32)
 */
#ifndef KV8_ORACLE_H
#define KV8_ORACLE_H
#include <stdint.h>

#define ORC_DL 512
#define ORC_DR 64
#define ORC_D 576

#ifdef __cplusplus
extern "C" {
#endif

/* ---- e4m3 codec (KV8 page, PR description, c/kv_fp8.h item) ---- */
float orc_e4m3_decode(uint8_t code);              /* 256-entry LUT from the closed form */
void orc_e4m3_decode_table(float out[256]);
uint8_t orc_e4m3_encode(float q);                 /* RNE bit-math encoder */
uint8_t orc_e4m3_encode_nearest(float q);         /* brute force over all codes (test of the test) */
uint8_t orc_e4m3_encode_bracket(float q);         /* sorted-midpoint search (test of the test) */
/* Array forms: which = 0 bit-math, 1 brute force, 2 bracket. */
void orc_e4m3_encode_array(const float* x, int64_t n, uint8_t* out, int which);
/* Count patterns u in [lo, hi) where bit-math and bracket encoders disagree (OpenMP). */
int64_t orc_e4m3_exhaustive_mismatches(uint64_t lo, uint64_t hi, uint32_t* first_bad);
/* Same, bit-math vs brute force, over an explicit list of f32 bit patterns. */
int64_t orc_e4m3_list_mismatches_nearest(const uint32_t* bits, int64_t n, uint32_t* first_bad);

/* ---- per-row quantizer (KV8 page, c/kv_fp8.h item and attention_rows item) ---- */
void orc_quantize_row(const float* x, uint8_t* codes, float* scales);
void orc_quantize_rows(const float* src, int64_t n_rows, int64_t src_row_stride,
                       const int64_t* dst_slot, uint8_t* codes, float* scales);

/* ---- fused producer (KV8 page, PR description, attention_rows item: the
 * producer quantizes the new row after normalisation and rotation instead of
 * keeping an f32 copy) ----
 * Our reading of the steps the page names but does not spell out:
 *   Lc: RMS norm with a weight, y_i = (x_i * inv) * w_i, inv = 1 / sqrt(ss/512 + eps);
 *   Rc: rotary embedding of the 32 pairs (x[2j], x[2j+1]) by the angle whose
 *       cosine and sine the caller tabulates per position (rope_cos/sin[pos][32]):
 *       y0 = x0*c - x1*s,  y1 = x0*s + x1*c;
 *   then the per-row quantizer above, into dst_slot[r].
 * Every f32 operation is rounded once (no FMA).  The sum of squares ss is the
 * plain sum: the squares (exact in double) added in index order in double, the
 * total rounded to f32 once -- the correctly rounded f32 sum except on rows whose
 * exact sum sits within about 2^-44 of an f32 rounding boundary.  Rows whose
 * position is outside [0, max_pos) are skipped (their slots are left as they
 * were).                                                                        */
void orc_rmsnorm_row(const float* x, const float* weight, float eps, float* y);
void orc_rope_pairs(const float* x, const float* cos_row, const float* sin_row, float* y);
void orc_produce_rows(const float* src, int64_t n_rows, int64_t src_row_stride,
                      const float* norm_weight, float eps, const int64_t* positions,
                      const float* rope_cos, const float* rope_sin, int64_t max_pos,
                      const int64_t* dst_slot, uint8_t* codes, float* scales);

/* ---- absorbed decode attention (KV8 page, attention_rows item) ----
 * One query (all H heads) against the rows of one sequence.  slot_of_token[t]
 * gives the cache slot of token t (NULL means slot == t).
 * out: [H][512], lse: [H] or NULL (natural log). */
void orc_attention_f32(const float* q_lat, const float* q_rope, const uint8_t* codes,
                       const float* scales, const int64_t* slot_of_token, int64_t T, int H,
                       float sm_scale, float* out, float* lse);
void orc_attention_f64(const float* q_lat, const float* q_rope, const uint8_t* codes,
                       const float* scales, const int64_t* slot_of_token, int64_t T, int H,
                       double sm_scale, double* out, double* lse);
/* Same arithmetic as orc_attention_f64 restricted to heads [h0, h0+nh). */
void orc_attention_heads_f64(const float* q_lat, const float* q_rope, const uint8_t* codes,
                             const float* scales, const int64_t* slot_of_token, int64_t T,
                             int H, int h0, int nh, double sm_scale, double* out, double* lse);

/* Partial attention over tokens [t0, t1) for the split-T (flash-decoding) form:
 * m = max score, l = sum exp(z - m), o = sum exp(z - m) * sLc * dec(Lc) (unnormalised). */
void orc_attention_partial_f64(const float* q_lat, const float* q_rope, const uint8_t* codes,
                               const float* scales, const int64_t* slot_of_token, int64_t t0,
                               int64_t t1, int H, double sm_scale, double* o, double* m,
                               double* l);
/* Log-sum-exp merge of n_parts partials (each o: [H][512], m, l: [H]). */
void orc_lse_merge_f64(int n_parts, int H, const double* o_parts, const double* m_parts,
                       const double* l_parts, double* out, double* lse);

/* Paged batch: token t of sequence b lives in slot block_table[b][t / bs] * bs + t % bs. */
void orc_paged_slots(const int32_t* block_table, int max_blocks, int block_size, int b,
                     int64_t T, int64_t* slots);
/* Batched f32 oracle (OpenMP over (sequence, head)); used for the CPU baseline timing. */
void orc_attention_batch_f32(const float* q_lat, const float* q_rope, const uint8_t* codes,
                             const float* scales, const int32_t* block_table,
                             const int32_t* seq_lens, int B, int H, int max_blocks,
                             int block_size, float sm_scale, float* out, float* lse,
                             int n_threads);
int orc_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
