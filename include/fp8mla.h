/*
 * fp8mla.h -- C ABI of libfp8mla.so: an fp8 e4m3 latent KV cache and absorbed
 * MLA decode attention over it, hand-written CUDA for one GB300 (sm_103a).
 *
 * Source of the method: the pull-request page "KV8=1: fp8 e4m3 latent KV cache
 * (CPU + CUDA) with .coli_kv v2" (the "KV8 page").  The page names the calls
 * (c/kv_fp8.h per-row quantizer; CUDA entry points for absorbed decode and its
 * batched form) but prints no signatures; the ones below are ours.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument is a DEVICE pointer unless stated otherwise.  The
 *   caller owns all memory, including the decode workspace; the library never
 *   allocates device memory and keeps no state between calls.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Every call is asynchronous on it: nothing synchronises, and
 *   results are ready only when the stream reaches them.  Calls are thread-safe.
 * - A call first validates its arguments on the host and returns a negative
 *   kv8_status before launching anything if they are bad.  A failed kernel
 *   launch returns KV8_ECUDA.  No kernel traps or spins without a bound.
 * - Cache layout (one layer; our reading, the page states no byte layout):
 *     kv_codes [n_slots][576] uint8 -- e4m3fn bytes; bytes 0..511 are the
 *               latent Lc (kv_lora, both key and value), 512..575 the RoPE key
 *               Rc (qk_rope).  Rows are 576 = 36 x 16 bytes, so every row starts
 *               on a 16-byte boundary when kv_codes does.
 *     kv_scales[n_slots][2]  float  -- {sLc, sRc}, each amax/448 of its segment.
 */
#ifndef FP8MLA_H
#define FP8MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KV8_DL 512    /* kv_lora: latent width (key and value)    */
#define KV8_DR 64     /* qk_rope: RoPE key width (key only)        */
#define KV8_D 576     /* bytes per cached row                      */
#define KV8_BLOCK 64  /* tokens per page of the paged batch layout */

typedef enum {
    KV8_OK = 0,
    KV8_EINVAL = -1,        /* null pointer, negative size, bad dimension            */
    KV8_EALIGN = -2,        /* a pointer or stride breaks the alignment rule stated  */
    KV8_EUNSUPPORTED = -3,  /* a size the library does not handle (e.g. block_size)  */
    KV8_ECUDA = -4,         /* a CUDA launch or runtime call failed                  */
    KV8_EBOUNDS = -5,       /* a device-side index (block table, seq_len) was bad    */
    KV8_EWORKSPACE = -6,    /* workspace missing or smaller than *_workspace_size    */
    KV8_ETIMEOUT = -7,      /* a bounded device-side wait gave up (internal error)   */
    KV8_ESCRATCH = -8,      /* problem too large for the library's static scratch    */
    KV8_EIO = -9,           /* a cache-file read, write or rename failed             */
    KV8_EFORMAT = -10       /* not a cache file, or shorter than its committed rows  */
} kv8_status;

/* Decode kernel choice.  All accumulate in f32.  Tolerance classes, as max-abs
 * error against the exact attention of the stored cache:
 *   SIMT     f32 operands:                      <= 2e-3 * max|out|
 *   TCGEN05  reduced-precision MMA operands on e4m3 tensor cores: the query as
 *            two e4m3 terms on a per-head power-of-two scale (about 8 significant
 *            bits) against the cache's e4m3 values for the scores, and the softmax
 *            weights as two e4m3 terms on one scale for the context; both read
 *            the e4m3 cache values as they are:  <= 1e-2 * max|out|
 * (see the test report for the measured worst case of each kernel).
 * TCGEN05 runs the SM-pair kernel (a cluster of two CTAs per work item: one
 * computes scores and softmax, the other the context, for 128 heads) when
 * H > 64, and the one-CTA kernel (16 or 32 heads per CTA) otherwise;
 * TCGEN05_CTA and TCGEN05_PAIR force one of the two at any H.              */
typedef enum {
    KV8_DECODE_AUTO = 0,         /* TCGEN05 when H >= 16, else SIMT              */
    KV8_DECODE_SIMT = 1,         /* CUDA-core split-T kernel, any H >= 1         */
    KV8_DECODE_TCGEN05 = 2,      /* tcgen05 tensor cores, H >= 1                 */
    KV8_DECODE_TCGEN05_CTA = 3,  /* tcgen05, one CTA per work item               */
    KV8_DECODE_TCGEN05_PAIR = 4  /* tcgen05, a pair of SMs per work item         */
} kv8_decode_variant;

/* ---------------------------------------------------------------------------
 * kv8_quantize_rows -- KV8 page, PR description, c/kv_fp8.h item (a per-row
 * quantizer that guards rows with a subnormal amax) and attention_rows item (the
 * producer quantizes the new row, once normalised and rotated, instead of keeping
 * an f32 copy).
 *
 * For each source row r, and for each segment (Lc = floats 0..511, Rc = floats
 * 512..575) separately:
 *   amax = max |x| over non-NaN entries;  scale = amax / 448 (f32, RN);
 *   inv  = 448 / amax (f32, RN);
 *   if inv is not finite (amax == 0 or amax < 448/FLT_MAX): every code is a
 *     signed zero (0x80 for negative x, 0x00 otherwise and for NaN);
 *   else code = e4m3(x * inv) with the product rounded once (no FMA), rounding
 *     to nearest even, saturating to +-448 (0x7E/0xFE), keeping the sign of
 *     zero, and storing NaN as 0x00.
 * The 576 codes go to kv_codes[slot] and {sLc, sRc} to kv_scales[slot], where
 * slot = dst_slot[r] (device int64 array), or r when dst_slot is NULL.
 * The result is bit-identical to the oracle for every f32 input.
 *
 *   src            device f32 [n_rows][src_row_stride]; 16-byte aligned,
 *                  src_row_stride (in floats) >= 576 and a multiple of 4.
 *   n_rows         >= 0 (0 launches nothing).
 *   dst_slot       device int64 [n_rows] or NULL.  A slot outside [0, n_slots)
 *                  is skipped (that row writes nothing).
 *   kv_codes       device uint8 [n_slots][576], 16-byte aligned.
 *   kv_scales      device f32 [n_slots][2], 8-byte aligned.
 *   n_slots        rows in the cache pool; with dst_slot == NULL, >= n_rows.
 * Errors: KV8_EINVAL, KV8_EALIGN, KV8_ECUDA.
 * ------------------------------------------------------------------------- */
int kv8_quantize_rows(const float* src, int64_t n_rows, int64_t src_row_stride,
                      const int64_t* dst_slot, uint8_t* kv_codes, float* kv_scales,
                      int64_t n_slots, void* stream);

/* ---------------------------------------------------------------------------
 * kv8_produce_rows -- KV8 page, PR description, attention_rows item: the
 * producer quantizes the new row after normalisation and rotation instead of
 * keeping an f32 copy.  The fused form of that producer: from the raw latent rows
 * to cache codes in one pass.  The page names the steps; the formulas are our reading.  For each row r
 * with position pos = positions[r]:
 *   Lc (floats 0..511):   ss  = sum of x_i^2 in a fixed order (32 partial sums
 *                         of x[16l..16l+15] in index order, then for o = 16, 8,
 *                         4, 2, 1 every partial p_l becomes p_l + p_(l xor o));
 *                         inv = 1 / sqrt(ss / 512 + eps);  y_i = (x_i * inv) * w_i
 *   Rc (floats 512..575): for pair j = 0..31, (x0, x1) = (x[512+2j], x[512+2j+1]),
 *                         c = rope_cos[pos][j], s = rope_sin[pos][j]:
 *                         y0 = x0*c - x1*s,  y1 = x0*s + x1*c
 *   then y is quantized exactly as by kv8_quantize_rows into slot dst_slot[r].
 * Every f32 operation is rounded once (no FMA), so the codes are bit-identical
 * to the oracle's for every input.
 *
 *   src            device f32 [n_rows][src_row_stride]; 16-byte aligned,
 *                  src_row_stride (in floats) >= 576 and a multiple of 4.
 *   norm_weight    device f32 [512], 16-byte aligned.
 *   eps            finite, >= 0.
 *   positions      device int64 [n_rows].  A row whose position is outside
 *                  [0, max_pos) is skipped (writes nothing) and, when err_word
 *                  is not NULL, sets bit 0 of *err_word (atomic OR; the caller
 *                  clears it).
 *   rope_cos/sin   device f32 [max_pos][32], 4-byte aligned.
 *   dst_slot, kv_codes, kv_scales, n_slots: as for kv8_quantize_rows.
 *   err_word       device uint32 or NULL.
 * Errors: KV8_EINVAL, KV8_EALIGN, KV8_ECUDA.
 * ------------------------------------------------------------------------- */
int kv8_produce_rows(const float* src, int64_t n_rows, int64_t src_row_stride,
                     const float* norm_weight, float eps, const int64_t* positions,
                     const float* rope_cos, const float* rope_sin, int64_t max_pos,
                     const int64_t* dst_slot, uint8_t* kv_codes, float* kv_scales,
                     int64_t n_slots, unsigned* err_word, void* stream);

/* ---------------------------------------------------------------------------
 * mla_wuv_epilogue -- the step after the absorbed attention (KV8 page, PR
 * description: in the absorbed attention the latent is key and value at once, so
 * the attention's output is a latent context per head): the per-head value
 * projection
 *   y[b][h][v] = sum_{d<512} o[b][h][d] * W_UV[h][d][v]      (f32 accumulation)
 *
 *   o        device f32 [B][H][512] (e.g. the decode call's out), 4-byte aligned.
 *   w_uv     device bf16 bit patterns [H][512][V], 2-byte aligned.
 *   B, H, V  B >= 0, 1 <= H <= 1024, 1 <= V <= 4096.
 *   y        device f32 [B][H][V].
 * Tolerance: f32 sums of 512 products in a fixed order (partial sums over
 * groups of latent rows, then added in a fixed order of groups), the same bits on
 * every call:
 * max-abs error <= 1e-5 * max|y| against float64.
 * Errors: KV8_EINVAL, KV8_EALIGN, KV8_ECUDA.
 * ------------------------------------------------------------------------- */
int mla_wuv_epilogue(const float* o, const uint16_t* w_uv, int B, int H, int V, float* y,
                     void* stream);

/* ---------------------------------------------------------------------------
 * kv8_prefill_project -- the non-absorbed projection of the cached latent (KV8
 * page, PR description: the projection path dequantizes the cached Lc rows
 * before the kv_b up-projection):
 *   Y[t][n] = sLc_t * sum_{d<512} dec(Lc_t[d]) * W_UKV[d][n]
 * on the tensor cores (bf16 operands: every e4m3 value is exact in bf16; f32
 * accumulation; the row scale applied to the f32 sum; Y rounded to bf16).
 *
 *   kv_codes, kv_scales  the cache, as written by kv8_quantize_rows
 *                        ([n_slots][576] e4m3, 16-byte aligned; [n_slots][2] f32).
 *   slots          device int64 [T]: cache slot of token t, or NULL for slot t.
 *                  A slot outside [0, n_slots) gives a zero row and sets bit 0
 *                  of *err_word.
 *   T              tokens, 0 <= T <= 2^30.
 *   w_ukv          device bf16 bit patterns [512][N], row-major, 16-byte aligned.
 *   N              columns, a positive multiple of 256 (H x (qk_nope + v_head)).
 *   y              device bf16 [T][N], 16-byte aligned.
 *   k_rope         device f32 [T][64], 16-byte aligned, or NULL: the token's rope
 *                  key dequantized, sRc_t * dec(Rc_t[j]) rounded once to f32
 *                  (bit-exact; a zero row for a slot out of range).
 *   err_word       device uint32 or NULL; bit 2 marks a device-side wait that
 *                  timed out (the launch then returns without finishing).
 * Tolerance: max-abs error <= 1e-2 * max|Y| against the float64 oracle (bf16
 * rounding of the result; f32 sums of 512 products).
 * Errors: KV8_EINVAL, KV8_EALIGN, KV8_EUNSUPPORTED, KV8_ECUDA.
 * ------------------------------------------------------------------------- */
int kv8_prefill_project(const uint8_t* kv_codes, const float* kv_scales, int64_t n_slots,
                        const int64_t* slots, int64_t T, const uint16_t* w_ukv, int N,
                        uint16_t* y, float* k_rope, unsigned* err_word, void* stream);

/* ---------------------------------------------------------------------------
 * kv8_selftest_wait_timeout -- check of the failure path of the device-side
 * waits.  The decode kernels' pipelines wait on mbarriers with a time limit; a
 * wait that runs out makes the kernel flag the workspace error word and return
 * (KV8_ETIMEOUT from kv8_workspace_error), never trap or hang.  This call runs
 * one warp that waits, through the same bounded wait, on a barrier nothing
 * arrives at, with the given limit (1 us .. 10 s): afterwards
 * kv8_workspace_error(workspace) reports KV8_ETIMEOUT and the context is usable.
 *   workspace  device, >= 256 bytes, 256-byte aligned (its error word is reset
 *              first).
 * Errors: KV8_EINVAL, KV8_EWORKSPACE, KV8_EALIGN, KV8_ECUDA.
 * ------------------------------------------------------------------------- */
int kv8_selftest_wait_timeout(void* workspace, int64_t workspace_bytes, int64_t limit_us,
                              void* stream);

/* ---------------------------------------------------------------------------
 * mla_absorb_decode_fp8 -- KV8 page, PR description, opening paragraph (the latent
 * is key and value at once in the absorbed attention), attention_rows item (the
 * score and context loops decode as they go, the row scale applied outside each
 * dot product), CUDA item (absorbed decode kernel over fp8 rows); the closing note's
 * split-T kernels for long caches.
 *
 * One decode query (H heads) against one contiguous cache of T rows (slots
 * 0..T-1).  For each head h:
 *   z_t  = sm_scale * ( sLc_t * <q_lat[h], dec(Lc_t)> + sRc_t * <q_rope[h], dec(Rc_t)> )
 *   p_t  = softmax_t(z)_t
 *   out[h][:] = sum_t p_t * sLc_t * dec(Lc_t)        (latent-space context)
 *   lse[h]    = log sum_t exp(z_t)                   (natural log)
 * T == 0 gives out = 0 and lse = -inf.
 *
 *   q_lat     device f32 [H][512], 16-byte aligned.
 *   q_rope    device f32 [H][64],  16-byte aligned.
 *   kv_codes  device uint8 [>= T][576], 16-byte aligned.
 *   kv_scales device f32 [>= T][2], 16-byte aligned.
 *   T         >= 0.  H >= 1 and H <= 1024.
 *   sm_scale  > 0 and finite (KV8_EINVAL otherwise).
 *   out       device f32 [H][512], 16-byte aligned.  lse: device f32 [H] or NULL.
 *   workspace device, >= mla_absorb_decode_fp8_workspace_size(T, H, variant)
 *             bytes, 256-byte aligned; scratch for the split-T partials.  Calls
 *             that overlap in time must not share a workspace.
 *   variant   a kv8_decode_variant.
 * Errors: KV8_EINVAL, KV8_EALIGN, KV8_EWORKSPACE, KV8_ECUDA.
 * ------------------------------------------------------------------------- */
int64_t mla_absorb_decode_fp8_workspace_size(int64_t T, int H, int variant);
int mla_absorb_decode_fp8(const float* q_lat, const float* q_rope, const uint8_t* kv_codes,
                          const float* kv_scales, int64_t T, int H, float sm_scale, float* out,
                          float* lse, void* workspace, int64_t workspace_bytes, int variant,
                          void* stream);

/* ---------------------------------------------------------------------------
 * mla_absorb_decode_fp8_batch -- the batched form (KV8 page, CUDA item: the
 * batched absorbed kernel).  Our reading of "batch": B ragged sequences, one
 * decode query each, whose rows sit in 64-token pages of one pool.  Token t of
 * sequence b is cache slot block_table[b][t / 64] * 64 + t % 64.  Per sequence
 * the arithmetic is that of mla_absorb_decode_fp8.
 *
 *   q_lat       device f32 [B][H][512];  q_rope device f32 [B][H][64].
 *   kv_codes    device uint8 [n_blocks * 64][576], 16-byte aligned;
 *               kv_scales f32 [n_blocks*64][2], 16-byte aligned.
 *   sm_scale    > 0 and finite (KV8_EINVAL otherwise).
 *   block_table device int32 [B][max_blocks];  seq_lens device int32 [B].
 *   block_size  must be 64 (KV8_EUNSUPPORTED otherwise).
 *   out         device f32 [B][H][512];  lse device f32 [B][H] or NULL.
 *   workspace   >= mla_absorb_decode_fp8_batch_workspace_size(B, H, max_blocks,
 *               block_size, variant) bytes, 256-byte aligned.
 * Device-side checks: a seq_len outside [0, max_blocks*64] is clamped, and a
 * block-table entry outside [0, n_blocks) makes its page read as empty; either
 * sets an error word in the workspace that kv8_workspace_error() reports.
 * Errors: KV8_EINVAL, KV8_EALIGN, KV8_EUNSUPPORTED, KV8_EWORKSPACE, KV8_ECUDA.
 * ------------------------------------------------------------------------- */
int64_t mla_absorb_decode_fp8_batch_workspace_size(int B, int H, int max_blocks, int block_size,
                                                   int variant);
int mla_absorb_decode_fp8_batch(const float* q_lat, const float* q_rope, const uint8_t* kv_codes,
                                const float* kv_scales, const int32_t* block_table,
                                const int32_t* seq_lens, int B, int H, int max_blocks,
                                int block_size, int64_t n_blocks, float sm_scale, float* out,
                                float* lse, void* workspace, int64_t workspace_bytes,
                                int variant, void* stream);

/* ---------------------------------------------------------------------------
 * Split phases of mla_absorb_decode_fp8_batch.  The batched call is exactly
 * _partials followed by _combine on the same stream and workspace.  _partials
 * runs the split-T kernel and leaves, per (sequence, split, head), the running
 * maximum m (log2 units), the sum l of 2^(z*log2e - m) and the unnormalised
 * context o in the workspace; _combine merges them into out/lse.  Exposed so a
 * caller can time the phases, or merge partials computed elsewhere (the same
 * log-sum-exp recombination joins the partials of one sequence split across
 * devices).  Arguments and errors as for mla_absorb_decode_fp8_batch.
 * ------------------------------------------------------------------------- */
int mla_absorb_decode_fp8_batch_partials(const float* q_lat, const float* q_rope,
                                         const uint8_t* kv_codes, const float* kv_scales,
                                         const int32_t* block_table, const int32_t* seq_lens,
                                         int B, int H, int max_blocks, int block_size,
                                         int64_t n_blocks, float sm_scale, void* workspace,
                                         int64_t workspace_bytes, int variant, void* stream);
int mla_absorb_decode_fp8_batch_combine(const int32_t* seq_lens, int B, int H, int max_blocks,
                                        int block_size, float* out, float* lse,
                                        const void* workspace, int64_t workspace_bytes,
                                        int variant, void* stream);

/* ---------------------------------------------------------------------------
 * mla_absorb_decode_fp8_batch_noalloc -- mla_absorb_decode_fp8_batch for
 * callers that cannot allocate device memory: code that runs where no
 * allocator may be called (a host runtime or plugin that owns every device
 * buffer and hands out only inputs and outputs, a hot loop whose memory budget
 * is fixed up front) and so has no way to provide a workspace.  The paper has no
 * counterpart; this is a convenience of this library.
 *
 * Same arguments, arithmetic and result as mla_absorb_decode_fp8_batch, minus
 * the workspace: the split-T partials go to one scratch array that the library
 * declares statically in device memory, KV8_NOALLOC_SCRATCH_BYTES (32 MiB) on
 * every GPU that loads the library, held until the process exits.  The call
 * allocates nothing and calls no allocating routine.
 * - Size limit: a problem whose workspace
 *   (mla_absorb_decode_fp8_batch_workspace_size) exceeds the scratch size is
 *   rejected with KV8_ESCRATCH before anything is launched.
 * - First call on a device: it looks up the scratch array's device address,
 *   with that device current, and caches it; make that first call before any
 *   stream capture on the device.
 * - Sharing: every call on a device uses the same scratch, which keeps the last
 *   call's contents.  Calls that can overlap on the GPU (different streams, or
 *   different host threads, without ordering between them) race on it and must
 *   not be issued that way; calls on one stream are ordered and safe.  The
 *   device-side error word is cleared by each call and can be read with
 *   kv8_noalloc_error().
 * Errors: as mla_absorb_decode_fp8_batch, plus KV8_ESCRATCH.
 * ------------------------------------------------------------------------- */
#define KV8_NOALLOC_SCRATCH_BYTES (32ll << 20)
int mla_absorb_decode_fp8_batch_noalloc(const float* q_lat, const float* q_rope,
                                        const uint8_t* kv_codes, const float* kv_scales,
                                        const int32_t* block_table, const int32_t* seq_lens,
                                        int B, int H, int max_blocks, int block_size,
                                        int64_t n_blocks, float sm_scale, float* out,
                                        float* lse, int variant, void* stream);
/* Synchronises `stream` and reports the error word of the last no-alloc call on
 * the current device, like kv8_workspace_error(). */
int kv8_noalloc_error(void* stream);

/* kv8_workspace_error -- synchronises `stream`, then reports the device-side
 * error word of the last decode call that used `workspace`: KV8_OK,
 * KV8_EBOUNDS (a bad block-table entry or seq_len) or KV8_ETIMEOUT (a kernel
 * gave up a wait after its bound and returned without a result).  A debugging
 * aid; the decode calls themselves never sync. */
int kv8_workspace_error(const void* workspace, void* stream);

/* Human-readable text for a kv8_status value (static storage). */
/* kv8_last_cuda_error -- the name of the CUDA error behind the calling thread's
 * most recent KV8_ECUDA (or KV8_EUNSUPPORTED) from a decode call, e.g.
 * "cudaErrorInvalidValue"; "cudaSuccess" if there was none.  Diagnostics only;
 * the paper has no counterpart.  Static string, never NULL. */
const char* kv8_last_cuda_error(void);
const char* kv8_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int kv8_abi_version(void);

/* ---------------------------------------------------------------------------
 * Cache file: save and resume of the fp8 cache (KV8 page, PR description,
 * persistence item: version 2 starts with the magic COLIKV2 and keeps its data
 * type in the header; rows are the fp8 codes with their scales, appended through
 * a persistent handle with a staging buffer; a version-1 file (f32 rows) is
 * quantized on resume and rewritten as version 2 at the first append; opening
 * repairs a damaged magic).  Byte layout (the page gives none), little-endian:
 *   header, 64 bytes: [0,8) magic "COLIKV2\0" (version 1: "COLIKV1\0");
 *     [8,12) u32 64 (header bytes); [12,16) u32 data type, 2 = e4m3 codes + two
 *     f32 scales, 1 = f32 values; [16,20) u32 576 (values per row); [20,24) u32
 *     bytes per record, 584 or 2304; [24,32) u64 rows committed; [32,64) zero.
 *   then the committed records: version 2: 576 code bytes, then sLc and sRc
 *     (f32); version 1: 576 f32.  Bytes after the last committed record (a torn
 *     append) are not content and are overwritten by the next append.
 * A handle is used by one host thread at a time.  Appends and loads are
 * synchronous: they synchronize `stream` and return when the file or the cache
 * holds the rows.
 * ------------------------------------------------------------------------- */
typedef struct kv8_disk kv8_disk;

/* Open (or create) the file at `path`.  A missing, empty or shorter-than-a-header
 * file becomes an empty version-2 file; a header whose fields after the magic are
 * a valid version-1 or version-2 header gets its magic rewritten.  The handle
 * owns a pinned, device-mapped host staging buffer of staging_rows x 2888 bytes
 * (1 <= staging_rows <= 2^22); it holds no device memory.
 * Errors: KV8_EINVAL, KV8_ECUDA (staging buffer), KV8_EIO, KV8_EFORMAT (a
 * header of neither version, or fewer bytes than the committed rows). */
int kv8_disk_open(const char* path, int64_t staging_rows, kv8_disk** out);

/* Committed rows and version (1 or 2) of an open file. */
int kv8_disk_info(const kv8_disk* d, int64_t* n_rows, int* version);

/* Append n rows taken from the cache (kv_codes [n_slots][576], 16-byte aligned;
 * kv_scales [n_slots][2]) at device slots[i] (int64, or NULL for slots 0..n-1).
 * A version-1 file is first rewritten as version 2.  The row count in the header
 * is rewritten only after the records are written.  A slot outside [0, n_slots)
 * gives KV8_EBOUNDS and commits nothing.
 * Errors: KV8_EINVAL, KV8_EALIGN, KV8_EBOUNDS, KV8_ECUDA, KV8_EIO. */
int kv8_disk_append(kv8_disk* d, const uint8_t* kv_codes, const float* kv_scales, int64_t n_slots,
                    const int64_t* slots, int64_t n, void* stream);

/* Load committed rows [first_row, first_row + n) into the cache at device
 * dst_slot[i] (int64, or NULL for slots first_row + i).  Version-1 rows are
 * quantized on the way in (the same codes as kv8_quantize_rows).  A row whose
 * slot is outside [0, n_slots) is not written and the call returns KV8_EBOUNDS.
 * Errors: KV8_EINVAL, KV8_EALIGN, KV8_EBOUNDS, KV8_ECUDA, KV8_EIO. */
int kv8_disk_load(kv8_disk* d, int64_t first_row, int64_t n, uint8_t* kv_codes, float* kv_scales,
                  int64_t n_slots, const int64_t* dst_slot, void* stream);

/* Close the file and free the staging buffer (NULL is accepted). */
int kv8_disk_close(kv8_disk* d);

#ifdef __cplusplus
}
#endif
#endif /* FP8MLA_H */
