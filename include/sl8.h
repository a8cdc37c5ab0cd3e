/*
 * sl8 -- W8A8 INT8 attention for NVIDIA GB300 (sm_103a): C ABI.
 *
 * The operations follow the "SuperL8" README (github.com/jajmangold/superl8):
 *   - "Supporting kernels" table, quant_rowwise: symmetric per-row int8 quantisation;
 *   - "Quantization" table, "Per-row int8": symmetric, with K-smoothing;
 *   - "Attention kernels" table, attn_int8_fwd: W8A8 FlashAttention-2 forward,
 *     causal, GQA/MQA, head dims 32/64/128/256 (this library: prefill and the int8-V
 *     decode all four, the fp16-V decode 64 and 128);
 *     attn_varlen_fwd: ragged variable-length prefill; attn_decode: split-KV decode
 *     with an int8 KV cache, int8-V variant;
 *   - "Quick start" section: q [B, Hq, N, d], k/v [B, Hkv, N, d],
 *     attn_int8_fwd(q, k, v, causal=True), quantising internally.
 * The pages give no formulas; the readings this library implements are:
 *   scale s = max|x| / 127 (IEEE fp32 division); code = clamp(round-half-even(x / s),
 *   -127, 127); a row with s == 0 has all-zero codes.  K-smoothing subtracts, per
 *   (sequence, kv head, channel), the fp32 mean of K over all the sequence's tokens
 *   (summed in 64-token chunks in token order, then the chunk sums in order).
 *   Logits x = int32(q_i8 . k_i8) * s_q * s_k / sqrt(d); the causal mask is top-left
 *   aligned (key j visible to query i iff j <= i); softmax is computed online
 *   (FlashAttention-2 style); O = P . V with P rounded to V's dtype and fp32
 *   accumulation.  GQA maps query head hq to kv head hq / (Hq / Hkv).
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must be device memory of the current CUDA
 *     device, 16-byte aligned, holding contiguous tensors in the stated layout.  The
 *     caller owns every buffer; the library allocates no device memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call only
 *     validates its arguments on the host and enqueues kernels on `stream`; it does
 *     not synchronise.
 *   - Argument errors are reported synchronously, before anything is launched.
 *     Conditions only the device can see (a cu_seqlens / seqlens entry out of range,
 *     a bounded device-side wait that gave up) are recorded in a per-device status
 *     word that sl8_last_device_status() reads.
 *   - No C++ exception crosses this interface.
 */
#ifndef SL8_H_
#define SL8_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SL8_API __attribute__((visibility("default")))
#else
#define SL8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sl8_status {
  SL8_OK = 0,
  SL8_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad shape or dtype, Hq % Hkv != 0 */
  SL8_ERR_UNSUPPORTED = 2, /* valid but not implemented here (e.g. the fp16-V decode at d = 256) */
  SL8_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the size query returned */
  SL8_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  SL8_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (see sl8_last_device_status) */
  SL8_ERR_DEVICE_ARG = 6   /* the device found an out-of-range length (cu_seqlens / seqlens) or page index */
} sl8_status;

typedef enum sl8_dtype { SL8_F16 = 0, SL8_BF16 = 1, SL8_F32 = 2, SL8_I8 = 3 } sl8_dtype;

/* Human-readable name of a status code (static string). */
SL8_API const char* sl8_status_string(int status);

/* Text of the CUDA error behind the calling thread's most recent SL8_ERR_CUDA from a
 * launch (a static string; "no CUDA error recorded" if there was none). */
SL8_API const char* sl8_last_cuda_error_string(void);

/* Library version, as major * 10000 + minor * 100 + patch. */
SL8_API int sl8_version(void);

/*
 * Symmetric per-row int8 quantisation ("Supporting kernels" table, quant_rowwise;
 * "Quantization" table, per-row int8).
 *   x          device, `rows` rows of `cols` elements of x_dtype (F16, BF16 or F32);
 *              row r starts at element r * row_stride_elems.
 *   sub_mean   device, nullable: [groups][cols] fp32; row r first has
 *              sub_mean[r / rows_per_group] subtracted (fp32), which is K-smoothing
 *              when the groups are (sequence, kv head) blocks of a dense [B,H,N,d] K.
 *   q_out      device, [rows][cols] int8 codes (contiguous).
 *   scale_out  device, [rows] fp32 scales s = max|x - mean| / 127.
 * Errors: SL8_ERR_INVALID_ARG for null x/q_out/scale_out, rows < 0, cols < 1,
 * row_stride_elems < cols, rows_per_group < 1 with sub_mean set, or a bad dtype.
 * rows == 0 returns SL8_OK at once (the pointers may then be null).
 */
SL8_API int sl8_quant_rowwise(const void* x, int x_dtype, int64_t rows, int32_t cols, int64_t row_stride_elems,
                      const float* sub_mean, int64_t rows_per_group, int8_t* q_out, float* scale_out,
                      void* stream);

/*
 * Per-channel mean of K over each sequence's tokens, the K-smoothing statistic
 * ("Quantization" table, per-row int8 with K-smoothing).
 *   k           device.  Dense (cu_seqlens NULL): [B][Hkv][N][d]; varlen:
 *               [total_tokens][Hkv][d] packed, sequence s = tokens
 *               [cu_seqlens[s], cu_seqlens[s+1]).
 *   cu_seqlens  device, nullable, [B + 1] int32, nondecreasing, each length <= N.
 *   mean_out    device, [B][Hkv][d] fp32.
 *   workspace   device scratch of at least sl8_k_channel_mean_workspace_size() bytes.
 */
SL8_API size_t sl8_k_channel_mean_workspace_size(int32_t B, int32_t Hkv, int32_t N, int32_t d);
SL8_API int sl8_k_channel_mean(const void* k, int k_dtype, int32_t B, int32_t Hkv, int32_t N, int32_t d,
                       const int32_t* cu_seqlens, int64_t total_tokens, float* mean_out, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * W8A8 INT8 attention prefill ("Attention kernels" table, attn_int8_fwd and
 * attn_varlen_fwd; "Quick start" section for the layouts).
 *   q, k, v     device.  Dense (cu_seqlens NULL): q [B][Hq][N][d], k/v [B][Hkv][N][d].
 *               Varlen: q [total_tokens][Hq][d], k/v [total_tokens][Hkv][d] packed,
 *               B = number of sequences, N = the longest sequence length (an upper
 *               bound every cu_seqlens length must respect).
 *   qk_dtype    F16 or BF16 (q and k); v_dtype F16 or BF16.
 *   d           32, 64, 128 or 256 (32 runs as 64 with zero channels past 32: exact, at the
 *               cost of d = 64).  Hq must be a multiple of Hkv.
 *   causal      nonzero: key j is visible to query i iff j <= i (positions within the
 *               sequence).
 *   smooth_k    nonzero: subtract K's per-channel mean before quantising K.
 *   out         device, same layout as q, of out_dtype (v_dtype, or F32).
 *   lse_out     device, nullable: fp32 log-sum-exp (natural log) per query row,
 *               dense [B][Hq][N], varlen [total_tokens][Hq].
 *   workspace   device scratch of at least sl8_attn_int8_fwd_workspace_size() bytes
 *               (the quantised codes, scales, K means and the work list live there).
 * Errors: SL8_ERR_INVALID_ARG, SL8_ERR_UNSUPPORTED (d not in {32,64,128,256}),
 * SL8_ERR_WORKSPACE, SL8_ERR_CUDA.  Empty inputs (B, N or total_tokens 0) return
 * SL8_OK without launching.
 */
SL8_API size_t sl8_attn_int8_fwd_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t N, int32_t d,
                                        int64_t total_tokens);
SL8_API int sl8_attn_int8_fwd(const void* q, const void* k, const void* v, int qk_dtype, int v_dtype, int32_t B, int32_t Hq,
                      int32_t Hkv, int32_t N, int32_t d, const int32_t* cu_seqlens, int64_t total_tokens,
                      int causal, int smooth_k, void* out, int out_dtype, float* lse_out, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * Prefill of a query chunk against a longer key sequence (the "Engine" table's chunked
 * prefill onto keys already present; bottom-right alignment, reading: the pages give
 * none): q [B][Hq][Nq][d] holds the last Nq positions of sequences whose keys and values
 * k, v [B][Hkv][Nk][d] cover all Nk positions, 0 <= Nq <= Nk.  Query i is position
 * i + Nk - Nq: causal, it sees keys j <= i + Nk - Nq.  K-smoothing, the K codes and the
 * V range run over all Nk keys, so the result equals rows Nk-Nq .. Nk-1 of
 * sl8_attn_int8_fwd on the full sequences.  out [B][Hq][Nq][d], lse_out [B][Hq][Nq].
 * Dense input only.  The workspace is at least sl8_attn_int8_fwd_workspace_size(B, Hq,
 * Hkv, Nk, d, 0) bytes.  Given sl8_attn_int8_fwd_chunk_workspace_size(B, Hq, Hkv, Nq, Nk,
 * d) bytes, a chunk whose (query tile, head) items fill at most half the current
 * device's SMs (d <= 128) also splits each item's keys into up to 8 parts, so that the
 * parts run as one wave.  Each part writes a normalised fp32 partial and its log-sum-exp
 * into the workspace, and a merge step (weights e^(lse - max lse), as the split-KV
 * decode's combine) forms out and lse_out: the same attention, with P rounded to fp16
 * against each part's own running maximum.  Other arguments and errors as
 * sl8_attn_int8_fwd.
 */
SL8_API size_t sl8_attn_int8_fwd_chunk_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t Nq, int32_t Nk,
                                                      int32_t d);
SL8_API int sl8_attn_int8_fwd_chunk(const void* q, const void* k, const void* v, int qk_dtype, int v_dtype, int32_t B,
                                    int32_t Hq, int32_t Hkv, int32_t Nq, int32_t Nk, int32_t d, int causal,
                                    int smooth_k, void* out, int out_dtype, float* lse_out, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * Prefill of a query chunk onto an int8 KV cache that already holds its keys (the
 * "Engine" table's chunked prefill onto a paged/int8 KV cache, with the cache format of
 * the "Attention kernels" table's attn_decode row; reading: the pages give no layout).
 * Nothing is re-quantised but Q: the cache's K codes and scales enter the exact int32
 * logits as they are, and V is dequantised (code * scale) into the fp16 operand of P.V.
 *   q                   device, [B][Hq][Nq][d] of q_dtype (F16 or BF16): the queries of
 *                       positions Nk - Nq .. Nk - 1 of every sequence, quantised per row
 *                       as in sl8_attn_int8_fwd.
 *   k_cache, v_cache    device, [B][Hkv][Lmax][d] int8 codes (16-byte aligned), as for
 *                       sl8_attn_int8_decode_splitkv; every sequence holds Nk positions
 *                       (rows 0 .. Nk-1, the chunk's own included), Nq <= Nk <= Lmax.
 *   k_scale, v_scale    device, [B][Hkv][Lmax] fp32 per-token scales.
 *   causal              nonzero: query i (position Nk - Nq + i) sees keys j <= Nk - Nq + i;
 *                       zero: every query sees all Nk keys.
 *   out                 device, [B][Hq][Nq][d] of out_dtype (F16, BF16 or F32).
 *   lse_out             device, nullable, [B][Hq][Nq] fp32 (natural log).
 *   workspace           at least sl8_attn_int8_fwd_chunk_workspace_size(B, Hq, Hkv, Nq,
 *                       Nk, d) bytes (the same layout, key splits of small chunks
 *                       included); sl8_attn_int8_fwd_workspace_size(B, Hq, Hkv, Nk, d, 0)
 *                       bytes run without key splits.
 * V enters P.V as fp16(code * scale * 2^-e), e >= 0 the least exponent with
 * max(v_scale) < 2^(e + 8) over the (sequence, kv head), and O is scaled back by 2^e.
 * Errors: SL8_ERR_INVALID_ARG (null or misaligned pointers, dtypes, shapes,
 * Nq > Nk > Lmax), SL8_ERR_UNSUPPORTED (d not in {32, 64, 128, 256}, B * Nk >= 2^31),
 * SL8_ERR_WORKSPACE, SL8_ERR_CUDA.  B or Nq 0: SL8_OK without launching.
 */
SL8_API int sl8_attn_int8_fwd_chunk_cache(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale,
                                          const int8_t* v_cache, const float* v_scale, int32_t B, int32_t Hq,
                                          int32_t Hkv, int32_t Nq, int32_t Nk, int32_t Lmax, int32_t d, int causal,
                                          void* out, int out_dtype, float* lse_out, void* workspace,
                                          size_t workspace_bytes, void* stream);

/*
 * W8A8 prefill with grouped ("per-warp") scales and outlier-aware Q ("Attention
 * kernels" table, attn_w8a8_fwd row: a W8A8 forward with scales set per warp that takes
 * outliers into account; "Quantization" table, per-row int8 row, which lists outlier
 * detection for Q).  The pages give no
 * formula; the reading implemented:
 *   - the rows of each (sequence, head) form groups of G consecutive positions from
 *     position 0 (q_group for Q, k_group for K after its channel mean); every row of a
 *     group quantises with s = (max |x| over the group's non-outlier rows) / 127 (fp32
 *     division) and codes RNE(x / s) clamped to +-127;
 *   - a Q row is an outlier when max|x| > q_outlier_ratio * m (one fp32 product), m the
 *     lower median of its group's row maxima (element (n - 1) / 2 of the ascending
 *     sort); an outlier row keeps its own scale max|x| / 127.  q_outlier_ratio = 0
 *     turns the test off.  K rows have no outlier test (K-smoothing handles K).
 * q_group = k_group = 1 is sl8_attn_int8_fwd exactly.  The attention after the
 * quantisation is that of sl8_attn_int8_fwd (exact int32 logits times the row
 * scales), so the same kernel runs at the same speed.
 *   q_group, k_group    powers of two, 1 .. 64 (SL8_ERR_INVALID_ARG otherwise); 32 are
 *                       the rows one warp of the softmax covers.
 *   q_outlier_ratio     finite, >= 0 (SL8_ERR_INVALID_ARG otherwise).
 * Everything else (layouts, varlen, causal, head dims, dtypes, workspace from
 * sl8_attn_int8_fwd_workspace_size, errors) as sl8_attn_int8_fwd.
 */
SL8_API int sl8_attn_w8a8_fwd(const void* q, const void* k, const void* v, int qk_dtype, int v_dtype, int32_t B,
                              int32_t Hq, int32_t Hkv, int32_t N, int32_t d, const int32_t* cu_seqlens,
                              int64_t total_tokens, int causal, int smooth_k, int32_t q_group, int32_t k_group,
                              float q_outlier_ratio, void* out, int out_dtype, float* lse_out, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Debug view of the prefill's quantisation and int32 logits (same kernels and
 * tensor-core path as sl8_attn_int8_fwd, without the mask).  q, k, qk_dtype, B, Hq,
 * Hkv, N, d, cu_seqlens and total_tokens as for sl8_attn_int8_fwd (dense or varlen).
 *   logits_out  device, nullable, [B][Hq][row_end - row_begin][N] int32:
 *               logits_out[s][h][i - row_begin][j] = int32(q_i8[s,h,i] . k_i8[s,hkv,j])
 *               for every key j < L_s of sequence s (L_s = N dense, else its
 *               cu_seqlens length) and every row row_begin <= i < min(row_end, L_s);
 *               other entries are left untouched.  0 <= row_begin <= row_end <= N.
 *   q_codes/q_scales    device, nullable: dense [B][Hq][N][d] int8 / [B][Hq][N] fp32,
 *                       varlen [total_tokens][Hq][d] / [total_tokens][Hq].
 *   k_codes/k_scales    device, nullable: dense [B][Hkv][N][d] int8 / [B][Hkv][N] fp32,
 *                       varlen [total_tokens][Hkv][d] / [total_tokens][Hkv] (after
 *                       smoothing when smooth_k is set).
 *   workspace   as for sl8_attn_int8_fwd (same size query).
 */
SL8_API int sl8_attn_int8_qk_logits_debug(const void* q, const void* k, int qk_dtype, int32_t B, int32_t Hq, int32_t Hkv,
                                  int32_t N, int32_t d, const int32_t* cu_seqlens, int64_t total_tokens,
                                  int smooth_k, int32_t row_begin, int32_t row_end, int32_t* logits_out,
                                  int8_t* q_codes, float* q_scales, int8_t* k_codes, float* k_scales,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * The same debug view for the grouped quantisation of sl8_attn_w8a8_fwd (q_group,
 * k_group and q_outlier_ratio as there); the codes, scales and logits are those the
 * sl8_attn_w8a8_fwd attention consumes.
 */
SL8_API int sl8_attn_w8a8_qk_logits_debug(const void* q, const void* k, int qk_dtype, int32_t B, int32_t Hq,
                                          int32_t Hkv, int32_t N, int32_t d, const int32_t* cu_seqlens,
                                          int64_t total_tokens, int smooth_k, int32_t q_group, int32_t k_group,
                                          float q_outlier_ratio, int32_t row_begin, int32_t row_end,
                                          int32_t* logits_out, int8_t* q_codes, float* q_scales, int8_t* k_codes,
                                          float* k_scales, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Split-KV decode over an int8 KV cache ("Attention kernels" table, attn_decode,
 * int8-V variant): one query token per sequence against its cached keys t < L_b.
 * d is 32, 64, 128 or 256.
 *   q                  device, [B][Hq][d] of q_dtype (F16, BF16 or F32); quantised
 *                      per row inside the kernel.
 *   k_cache, v_cache   device, [B][Hkv][Lmax][d] int8 codes.
 *   k_scale, v_scale   device, [B][Hkv][Lmax] fp32 per-token scales.
 *   seqlens            device, [B] int32, 0 <= L_b <= Lmax.
 *   num_splits         requested number of contiguous key splits (0 = automatic: about
 *                      10 (split, sequence, kv head) work slots per SM of the current
 *                      device).  Split s covers tokens [s * split_size, (s + 1) * split_size)
 *                      with split_size = ceil(Lmax / S) rounded up to whole stages of the
 *                      split kernel (160 tokens for d <= 128, 128 for d = 256; to 16 tokens
 *                      below one stage); the effective count
 *                      S = sl8_attn_decode_num_splits(B, Hkv, Lmax, d, num_splits) can be
 *                      below the request after that rounding.
 *   o_partial          device, [B][Hq][S][d] fp32; each non-empty split's normalised partial
 *                      (the O of an empty split is not written).
 *   lse_partial        device, [B][Hq][S] fp32 log-sum-exp per split (-inf if empty).
 * GQA and MQA: any Hq that is a multiple of Hkv.  A work slot of the split kernel holds at
 * most 8 query heads, so with G = Hq / Hkv > 8 each kv head's G query heads are cut into
 * the fewest equal groups of at most 8 (G = 16: 2 groups of 8; G = 32: 4; G = 12: 2 of 6)
 * and each group streams that kv head's cache: the cache is read once per group.
 */
SL8_API int32_t sl8_attn_decode_num_splits(int32_t B, int32_t Hkv, int32_t Lmax, int32_t d, int32_t num_splits);
SL8_API int32_t sl8_attn_decode_split_size(int32_t B, int32_t Hkv, int32_t Lmax, int32_t d, int32_t num_splits);

/*
 * Scratch of the split-KV decode ("Attention kernels" table, attn_decode: the partials
 * that a split-KV decode merges): the bytes of o_partial and lse_partial for the
 * effective split count S = sl8_attn_decode_num_splits(B, Hkv, Lmax, d, num_splits),
 * laid out in one caller-owned buffer as
 *   o_partial   at byte 0:                          [B][Hq][S][d] fp32;
 *   lse_partial at sl8_attn_decode_lse_offset(...):  [B][Hq][S] fp32
 * (the offset is B * Hq * S * d * 4 rounded up to 256 bytes).  Returns 0 for an
 * invalid or unsupported shape (as sl8_attn_decode_num_splits, or Hq not a multiple
 * of Hkv).  Pure host arithmetic: no device is touched except for the SM count that
 * the automatic split count (num_splits = 0) uses.
 */
SL8_API size_t sl8_attn_decode_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax, int32_t d,
                                              int32_t num_splits);
SL8_API size_t sl8_attn_decode_lse_offset(int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax, int32_t d,
                                          int32_t num_splits);
SL8_API int sl8_attn_int8_decode_splitkv(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale,
                                 const int8_t* v_cache, const float* v_scale, const int32_t* seqlens, int32_t B,
                                 int32_t Hq, int32_t Hkv, int32_t Lmax, int32_t d, int32_t num_splits,
                                 float* o_partial, float* lse_partial, void* stream);

/*
 * Speculative-decode verification over the int8 cache: the attn_decode row's "verify
 * mask" variant and the attn_tree_fwd row ("Attention kernels" table; tree or chain
 * masks from the "Speculative decoding" table's drafters).  Reading (the pages give no
 * layout): the cache (as sl8_attn_int8_decode_splitkv) already holds each sequence's T
 * draft tokens at positions L_b - T .. L_b - 1, and
 *   q          device, [B][T][Hq][d] (q_dtype F16, BF16 or F32): the drafts' queries.
 *   tree_mask  device, [B][T] uint32: query t sees every position below L_b - T and
 *              draft token u (position L_b - T + u, if >= 0) iff bit u is set.
 *   T          1 .. 32 draft tokens per sequence; B * T <= 65535.
 *   o_partial, lse_partial  scratch, [B * T][Hq][S][d] and [B * T][Hq][S] fp32 with
 *              S = sl8_attn_decode_verify_num_splits(B, T, Hq, Hkv, Lmax, d, num_splits).
 *   out        device, [B][T][Hq][d] of out_dtype (F16, BF16 or F32); lse_out nullable
 *              [B][T][Hq].
 * Runs the split kernel and the combine.  A work slot takes min(T, 8 / (Hq / Hkv)) draft
 * queries beside their query heads, so sequence b's cache is read ceil(T / that) times;
 * Hq / Hkv must be at most 8 (SL8_ERR_UNSUPPORTED otherwise).
 */
SL8_API int32_t sl8_attn_decode_verify_num_splits(int32_t B, int32_t T, int32_t Hq, int32_t Hkv, int32_t Lmax,
                                                  int32_t d, int32_t num_splits);
SL8_API int sl8_attn_int8_decode_verify(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale,
                                        const int8_t* v_cache, const float* v_scale, const int32_t* seqlens,
                                        const uint32_t* tree_mask, int32_t T, int32_t B, int32_t Hq, int32_t Hkv,
                                        int32_t Lmax, int32_t d, int32_t num_splits, float* o_partial,
                                        float* lse_partial, void* out, int out_dtype, float* lse_out, void* stream);

/*
 * Split-KV decode with an int8 K cache and an fp16 V cache: the attn_decode row's
 * "fp16 V" variant ("Attention kernels" table).  Same operation, split plan and outputs
 * as sl8_attn_int8_decode_splitkv, with O = sum_t p_t * v[t] (V has no scale):
 *   k_cache, k_scale  as there ([B][Hkv][Lmax][d] int8 codes, [B][Hkv][Lmax] fp32).
 *   v_cache           device, [B][Hkv][Lmax][d] fp16 (16-byte aligned).
 * d must be 64 or 128 (SL8_ERR_UNSUPPORTED for 32 and 256).  The partials are merged with
 * sl8_attn_decode_combine.
 */
SL8_API int sl8_attn_int8_decode_splitkv_f16v(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale,
                                              const void* v_cache, const int32_t* seqlens, int32_t B, int32_t Hq,
                                              int32_t Hkv, int32_t Lmax, int32_t d, int32_t num_splits,
                                              float* o_partial, float* lse_partial, void* stream);

/*
 * Split-KV decode over a paged int8 KV cache: the "Engine" table's "Paged KV cache" row
 * (int8 / k8v3 / k8v8 cache formats) with the k8v8 format, and the "Attention kernels"
 * table's attn_paged_decode row.  Same operation, split plan and outputs as
 * sl8_attn_int8_decode_splitkv with Lmax = max_blocks * page_size; only the cache's
 * storage differs (reading: the pages give no layout):
 *   k_pages, v_pages            device, [num_pages][Hkv][page_size][d] int8 codes
 *                               (16-byte aligned).
 *   k_scale_pages, v_scale_pages device, [num_pages][Hkv][page_size] fp32 per-token
 *                               scales (16-byte aligned).
 *   block_table                 device, [B][max_blocks] int32: page of the logical block
 *                               i = tokens [i * page_size, (i + 1) * page_size) of
 *                               sequence b.  Token t of sequence b is row t % page_size
 *                               of page block_table[b][t / page_size].  Entries past a
 *                               sequence's last block are never read; pages may be
 *                               shared between sequences (common prefixes).
 *   page_size                   a multiple of 16 (SL8_ERR_UNSUPPORTED otherwise).
 *   num_pages * Hkv * page_size must stay below 2^31.
 * A block-table entry outside [0, num_pages) is reported as SL8_ERR_DEVICE_ARG by
 * sl8_last_device_status and page 0 is read in its place.  The partials are merged
 * with sl8_attn_decode_combine(..., Lmax = max_blocks * page_size, ...).
 */
SL8_API int sl8_attn_int8_paged_decode_splitkv(const void* q, int q_dtype, const int8_t* k_pages,
                                               const float* k_scale_pages, const int8_t* v_pages,
                                               const float* v_scale_pages, const int32_t* block_table,
                                               int32_t max_blocks, int32_t page_size, int32_t num_pages,
                                               const int32_t* seqlens, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                                               int32_t num_splits, float* o_partial, float* lse_partial,
                                               void* stream);

/*
 * Decode combine: merge the split partials of each (b, hq) row,
 * O = sum_s e^(lse_s - M) O_s / sum_s e^(lse_s - M), M = max_s lse_s, over the
 * non-empty splits.  A row with L_b = 0 gets O = 0 (lse -inf).
 *   out      device, [B][Hq][d] of out_dtype (F16, BF16 or F32).
 *   lse_out  device, nullable, [B][Hq] fp32.
 *   num_splits must be the effective count S of the split call (same Lmax); the split
 *   size is derived from Lmax and S as there.
 */
SL8_API int sl8_attn_decode_combine(const float* o_partial, const float* lse_partial, const int32_t* seqlens, int32_t B,
                            int32_t Hq, int32_t Lmax, int32_t d, int32_t num_splits, void* out, int out_dtype,
                            float* lse_out, void* stream);

/*
 * Debug view of the decode's q quantisation and int32 logits (same kernel as the
 * split call, with num_splits automatic: o_partial/lse_partial sized for
 * S = sl8_attn_decode_num_splits(B, Hkv, Lmax, d, 0)).
 *   logits_out  device, [B][Hq][Lmax] int32: entry t < L_b is int32(q_i8 . k_i8[t]);
 *               entries t >= L_b are left untouched.
 *   q_codes/q_scales  device, nullable, [B][Hq][d] int8 (4-byte aligned) / [B][Hq] fp32.
 *   o_partial/lse_partial  scratch as for the split call.
 */
SL8_API int sl8_attn_int8_decode_logits_debug(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale,
                                      const int8_t* v_cache, const float* v_scale, const int32_t* seqlens,
                                      int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax, int32_t d,
                                      int32_t* logits_out, int8_t* q_codes, float* q_scales, float* o_partial,
                                      float* lse_partial, void* stream);

/*
 * Decode without any allocation (no counterpart on the SuperL8 pages: it exists for
 * callers that cannot allocate GPU memory where they run decode -- a serving loop with
 * a fixed memory budget, code that only holds tensors another framework owns, a C
 * caller without an allocator -- and for whom cudaMalloc would also stall the device).
 * Same inputs and result as sl8_attn_int8_decode_splitkv followed by
 * sl8_attn_decode_combine (out [B][Hq][d] of out_dtype, F16/BF16/F32), but the split
 * partials live in a fixed SL8_NOALLOC_SCRATCH_BYTES device array inside the library,
 * which every GPU that loads the library holds until the process exits.
 *   - The automatic split count is lowered to what the array holds; a problem whose
 *     single split needs more than the array (B * Hq * (d + 1) * 4 bytes >
 *     SL8_NOALLOC_SCRATCH_BYTES) is refused with SL8_ERR_WORKSPACE before any launch.
 *   - The first call on each device looks up the array's device address (with that
 *     device current); make that first call before any stream capture.  The address is
 *     kept for the life of the process: it does not survive cudaDeviceReset() or any
 *     other teardown of the device's primary context, after which this entry point
 *     must not be called again in the same process.
 *   - Every call uses the same array: calls whose work overlaps on the GPU (other
 *     streams, other threads) race on it and must be serialised by the caller.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define SL8_NOALLOC_SCRATCH_BYTES (16u << 20)
SL8_API int sl8_attn_int8_decode_noalloc(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale,
                                         const int8_t* v_cache, const float* v_scale, const int32_t* seqlens,
                                         int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax, int32_t d, void* out,
                                         int out_dtype, void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status word (its
 * address is looked up once per device and, like the no-allocation scratch above, is
 * not valid after cudaDeviceReset()):
 * SL8_OK, SL8_ERR_TIMEOUT (a bounded wait gave up; *site names the wait) or
 * SL8_ERR_DEVICE_ARG (an out-of-range device-side length).  site may be NULL.
 */
SL8_API int sl8_last_device_status(void* stream, int* site);

/* Upper bound, in nanoseconds, on every device-side wait (default 2e9). */
SL8_API void sl8_set_spin_limit_ns(uint64_t limit_ns);
SL8_API uint64_t sl8_get_spin_limit_ns(void);

/*
 * Self-test of the bounded waits: launches one kernel whose wait on a barrier that
 * nothing arrives on must give up after limit_ns and record SL8_ERR_TIMEOUT.
 */
SL8_API int sl8_selftest_timeout(uint64_t limit_ns, void* stream);

/*
 * Kernel tracing.  While enabled, every kernel the library launches is bracketed by
 * CUDA events on its stream.  sl8_trace_collect() synchronises those events and
 * returns, per kernel name, the number of launches and their summed device time;
 * it then clears the record.  Returns the number of names written (at most max).
 */
SL8_API void sl8_trace_enable(int on);
SL8_API int sl8_trace_collect(const char** names, int64_t* launches, double* total_ms, int max);

#ifdef __cplusplus
}
#endif

#endif /* SL8_H_ */
