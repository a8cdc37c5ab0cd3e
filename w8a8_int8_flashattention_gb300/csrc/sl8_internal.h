// Internal declarations shared by the ABI layer and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/sl8.h"
#include "sm103_ptx.cuh"

namespace sl8 {

constexpr int kQTile = 128;      // query rows per prefill work item (MMA M)
constexpr int kPadRows = 128;    // each sequence starts at a multiple of this in the code workspace
constexpr int kMeanChunk = 64;   // K-smoothing summation chunk (tokens)
constexpr int kMaxKeySplit = 8;  // key-split parts of a query chunk, merged by prefill_combine

// Per-sequence table and work list written by the scheduler kernel into the
// prefill workspace.  All arrays are int32.
struct SeqTable {
  int32_t* pstart;   // [nseq]  first padded row of the sequence in the code workspace
  int32_t* len;      // [nseq]  sequence length
  int32_t* tok0;     // [nseq]  first token of the sequence in the caller's tensors (varlen: cu_seqlens[s])
  int32_t* pair_seq; // [max_pairs] work list: sequence of each (sequence, q-tile) pair
  int32_t* pair_qt;  // [max_pairs] q-tile index of each pair
  int32_t* counts;   // [4]: 0 = number of pairs, 1 = total padded rows, 2 = attention items
                     //      claimed past the first wave (zeroed by the quantiser)
  int32_t* hist;     // [max_tiles + 2] scratch for the scheduler
  int32_t* sorted;   // [nseq] scratch: sequences ordered by tile count, longest first
};

// Carve-up of the prefill workspace (byte offsets from its base).
struct PrefillWorkspace {
  size_t q_codes, q_scales, k_codes, k_scales, v16, k_mean, k_partials, v_partials, v_exp, kv_done;
  size_t pstart, len, tok0, pair_seq, pair_qt, counts, hist, sorted;
  size_t total;
  int64_t t_pad_max;   // rows reserved per head in the code workspace
  int32_t max_chunks;  // 64-token chunks per sequence (upper bound)
  int32_t max_tiles;   // q tiles per sequence (upper bound)
  int64_t max_pairs;
};
PrefillWorkspace plan_prefill_workspace(int32_t nseq, int32_t Hq, int32_t Hkv, int32_t N, int32_t d,
                                        int64_t total_tokens, bool varlen);

// Device pointer of the library's status word on the current device.
DeviceStatus* device_status_ptr();
uint64_t spin_limit_ns();
int num_sms();
// Raise a kernel's dynamic shared memory limit to at least `bytes` on the current device.
// Each (kernel, device) is raised once, so the launches that follow (including those
// recorded into a CUDA graph by stream capture) make no attribute call.
cudaError_t ensure_smem(const void* kernel, int bytes);

// ---- tracing (CUDA events around each launch when enabled)
struct TraceScope {
  TraceScope(const char* name, cudaStream_t s);
  ~TraceScope();
  int slot;
  cudaStream_t stream;
};

// Launch with programmatic stream serialization: the kernel may start while the
// previous kernel of the stream finishes, and must call grid_dependency_wait() before
// it touches that kernel's results (every kernel launched this way does so first).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- launchers (return a cudaError_t from the launch)
// cu_seqlens (nullable = dense) must describe sequences inside [0, total_tokens) whose
// padded rows fit in t_pad_max; violations are recorded as a device-side argument
// error and the affected work is dropped.
// Work-list items are `item_rows` (a multiple of 128) consecutive query rows.
// kv_done [n_done] (the K/V statistics kernel's completion counters) is zeroed too.
cudaError_t launch_schedule(const int32_t* cu_seqlens, int32_t nseq, int32_t N, int64_t total_tokens,
                            int64_t t_pad_max, const SeqTable& t, int32_t item_rows, int32_t* kv_done,
                            int32_t n_done, cudaStream_t s);
// Query rows per work-list item of the prefill kernel for head dim d and group size
// Hq / Hkv; prefill_head_pairs: whether an item of the two-tile kernel is one Q tile of
// two query heads of the same kv head (else two Q tiles of one head).
int prefill_item_rows(int d, int group);
bool prefill_head_pairs(int d, int group);
// K chunk sums (k_partials, nullable) and V chunk abs-max (v_partials, nullable; V bf16);
// the last chunk of each (sequence, kv head) to finish forms the K mean [nseq][Hkv][d]
// and the V power-of-two exponent [nseq][Hkv].  kv_done [nseq][Hkv] must be zero.
cudaError_t launch_kv_stats(const void* k, sl8_dtype dt, const void* v, bool varlen, int32_t nseq, int32_t Hkv,
                            int32_t N, int32_t d, const int32_t* len, const int32_t* tok0, float* k_partials,
                            float* v_partials, int32_t max_chunks, float* mean, int32_t* v_exp, int32_t* kv_done,
                            cudaStream_t s);
// Prefill K chunk sums and V chunk abs-max (v_partials nullable), rows staged in shared
// memory; len / tok0 nullable for dense input; total_tokens: rows of a varlen K / V.
cudaError_t launch_kv_partials(const void* k, sl8_dtype dt, const void* v, bool varlen, int32_t nseq, int32_t Hkv,
                               int32_t N, int32_t d, const int32_t* len, const int32_t* tok0, float* k_partials,
                               float* v_partials, int32_t max_chunks, int64_t total_tokens, cudaStream_t s);
// From the chunk results of launch_kv_partials (either nullable): the K mean
// [nseq][Hkv][d_io] and the V exponent [nseq][Hkv] (0 without v_partials); one CTA per
// (sequence, kv head); len nullable for dense input (every sequence N long).
cudaError_t launch_kv_finalize(bool varlen, int32_t nseq, int32_t Hkv, int32_t N, int32_t d_io, const int32_t* len,
                               const float* k_partials, const float* v_partials, int32_t max_chunks, float* mean,
                               int32_t* v_exp, cudaStream_t s);
// Q and K rows of prefill in one launch.  With k_partials or v_partials set, the chunk
// kernels and launch_kv_finalize ran just before: K rows are smoothed with k_mean (set
// iff k_partials is) and, with v16 set, V is written as fp16 * 2^-v_exp with the exponent
// kv_finalize left in v_exp; otherwise the exponent is 0 and is written to v_exp here.
// t is read for varlen input only.  q_off > 0 (dense): q holds N - q_off rows per
// (sequence, head), the positions q_off .. N-1; the Q code rows of the positions before it
// in the attention's first item are zero, those of earlier items are not written.  d_io < d (head dim 32 run as 64): the inputs hold d_io values per row and the
// code rows are zero past them; k_partials then has d_io columns; v_f16: V is fp16
// (copied, v_partials unused and the exponent 0), else bf16.  k == nullptr: Q rows only
// (the K codes, K scales and V come from elsewhere, e.g. launch_cache_codes).
// Grouped scales for attn_w8a8_fwd (all 1 / 0: per-row scales, the attn_int8_fwd path).
struct QuantGroups {
  int32_t q_group = 1, k_group = 1;  // rows per shared scale, powers of two <= 64
  float q_tau = 0.0f;                // Q outlier ratio against the group's lower median; 0: none
};
cudaError_t launch_quant_qk(const void* q, const void* k, sl8_dtype dt, bool varlen, int32_t nseq, int32_t Hq,
                            int32_t Hkv, int32_t N, int32_t d, int64_t total_tokens, const SeqTable& t,
                            int64_t t_pad_max, const float* k_partials, const float* v_partials,
                            int32_t max_chunks, uint16_t* q_codes, float* q_scales, uint16_t* k_codes,
                            float* k_scales, const void* v, int32_t* v_exp, uint16_t* v16, cudaStream_t s,
                            int32_t q_off = 0, int32_t d_io = 0, bool v_f16 = false,
                            const QuantGroups& groups = QuantGroups(), const float* k_mean = nullptr);
// K and V rows of a dense int8 cache (every sequence holding N positions, Lmax rows apart)
// into the attention kernel's code workspace: K codes widened to bf16 with their scales;
// V dequantised (code * scale) and stored as fp16 * 2^-v_exp, the exponent per (sequence,
// kv head) from the largest V scale, written to v_exp.  Rows from N to the end of the
// sequence's padded rows (and columns from d_io to d) are zero.  d: the code row width
// (64 when head dim 32 runs as 64).
cudaError_t launch_cache_codes(const int8_t* k_cache, const float* k_scale, const int8_t* v_cache,
                               const float* v_scale, int32_t nseq, int32_t Hkv, int32_t N, int32_t Lmax, int32_t d,
                               int32_t d_io, int64_t t_pad_max, uint16_t* k_codes, float* k_scales, uint16_t* v16,
                               int32_t* v_exp, cudaStream_t s);
cudaError_t launch_quant_rowwise(const void* x, sl8_dtype dt, int64_t rows, int32_t cols, int64_t row_stride,
                                 const float* sub_mean, int64_t rows_per_group, int8_t* q_out, float* scale_out,
                                 cudaStream_t s);
cudaError_t launch_export_codes(const uint16_t* codes, const float* scales, bool varlen, int32_t nseq, int32_t H,
                                int32_t N, int32_t d, const SeqTable& t, int64_t t_pad_max, int8_t* codes_out,
                                float* scales_out, cudaStream_t s, int32_t d_io = 0);

struct PrefillArgs {
  const uint16_t* q_codes;  // [Hq][t_pad][d] bf16 codes
  const float* q_scales;    // [Hq][t_pad]
  const uint16_t* k_codes;  // [Hkv][t_pad][d]
  const float* k_scales;    // [Hkv][t_pad]
  const void* v;            // caller's V (used when it is fp16)
  sl8_dtype v_dtype;
  const uint16_t* v16;      // [Hkv][t_pad][d] fp16 copy of a bf16 V scaled by 2^-v_exp (nullable)
  const int32_t* v_exp;     // [nseq][Hkv] (nullable = 0)
  bool varlen;
  int32_t nseq, Hq, Hkv, N, d;
  int32_t d_io;              // values per row of q, k, v and out (d, or 32 when head dim 32 runs as 64)
  int32_t q_off;             // dense query chunk: q and out hold positions q_off .. N-1 (N keys)
  int64_t total_tokens;
  int64_t t_pad_max;
  SeqTable table;            // varlen only: the dense layout is arithmetic
  int32_t dense_items;       // items per sequence of a dense input (ceil(N / item rows) - dense_first)
  int32_t dense_first;       // first item of a dense query chunk (q_off / item rows; 0 otherwise)
  bool head_pairs;           // see prefill_head_pairs
  int64_t max_pairs;
  bool causal;
  void* out;                // caller's output
  sl8_dtype out_dtype;
  float* lse;               // nullable
  int32_t* logits;          // debug mode: [nseq][Hq][row_end-row_begin][N] int32 (dense only)
  int32_t row_begin, row_end;
  // key splits (dense query chunks, d <= 128): each item's key tiles are cut into kv_split
  // contiguous parts run as separate items; a part writes its normalised O (fp32) and its
  // log-sum-exp (natural log, -inf for a part with no key) for the chunk's output rows
  // r = (s * Hq + hq) * (N - q_off) + position - q_off to o_part [kv_split][rows][d_io] and
  // lse_part [kv_split][rows], which launch_prefill_combine merges.  1: no split.
  int32_t kv_split;
  float* o_part;
  float* lse_part;
};
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);
// Merge the kv_split partials of `rows` output rows (layout as PrefillArgs::o_part) into
// out [rows][d_io] of out_dtype and lse (nullable, fp32 natural log).
cudaError_t launch_prefill_combine(const float* o_part, const float* lse_part, int64_t rows, int32_t d_io,
                                   int32_t kv_split, void* out, sl8_dtype out_dtype, float* lse, cudaStream_t s);

struct DecodeArgs {
  const void* q;
  sl8_dtype q_dtype;
  const int8_t* k_cache;
  const float* k_scale;
  const int8_t* v_cache;
  const float* v_scale;
  const int32_t* seqlens;
  int32_t B, Hq, Hkv, Lmax, d, num_splits, split_size;
  float* o_partial;
  float* lse_partial;
  int32_t* logits;   // debug: [B][Hq][Lmax] int32 (nullable)
  int8_t* q_codes;   // nullable
  float* q_scales;   // nullable
  // paged cache (block_table non-null): k_cache / v_cache are pages [num_pages][Hkv]
  // [page_size][d], the scales [num_pages][Hkv][page_size]; token t of sequence b is
  // row t % page_size of page block_table[b * max_blocks + t / page_size]; Lmax is
  // max_blocks * page_size
  const int32_t* block_table;
  int32_t page_size, max_blocks, num_pages;
  // fp16 V cache (v_cache holds [B][Hkv][Lmax][d] fp16 values, v_scale unused); d <= 128,
  // contiguous caches only
  bool v16;
  // speculative verify (verify_T > 0): the verify_T draft queries of cache sequence b
  // (q [B_cache][T][Hq][d]) go verify_dps at a time into the query columns of one slot
  // (verify_dps * G <= 8): B counts B_cache * verify_ng virtual sequences v = b * verify_ng
  // + group, group g holding drafts g * verify_dps ..; seqlens and the caches are indexed
  // by b = v / verify_ng.  The last verify_T positions of b are the draft tokens: draft
  // query t sees draft token u iff bit u of tree_mask[b * verify_T + t] is set.  The
  // partials are [B_cache * T][Hq][S][d], row (b * T + t) * Hq + hq.
  int32_t verify_T, verify_dps, verify_ng;
  const uint32_t* tree_mask;
  // query heads per kv head above 8 (MQA): each cache kv head serves kv_groups virtual kv
  // heads of Hq / Hkv <= 8 query heads each.  Hkv here counts the virtual heads (the
  // cache holds Hkv / kv_groups), so virtual head hv reads cache head hv / kv_groups and
  // its query columns are heads hv * (Hq / Hkv) + c, i.e. consecutive groups of the cache
  // head's query heads.  1 otherwise.
  int32_t kv_groups;
};
cudaError_t launch_decode_split(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_combine(const float* o_partial, const float* lse_partial, const int32_t* seqlens,
                                  int32_t B, int32_t Hq, int32_t d, int32_t num_splits, int32_t split_size,
                                  void* out, sl8_dtype out_dtype, float* lse_out, cudaStream_t s,
                                  int32_t seq_div = 1);
cudaError_t launch_timeout_selftest(uint64_t limit_ns, cudaStream_t s);

// tokens per stage of the decode kernel for head dim d
int decode_chunk_tokens(int d);

// 3-D tiled tensor map, zero fill out of bounds, 128-byte swizzle (or none); *ok = false
// on failure.
CUtensorMap make_tmap_3d(const void* base, CUtensorMapDataType dt, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                         bool* ok, bool swizzle128 = true);

}  // namespace sl8
