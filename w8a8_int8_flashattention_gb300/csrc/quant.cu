// Quantisation-side kernels of the W8A8 path:
//   - the prefill scheduler (per-sequence table + longest-first work list),
//   - the K channel mean used for K-smoothing,
//   - symmetric per-row int8 quantisation (into the padded bf16-code workspace
//     for prefill, and the plain int8 form behind sl8_quant_rowwise),
//   - export of workspace codes to the caller's int8 layout (debug/parity).
//
// Operations: the "SuperL8" README (github.com/jajmangold/superl8), "Supporting
// kernels" table (quant_rowwise: symmetric per-row int8) and "Quantization" table
// (per-row int8: symmetric, K-smoothing).  Reading taken for the arithmetic:
// s = max|x| / 127 as an IEEE fp32 division, code = clamp(round-half-even(x / s),
// -127, 127), a row with s == 0 gets zero codes; the K mean sums fp32 in fixed
// 64-token chunks in ascending token order, then the chunk sums in ascending
// order, then divides by the token count.  This file is built without fast-math
// and spells every rounding step as an explicit _rn intrinsic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sl8_internal.h"

namespace sl8 {

// ---------------------------------------------------------------- element loads
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ float f16_bits_to_float(uint32_t b) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
}

template <sl8_dtype DT>
__device__ __forceinline__ float load_elem(const void* base, int64_t i) {
  if constexpr (DT == SL8_F32) {
    return static_cast<const float*>(base)[i];
  } else {
    const uint32_t b = static_cast<const uint16_t*>(base)[i];
    return DT == SL8_BF16 ? bf16_bits_to_float(b) : f16_bits_to_float(b);
  }
}

// EPL consecutive 16-bit elements starting at element index i (16-bit aligned by the caller's layout).
template <sl8_dtype DT, int EPL>
__device__ __forceinline__ void load_vec16(const void* base, int64_t i, float (&x)[EPL]) {
  const uint16_t* p = static_cast<const uint16_t*>(base) + i;
  uint16_t h[EPL];
  if constexpr (EPL == 8) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    memcpy(h, &v, 16);
  } else if constexpr (EPL == 4) {
    uint2 v = *reinterpret_cast<const uint2*>(p);
    memcpy(h, &v, 8);
  } else {
    uint32_t v = *reinterpret_cast<const uint32_t*>(p);
    memcpy(h, &v, 4);
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) x[e] = DT == SL8_BF16 ? bf16_bits_to_float(h[e]) : f16_bits_to_float(h[e]);
}

// One quantised value: clamp(RNE(x / s), -127, 127) with an IEEE division.  s > 0.
__device__ __forceinline__ int quant_code(float x, float s) {
  int c = __float2int_rn(__fdiv_rn(x, s));
  return c > 127 ? 127 : (c < -127 ? -127 : c);
}

__device__ __forceinline__ float warp_max(float a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  return a;
}

// bf16 bit pattern of a small integer code (|c| <= 127 is exact in bf16).
__device__ __forceinline__ uint16_t code_to_bf16_bits(int c) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(static_cast<float>(c)));
}

// ---------------------------------------------------------------- scheduler
// Exclusive prefix sum of v over the 1024 threads of the block; *total gets the sum.
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t* s_warp, int32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) s_warp[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    int32_t w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  *total = s_warp[31];
  return inc - v + (wid > 0 ? s_warp[wid - 1] : 0);
}

// One CTA of 1024 threads.  Fills the per-sequence table (length, first token, first
// padded row; sequences start on 128-row boundaries of the code workspace) and the work
// list of (sequence, item) pairs, an item being `item_rows` consecutive query rows.
// Order: by item index from the largest down (under a causal mask the last item of a
// sequence has the most key tiles), sequences with more items first within a level.
__global__ void __launch_bounds__(1024) schedule_kernel(const int32_t* __restrict__ cu, int32_t nseq, int32_t N,
                                                        int64_t total_tokens, int64_t t_pad_max, SeqTable t,
                                                        int32_t max_items, int32_t item_rows, DeviceStatus* st) {
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_fits;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int H = max_items + 2;
  int32_t* bucket = t.hist;             // [H] counts, then bucket starts
  int32_t* fill = t.hist + H;           // [H]
  int32_t* level_off = t.hist + 2 * H;  // [H]
  for (int i = tid; i < 3 * H; i += nt) t.hist[i] = 0;
  __syncthreads();
  for (int s = tid; s < nseq; s += nt) {
    int32_t L = N, tok0 = s * N;
    if (cu) {
      tok0 = cu[s];
      L = cu[s + 1] - cu[s];
      if (L < 0 || L > N || tok0 < 0 || static_cast<int64_t>(tok0) + L > total_tokens) {
        record_status(st, kStatusBadArg, 900);
        L = L < 0 ? 0 : (L > N ? N : L);
        if (tok0 < 0 || tok0 >= total_tokens) { tok0 = 0; L = 0; }
        if (static_cast<int64_t>(tok0) + L > total_tokens) L = static_cast<int32_t>(total_tokens - tok0);
      }
    }
    t.len[s] = L;
    t.tok0[s] = tok0;
    atomicAdd(&bucket[(L + item_rows - 1) / item_rows], 1);
  }
  __syncthreads();
  // padded row starts: exclusive scan of ceil(L / 128) * 128 in sequence order
  const int per = (nseq + nt - 1) / nt;
  const int b = tid * per, e = min(b + per, nseq);
  int32_t acc = 0;
  for (int s = b; s < e; ++s) acc += ((t.len[s] + kQTile - 1) / kQTile) * kPadRows;
  int32_t rows_total = 0;
  acc = block_exclusive_scan(acc, s_warp, &rows_total);
  for (int s = b; s < e; ++s) {
    t.pstart[s] = acc;
    acc += ((t.len[s] + kQTile - 1) / kQTile) * kPadRows;
  }
  if (tid == 0) {
    const bool fits = rows_total <= t_pad_max;  // overlapping sequences could overflow the workspace
    if (!fits) record_status(st, kStatusBadArg, 902);
    s_fits = fits;
    t.counts[1] = fits ? rows_total : 0;
    // buckets in descending item count: start of bucket n = number of sequences with more than n items
    int32_t r = 0;
    for (int n = max_items; n >= 0; --n) {
      const int32_t c = bucket[n];
      bucket[n] = r;
      r += c;
    }
    // level it holds the bucket[it] sequences with more than it items; levels run from the
    // largest item index down
    int32_t o = 0;
    for (int it = max_items - 1; it >= 0; --it) {
      level_off[it] = o;
      o += bucket[it];
    }
    t.counts[0] = fits ? o : 0;
  }
  __syncthreads();
  for (int s = tid; s < nseq; s += nt) {
    const int nit = (t.len[s] + item_rows - 1) / item_rows;
    const int slot = atomicAdd(&fill[nit], 1);
    t.sorted[bucket[nit] + slot] = s;
  }
  __syncthreads();
  const int32_t P = s_fits ? t.counts[0] : 0;
  for (int32_t p = tid; p < P; p += nt) {
    // level_off does not increase with the item index and only empty levels share an
    // offset with the next lower one, so p belongs to the smallest level whose offset <= p
    int lo = 0, hi = max_items - 1;
    while (lo < hi) {
      const int mid = (lo + hi) / 2;
      if (level_off[mid] <= p) hi = mid; else lo = mid + 1;
    }
    t.pair_seq[p] = t.sorted[p - level_off[lo]];
    t.pair_qt[p] = lo;
  }
}

cudaError_t launch_schedule(const int32_t* cu_seqlens, int32_t nseq, int32_t N, int64_t total_tokens,
                            int64_t t_pad_max, const SeqTable& t, int32_t item_rows, cudaStream_t s) {
  TraceScope tr("schedule", s);
  const int32_t max_items = (N + item_rows - 1) / item_rows;
  schedule_kernel<<<1, 1024, 0, s>>>(cu_seqlens, nseq, N, total_tokens, t_pad_max, t, max_items, item_rows,
                                     device_status_ptr());
  return cudaGetLastError();
}

// ---------------------------------------------------------------- K channel mean
// Row offset (elements) of token t of sequence s, head h.
__device__ __forceinline__ int64_t row_offset(bool varlen, int32_t s, int32_t h, int32_t t, int32_t H, int32_t N,
                                              int32_t d, int32_t tok0) {
  return varlen ? (static_cast<int64_t>(tok0 + t) * H + h) * d : ((static_cast<int64_t>(s) * H + h) * N + t) * d;
}

// One CTA per (64-token chunk, kv head, sequence), one thread per channel:
//   k_partials (nullable): fp32 sum of the chunk's K values per channel, in token order;
//   v_partials (nullable): max |V| over the chunk (V is bf16 whenever this is asked for).
template <sl8_dtype DT>
__global__ void kv_stats_partial_kernel(const void* __restrict__ k, const void* __restrict__ v, bool varlen,
                                        int32_t Hkv, int32_t N, int32_t d, const int32_t* __restrict__ len,
                                        const int32_t* __restrict__ tok0, float* __restrict__ k_partials,
                                        float* __restrict__ v_partials, int32_t max_chunks) {
  __shared__ float s_max[32];
  const int ch = blockIdx.x, h = blockIdx.y, s = blockIdx.z, c = threadIdx.x;
  const int L = len[s];
  const int t0 = ch * kMeanChunk;
  if (t0 >= L) return;
  const int t1 = min(t0 + kMeanChunk, L);
  const int32_t base = varlen ? tok0[s] : 0;
  const bool active = c < d;
  const int64_t slot = (static_cast<int64_t>(s) * Hkv + h) * max_chunks + ch;
  if (k_partials && active) {
    float part = 0.0f;
    for (int t = t0; t < t1; ++t)
      part = __fadd_rn(part, load_elem<DT>(k, row_offset(varlen, s, h, t, Hkv, N, d, base) + c));
    k_partials[slot * d + c] = part;
  }
  if (v_partials) {
    float m = 0.0f;
    if (active)
      for (int t = t0; t < t1; ++t)
        m = fmaxf(m, fabsf(load_elem<SL8_BF16>(v, row_offset(varlen, s, h, t, Hkv, N, d, base) + c)));
    m = warp_max(m);
    if ((c & 31) == 0) s_max[c / 32] = m;
    __syncthreads();
    if (c == 0) {
      for (int w = 1; w < (static_cast<int>(blockDim.x) + 31) / 32; ++w) m = fmaxf(m, s_max[w]);
      v_partials[slot] = m;
    }
  }
}

// One CTA per (kv head, sequence): K mean = (chunk sums added in chunk order) / L, and
// the power-of-two exponent e >= 0 with max|V| * 2^-e <= 2^15, so that V * 2^-e is
// exact in fp16 (up to fp16 subnormals) and cannot overflow.
__global__ void kv_stats_finalize_kernel(const float* __restrict__ k_partials, const float* __restrict__ v_partials,
                                         const int32_t* __restrict__ len, int32_t Hkv, int32_t d, int32_t max_chunks,
                                         float* __restrict__ mean, int32_t* __restrict__ v_exp) {
  const int h = blockIdx.x, s = blockIdx.y, c = threadIdx.x;
  const int L = len[s];
  const int nch = (L + kMeanChunk - 1) / kMeanChunk;
  const int64_t row = static_cast<int64_t>(s) * Hkv + h;
  if (k_partials && c < d) {
    const float* p = k_partials + row * max_chunks * d + c;
    float total = 0.0f;
    for (int ch = 0; ch < nch; ++ch) total = __fadd_rn(total, p[static_cast<int64_t>(ch) * d]);
    mean[row * d + c] = L > 0 ? __fdiv_rn(total, static_cast<float>(L)) : 0.0f;
  }
  if (v_partials && c == 0) {
    float m = 0.0f;
    for (int ch = 0; ch < nch; ++ch) m = fmaxf(m, v_partials[row * max_chunks + ch]);
    int e = 0;
    if (m > 0.0f) {
      int k2 = 0;
      frexpf(m, &k2);  // m < 2^k2
      e = k2 > 15 ? k2 - 15 : 0;
    }
    v_exp[row] = e;
  }
}

cudaError_t launch_kv_stats(const void* k, sl8_dtype dt, const void* v, bool varlen, int32_t nseq, int32_t Hkv,
                            int32_t N, int32_t d, const int32_t* len, const int32_t* tok0, float* k_partials,
                            float* v_partials, int32_t max_chunks, float* mean, int32_t* v_exp, cudaStream_t s) {
  {
    TraceScope tr("kv_stats_partial", s);
    dim3 grid(max_chunks, Hkv, nseq);
    const int threads = (d + 31) / 32 * 32;
    switch (dt) {
      case SL8_BF16: kv_stats_partial_kernel<SL8_BF16><<<grid, threads, 0, s>>>(k, v, varlen, Hkv, N, d, len, tok0, k_partials, v_partials, max_chunks); break;
      case SL8_F16: kv_stats_partial_kernel<SL8_F16><<<grid, threads, 0, s>>>(k, v, varlen, Hkv, N, d, len, tok0, k_partials, v_partials, max_chunks); break;
      default: kv_stats_partial_kernel<SL8_F32><<<grid, threads, 0, s>>>(k, v, varlen, Hkv, N, d, len, tok0, k_partials, v_partials, max_chunks); break;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  TraceScope tr("kv_stats_finalize", s);
  kv_stats_finalize_kernel<<<dim3(Hkv, nseq), (d + 31) / 32 * 32, 0, s>>>(k_partials, v_partials, len, Hkv, d,
                                                                           max_chunks, mean, v_exp);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- prefill codes
// One warp quantises one row of d = 32 * EPL values.  Rows live in the padded code
// workspace [H][t_pad][d]; padded rows past a sequence's end are written as zeros.
constexpr int kQuantWarps = 8;
constexpr int kQuantRowsPerWarp = 4;

// With v16 set (the K pass when V is bf16), each warp also writes the same row of V
// as fp16, scaled by the sequence/head's 2^-v_exp (exact), into v16 [H][t_pad][d].
template <sl8_dtype DT, int EPL>
__global__ void __launch_bounds__(kQuantWarps * 32) quant_codes_kernel(
    const void* __restrict__ x, bool varlen, int32_t nseq, int32_t H, int32_t N, int64_t total_tokens, SeqTable t,
    int64_t t_pad_max, const float* __restrict__ mean, uint16_t* __restrict__ codes, float* __restrict__ scales,
    const void* __restrict__ v, const int32_t* __restrict__ v_exp, uint16_t* __restrict__ v16, DeviceStatus* st) {
  constexpr int D = 32 * EPL;
  const int h = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int32_t rows_used = t.counts[1];
  const int64_t row0 = (static_cast<int64_t>(blockIdx.x) * kQuantWarps + warp) * kQuantRowsPerWarp;
  for (int r = 0; r < kQuantRowsPerWarp; ++r) {
    const int64_t pr = row0 + r;
    if (pr >= rows_used || pr >= t_pad_max) return;
    // sequence owning padded row pr: the last s with pstart[s] <= pr
    int lo = 0, hi = nseq - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (t.pstart[mid] <= pr) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int32_t tt = static_cast<int32_t>(pr - t.pstart[s]);
    const int32_t L = t.len[s];
    uint16_t* crow = codes + (static_cast<int64_t>(h) * t_pad_max + pr) * D + lane * EPL;
    float* srow = scales + static_cast<int64_t>(h) * t_pad_max + pr;
    bool valid = tt < L;
    if (valid && varlen && static_cast<int64_t>(t.tok0[s]) + tt >= total_tokens) {
      if (lane == 0) record_status(st, kStatusBadArg, 901);
      valid = false;
    }
    uint16_t out[EPL];
    float scale = 0.0f;
    if (valid) {
      float v[EPL];
      load_vec16<DT, EPL>(x, row_offset(varlen, s, h, tt, H, N, D, t.tok0[s]) + lane * EPL, v);
      if (mean) {
        const float* mu = mean + (static_cast<int64_t>(s) * H + h) * D + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e) v[e] = __fsub_rn(v[e], mu[e]);
      }
      float a = 0.0f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) a = fmaxf(a, fabsf(v[e]));
      a = warp_max(a);
      scale = __fdiv_rn(a, 127.0f);
#pragma unroll
      for (int e = 0; e < EPL; ++e) out[e] = scale == 0.0f ? 0 : code_to_bf16_bits(quant_code(v[e], scale));
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) out[e] = 0;
    }
    if constexpr (EPL == 8) {
      uint4 w; memcpy(&w, out, 16); *reinterpret_cast<uint4*>(crow) = w;
    } else if constexpr (EPL == 4) {
      uint2 w; memcpy(&w, out, 8); *reinterpret_cast<uint2*>(crow) = w;
    } else {
      uint32_t w; memcpy(&w, out, 4); *reinterpret_cast<uint32_t*>(crow) = w;
    }
    if (lane == 0) *srow = scale;
    if (v16) {
      uint16_t vo[EPL];
      if (valid) {
        float vv[EPL];
        load_vec16<SL8_BF16, EPL>(v, row_offset(varlen, s, h, tt, H, N, D, t.tok0[s]) + lane * EPL, vv);
        const float vscale = __int_as_float((127 - v_exp[static_cast<int64_t>(s) * H + h]) << 23);  // 2^-e
#pragma unroll
        for (int e = 0; e < EPL; ++e) vo[e] = __half_as_ushort(__float2half_rn(__fmul_rn(vv[e], vscale)));
      } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) vo[e] = 0;
      }
      uint16_t* vrow = v16 + (static_cast<int64_t>(h) * t_pad_max + pr) * D + lane * EPL;
      if constexpr (EPL == 8) {
        uint4 w; memcpy(&w, vo, 16); *reinterpret_cast<uint4*>(vrow) = w;
      } else if constexpr (EPL == 4) {
        uint2 w; memcpy(&w, vo, 8); *reinterpret_cast<uint2*>(vrow) = w;
      } else {
        uint32_t w; memcpy(&w, vo, 4); *reinterpret_cast<uint32_t*>(vrow) = w;
      }
    }
  }
}

template <sl8_dtype DT>
static cudaError_t launch_quant_codes_dt(const void* x, bool varlen, int32_t nseq, int32_t H, int32_t N, int32_t d,
                                         int64_t total_tokens, const SeqTable& t, int64_t t_pad_max,
                                         const float* mean, uint16_t* codes, float* scales, const void* v,
                                         const int32_t* v_exp, uint16_t* v16, cudaStream_t s) {
  const int64_t rows_per_cta = kQuantWarps * kQuantRowsPerWarp;
  dim3 grid(static_cast<unsigned>((t_pad_max + rows_per_cta - 1) / rows_per_cta), H);
  DeviceStatus* st = device_status_ptr();
  switch (d) {
    case 64: quant_codes_kernel<DT, 2><<<grid, kQuantWarps * 32, 0, s>>>(x, varlen, nseq, H, N, total_tokens, t, t_pad_max, mean, codes, scales, v, v_exp, v16, st); break;
    case 128: quant_codes_kernel<DT, 4><<<grid, kQuantWarps * 32, 0, s>>>(x, varlen, nseq, H, N, total_tokens, t, t_pad_max, mean, codes, scales, v, v_exp, v16, st); break;
    default: quant_codes_kernel<DT, 8><<<grid, kQuantWarps * 32, 0, s>>>(x, varlen, nseq, H, N, total_tokens, t, t_pad_max, mean, codes, scales, v, v_exp, v16, st); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_quant_codes(const void* x, sl8_dtype dt, bool varlen, int32_t nseq, int32_t H, int32_t N, int32_t d,
                               int64_t total_tokens, const SeqTable& t, int64_t t_pad_max, const float* mean,
                               uint16_t* codes, float* scales, const void* v, const int32_t* v_exp, uint16_t* v16,
                               bool is_k, cudaStream_t s) {
  TraceScope tr(is_k ? "quant_k" : "quant_q", s);
  if (dt == SL8_BF16)
    return launch_quant_codes_dt<SL8_BF16>(x, varlen, nseq, H, N, d, total_tokens, t, t_pad_max, mean, codes, scales,
                                           v, v_exp, v16, s);
  return launch_quant_codes_dt<SL8_F16>(x, varlen, nseq, H, N, d, total_tokens, t, t_pad_max, mean, codes, scales, v,
                                        v_exp, v16, s);
}

// ---------------------------------------------------------------- generic rowwise int8
// One warp per row of any width; two passes (max, then codes) over the row.
template <sl8_dtype DT>
__global__ void __launch_bounds__(256) quant_rowwise_kernel(const void* __restrict__ x, int64_t rows, int32_t cols,
                                                            int64_t row_stride, const float* __restrict__ sub_mean,
                                                            int64_t rows_per_group, int8_t* __restrict__ q_out,
                                                            float* __restrict__ scale_out) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int64_t base = row * row_stride;
  const float* mu = sub_mean ? sub_mean + (row / rows_per_group) * cols : nullptr;
  float a = 0.0f;
  for (int c = lane; c < cols; c += 32) {
    float v = load_elem<DT>(x, base + c);
    if (mu) v = __fsub_rn(v, mu[c]);
    a = fmaxf(a, fabsf(v));
  }
  a = warp_max(a);
  const float s = __fdiv_rn(a, 127.0f);
  int8_t* q = q_out + row * cols;
  for (int c = lane; c < cols; c += 32) {
    float v = load_elem<DT>(x, base + c);
    if (mu) v = __fsub_rn(v, mu[c]);
    q[c] = s == 0.0f ? 0 : static_cast<int8_t>(quant_code(v, s));
  }
  if (lane == 0) scale_out[row] = s;
}

cudaError_t launch_quant_rowwise(const void* x, sl8_dtype dt, int64_t rows, int32_t cols, int64_t row_stride,
                                 const float* sub_mean, int64_t rows_per_group, int8_t* q_out, float* scale_out,
                                 cudaStream_t s) {
  TraceScope tr("quant_rowwise", s);
  const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
  switch (dt) {
    case SL8_BF16: quant_rowwise_kernel<SL8_BF16><<<grid, 256, 0, s>>>(x, rows, cols, row_stride, sub_mean, rows_per_group, q_out, scale_out); break;
    case SL8_F16: quant_rowwise_kernel<SL8_F16><<<grid, 256, 0, s>>>(x, rows, cols, row_stride, sub_mean, rows_per_group, q_out, scale_out); break;
    default: quant_rowwise_kernel<SL8_F32><<<grid, 256, 0, s>>>(x, rows, cols, row_stride, sub_mean, rows_per_group, q_out, scale_out); break;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------- export codes
// Workspace bf16 codes [H][t_pad][d] -> caller's int8 layout (dense [nseq,H,N,d] or
// packed [T,H,d]) and scales (dense [nseq,H,N] or packed [T,H]).
__global__ void export_codes_kernel(const uint16_t* __restrict__ codes, const float* __restrict__ scales, bool varlen,
                                    int32_t nseq, int32_t H, int32_t N, int32_t d, SeqTable t, int64_t t_pad_max,
                                    int8_t* __restrict__ codes_out, float* __restrict__ scales_out) {
  const int s = blockIdx.y, h = blockIdx.z;
  const int32_t L = t.len[s];
  const int32_t tok = blockIdx.x;
  if (tok >= L) return;
  const int64_t src = static_cast<int64_t>(h) * t_pad_max + t.pstart[s] + tok;
  const int64_t dst_row = varlen ? (static_cast<int64_t>(t.tok0[s]) + tok) * H + h
                                 : (static_cast<int64_t>(s) * H + h) * N + tok;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    const float v = __bfloat162float(__ushort_as_bfloat16(codes[src * d + c]));
    codes_out[dst_row * d + c] = static_cast<int8_t>(__float2int_rn(v));
  }
  if (threadIdx.x == 0) scales_out[dst_row] = scales[src];
}

cudaError_t launch_export_codes(const uint16_t* codes, const float* scales, bool varlen, int32_t nseq, int32_t H,
                                int32_t N, int32_t d, const SeqTable& t, int64_t t_pad_max, int8_t* codes_out,
                                float* scales_out, cudaStream_t s) {
  TraceScope tr("export_codes", s);
  export_codes_kernel<<<dim3(N, nseq, H), 64, 0, s>>>(codes, scales, varlen, nseq, H, N, d, t, t_pad_max, codes_out,
                                                       scales_out);
  return cudaGetLastError();
}

}  // namespace sl8
