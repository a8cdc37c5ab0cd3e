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
#include <atomic>
#include <cstring>

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

// Round-half-even of |y| < 2^22 to an integer-valued float, in two additions.
__device__ __forceinline__ float rint_add(float y) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: its ulp is 1
  return __fsub_rn(__fadd_rn(y, kMagic), kMagic);
}
// Packed f32x2 arithmetic (two lanes per instruction, each rounded like its scalar op).
__device__ __forceinline__ uint64_t q_pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void q_upk2(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t q_mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t q_add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t q_sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Three-input max (one instruction).
__device__ __forceinline__ float q_max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// The same code as an integer-valued float, from rs = RN(1 / s): for |x / s| <= 127.5 the
// product x * rs lies within 3e-5 of the correctly rounded quotient, so both round to
// the same integer unless the product is within 1e-4 of a half-integer; only then is
// the quotient formed.
__device__ __forceinline__ float quant_code_rcp(float x, float s, float rs) {
  const float y = __fmul_rn(x, rs);
  float r = rint_add(y);
  if (fabsf(__fsub_rn(y, r)) > 0.4999f) r = rint_add(__fdiv_rn(x, s));
  return fminf(fmaxf(r, -127.0f), 127.0f);
}

__device__ __forceinline__ float warp_max(float a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  return a;
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
// The histogram lives in shared memory when it fits (kSmemHist), else in t.hist.  It
// also zeroes the n_done completion counters of the K/V statistics kernel.
template <bool kSmemHist>
__global__ void __launch_bounds__(1024) schedule_kernel(const int32_t* __restrict__ cu, int32_t nseq, int32_t N,
                                                        int64_t total_tokens, int64_t t_pad_max, SeqTable t,
                                                        int32_t max_items, int32_t item_rows, int32_t* kv_done,
                                                        int32_t n_done, DeviceStatus* st) {
  extern __shared__ int32_t sh_hist[];
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_fits;
  grid_dependency_wait();
  const int tid = threadIdx.x, nt = blockDim.x;
  const int H = max_items + 2;
  int32_t* hist = kSmemHist ? sh_hist : t.hist;
  int32_t* bucket = hist;           // [H] counts, then bucket starts
  int32_t* fill = hist + H;         // [H]
  int32_t* level_off = hist + 2 * H;  // [H]
  for (int i = tid; i < 3 * H; i += nt) hist[i] = 0;
  for (int i = tid; i < n_done; i += nt) kv_done[i] = 0;
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
  grid_dependents_launch();
}

cudaError_t launch_schedule(const int32_t* cu_seqlens, int32_t nseq, int32_t N, int64_t total_tokens,
                            int64_t t_pad_max, const SeqTable& t, int32_t item_rows, int32_t* kv_done,
                            int32_t n_done, cudaStream_t s) {
  TraceScope tr("schedule", s);
  const int32_t max_items = (N + item_rows - 1) / item_rows;
  const size_t hist_bytes = static_cast<size_t>(3) * (max_items + 2) * 4;
  if (hist_bytes <= 32768)
    return launch_pdl(schedule_kernel<true>, dim3(1), dim3(1024), hist_bytes, s, cu_seqlens, nseq, N, total_tokens,
                      t_pad_max, t, max_items, item_rows, kv_done, n_done, device_status_ptr());
  return launch_pdl(schedule_kernel<false>, dim3(1), dim3(1024), 0, s, cu_seqlens, nseq, N, total_tokens, t_pad_max,
                    t, max_items, item_rows, kv_done, n_done, device_status_ptr());
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
// The chunk's loads are issued kBatch at a time before they are summed in order.  The
// last CTA of a (sequence, kv head) to finish (counted in done) then forms the K mean
// = (chunk sums added in chunk order) / L, and the power-of-two exponent e >= 0 with
// max|V| * 2^-e <= 2^15, so that V * 2^-e is exact in fp16 (up to fp16 subnormals)
// and cannot overflow.
template <sl8_dtype DT, int kMaxThreads>
__global__ void __launch_bounds__(kMaxThreads) kv_stats_kernel(
    const void* __restrict__ k, const void* __restrict__ v, bool varlen, int32_t Hkv, int32_t N, int32_t d,
    const int32_t* __restrict__ len, const int32_t* __restrict__ tok0, float* __restrict__ k_partials,
    float* __restrict__ v_partials, int32_t max_chunks, float* __restrict__ mean, int32_t* __restrict__ v_exp,
    int32_t* __restrict__ done) {
  constexpr int kBatch = kMaxThreads <= 256 ? 32 : 16;
  __shared__ float s_max[32];
  __shared__ int s_last;
  grid_dependency_wait();
  const int ch = blockIdx.x, h = blockIdx.y, s = blockIdx.z, c = threadIdx.x;
  const int L = len[s];
  const int t0 = ch * kMeanChunk;
  if (t0 >= L) return;
  const int t1 = min(t0 + kMeanChunk, L);
  const int nch = (L + kMeanChunk - 1) / kMeanChunk;
  const int32_t base = varlen ? tok0[s] : 0;
  const bool active = c < d;
  const int64_t row = static_cast<int64_t>(s) * Hkv + h;
  const int64_t slot = row * max_chunks + ch;
  // element (t0 + i, c) sits at row_offset(t0) + c + i * stride
  const int64_t e0 = row_offset(varlen, s, h, t0, Hkv, N, d, base) + c;
  const int stride = varlen ? Hkv * d : d;
  if (k_partials && active) {
    float part = 0.0f;
    for (int tb = 0; tb < t1 - t0; tb += kBatch) {
      float x[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        x[i] = tb + i < t1 - t0 ? load_elem<DT>(k, e0 + static_cast<int64_t>((tb + i) * stride)) : 0.0f;
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        if (tb + i < t1 - t0) part = __fadd_rn(part, x[i]);
    }
    k_partials[slot * d + c] = part;
  }
  if (v_partials) {
    float m = 0.0f;
    if (active) {
      for (int tb = 0; tb < t1 - t0; tb += kBatch) {
        float x[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
          x[i] = tb + i < t1 - t0 ? load_elem<SL8_BF16>(v, e0 + static_cast<int64_t>((tb + i) * stride)) : 0.0f;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) m = fmaxf(m, fabsf(x[i]));
      }
    }
    m = warp_max(m);
    if ((c & 31) == 0) s_max[c / 32] = m;
    __syncthreads();
    if (c == 0) {
      for (int w = 1; w < (static_cast<int>(blockDim.x) + 31) / 32; ++w) m = fmaxf(m, s_max[w]);
      v_partials[slot] = m;
    }
  }
  // ---- the last chunk of (s, h) finalises
  __threadfence();
  __syncthreads();
  if (c == 0) s_last = atomicAdd(&done[row], 1) == nch - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (k_partials && active) {
    const float* p = k_partials + row * max_chunks * d + c;
    float total = 0.0f;
    for (int cb = 0; cb < nch; cb += kBatch) {
      float x[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) x[i] = cb + i < nch ? p[static_cast<int64_t>(cb + i) * d] : 0.0f;
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        if (cb + i < nch) total = __fadd_rn(total, x[i]);
    }
    mean[row * d + c] = __fdiv_rn(total, static_cast<float>(L));
  }
  if (v_partials) {
    float m = 0.0f;
    for (int cb = c; cb < nch; cb += blockDim.x) m = fmaxf(m, v_partials[row * max_chunks + cb]);
    m = warp_max(m);
    __syncthreads();
    if ((c & 31) == 0) s_max[c / 32] = m;
    __syncthreads();
    if (c == 0) {
      for (int w = 1; w < (static_cast<int>(blockDim.x) + 31) / 32; ++w) m = fmaxf(m, s_max[w]);
      int e = 0;
      if (m > 0.0f) {
        int k2 = 0;
        frexpf(m, &k2);  // m < 2^k2
        e = k2 > 15 ? k2 - 15 : 0;
      }
      v_exp[row] = e;
    }
  }
}

// The same statistics with 16-byte loads: a thread owns VW consecutive channels of one
// chunk (d / VW threads per chunk, 128 / (d / VW) chunks of one (sequence, kv head) per
// CTA), so a CTA keeps 16 rows of 16-byte loads per thread in flight.  Each channel is
// still summed in token order.  Requires d % VW == 0, d / VW <= 32 and V (if any) in
// bf16 with K in a 16-bit type.
template <sl8_dtype DT>
__global__ void __launch_bounds__(128) kv_stats_vec_kernel(
    const void* __restrict__ k, const void* __restrict__ v, bool varlen, int32_t Hkv, int32_t N, int32_t d,
    const int32_t* __restrict__ len, const int32_t* __restrict__ tok0, float* __restrict__ k_partials,
    float* __restrict__ v_partials, int32_t max_chunks, float* __restrict__ mean, int32_t* __restrict__ v_exp,
    int32_t* __restrict__ done) {
  constexpr int VW = DT == SL8_F32 ? 4 : 8;  // channels per 16-byte load
  constexpr int kBatch = 16;
  __shared__ float s_max[4];
  __shared__ int s_last;
  grid_dependency_wait();
  const int tpi = d / VW, ipc = 128 / tpi;
  const int h = blockIdx.y, s = blockIdx.z, tid = threadIdx.x;
  const int item = tid / tpi, sub = tid % tpi;
  const int L = len[s];
  const int nch = (L + kMeanChunk - 1) / kMeanChunk;
  const int n_cta = (nch + ipc - 1) / ipc;  // CTAs of (s, h) with work
  if (static_cast<int>(blockIdx.x) >= n_cta) return;
  const int ch = blockIdx.x * ipc + item;
  const bool active = item < ipc && ch < nch;
  const int64_t row = static_cast<int64_t>(s) * Hkv + h;
  const int c0 = sub * VW;
  float vmax = 0.0f;
  if (active) {
    const int t0 = ch * kMeanChunk, n = min(kMeanChunk, L - t0);
    const int32_t base = varlen ? tok0[s] : 0;
    const int64_t e0 = row_offset(varlen, s, h, t0, Hkv, N, d, base) + c0;
    const int64_t stride = varlen ? static_cast<int64_t>(Hkv) * d : d;
    const int64_t slot = row * max_chunks + ch;
    if (k_partials) {
      float part[VW];
#pragma unroll
      for (int e = 0; e < VW; ++e) part[e] = 0.0f;
      for (int tb = 0; tb < n; tb += kBatch) {
        uint4 w[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          w[i] = make_uint4(0u, 0u, 0u, 0u);
          if (tb + i < n) {
            const int64_t off = e0 + (tb + i) * stride;
            w[i] = DT == SL8_F32 ? *reinterpret_cast<const uint4*>(static_cast<const float*>(k) + off)
                                 : *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(k) + off);
          }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          if (tb + i >= n) continue;
          const uint32_t ww[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            float x;
            if constexpr (DT == SL8_F32) x = __uint_as_float(ww[e]);
            else {
              const uint32_t b = (e & 1) ? ww[e / 2] >> 16 : ww[e / 2] & 0xffffu;
              x = DT == SL8_BF16 ? bf16_bits_to_float(b) : f16_bits_to_float(b);
            }
            part[e] = __fadd_rn(part[e], x);
          }
        }
      }
      float* dst = k_partials + slot * d + c0;
#pragma unroll
      for (int e = 0; e < VW; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(part[e], part[e + 1], part[e + 2], part[e + 3]);
    }
    if (v_partials) {
      for (int tb = 0; tb < n; tb += kBatch) {
        uint4 w[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
          w[i] = tb + i < n ? *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(v) + e0 + (tb + i) * stride)
                            : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const uint32_t ww[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            vmax = fmaxf(vmax, fmaxf(fabsf(bf16_bits_to_float(ww[e] & 0xffffu)), fabsf(bf16_bits_to_float(ww[e] >> 16))));
        }
      }
    }
  }
  if (v_partials) {
    // max over the tpi threads of one chunk (aligned groups of lanes)
    for (int o = tpi / 2; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    if (active && sub == 0) v_partials[row * max_chunks + ch] = vmax;
  }
  // ---- the last CTA of (s, h) finalises
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&done[row], 1) == n_cta - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (k_partials) {
    for (int c = tid; c < d; c += blockDim.x) {
      const float* p = k_partials + row * max_chunks * d + c;
      float total = 0.0f;
      for (int cb = 0; cb < nch; cb += kBatch) {
        float x[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) x[i] = cb + i < nch ? p[static_cast<int64_t>(cb + i) * d] : 0.0f;
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
          if (cb + i < nch) total = __fadd_rn(total, x[i]);
      }
      mean[row * d + c] = __fdiv_rn(total, static_cast<float>(L));
    }
  }
  if (v_partials) {
    float m = 0.0f;
    for (int cb = tid; cb < nch; cb += blockDim.x) m = fmaxf(m, v_partials[row * max_chunks + cb]);
    m = warp_max(m);
    if ((tid & 31) == 0) s_max[tid / 32] = m;
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < 4; ++w) m = fmaxf(m, s_max[w]);
      int e = 0;
      if (m > 0.0f) {
        int k2 = 0;
        frexpf(m, &k2);  // m < 2^k2
        e = k2 > 15 ? k2 - 15 : 0;
      }
      v_exp[row] = e;
    }
  }
}

template <sl8_dtype DT>
static cudaError_t launch_kv_stats_dt(const void* k, const void* v, bool varlen, int32_t nseq, int32_t Hkv, int32_t N,
                                      int32_t d, const int32_t* len, const int32_t* tok0, float* k_partials,
                                      float* v_partials, int32_t max_chunks, float* mean, int32_t* v_exp,
                                      int32_t* done, cudaStream_t s) {
  constexpr int VW = DT == SL8_F32 ? 4 : 8;
  if (d % VW == 0 && d / VW <= 32 && (!v || DT != SL8_F32)) {
    const int ipc = 128 / (d / VW);
    return launch_pdl(kv_stats_vec_kernel<DT>, dim3((max_chunks + ipc - 1) / ipc, Hkv, nseq), dim3(128), 0, s, k, v,
                      varlen, Hkv, N, d, len, tok0, k_partials, v_partials, max_chunks, mean, v_exp, done);
  }
  const dim3 grid(max_chunks, Hkv, nseq);
  const int threads = (d + 31) / 32 * 32;
  if (threads <= 256)
    return launch_pdl(kv_stats_kernel<DT, 256>, grid, dim3(threads), 0, s, k, v, varlen, Hkv, N, d, len, tok0,
                      k_partials, v_partials, max_chunks, mean, v_exp, done);
  return launch_pdl(kv_stats_kernel<DT, 1024>, grid, dim3(threads), 0, s, k, v, varlen, Hkv, N, d, len, tok0,
                    k_partials, v_partials, max_chunks, mean, v_exp, done);
}

cudaError_t launch_kv_stats(const void* k, sl8_dtype dt, const void* v, bool varlen, int32_t nseq, int32_t Hkv,
                            int32_t N, int32_t d, const int32_t* len, const int32_t* tok0, float* k_partials,
                            float* v_partials, int32_t max_chunks, float* mean, int32_t* v_exp, int32_t* kv_done,
                            cudaStream_t s) {
  TraceScope tr("kv_stats", s);
  switch (dt) {
    case SL8_BF16: return launch_kv_stats_dt<SL8_BF16>(k, v, varlen, nseq, Hkv, N, d, len, tok0, k_partials, v_partials, max_chunks, mean, v_exp, kv_done, s);
    case SL8_F16: return launch_kv_stats_dt<SL8_F16>(k, v, varlen, nseq, Hkv, N, d, len, tok0, k_partials, v_partials, max_chunks, mean, v_exp, kv_done, s);
    default: return launch_kv_stats_dt<SL8_F32>(k, v, varlen, nseq, Hkv, N, d, len, tok0, k_partials, v_partials, max_chunks, mean, v_exp, kv_done, s);
  }
}

// ---------------------------------------------------------------- prefill K/V partials
// One CTA per (64-token chunk, kv head, sequence): the chunk's K rows (and V rows when
// v_partials is set) are staged in shared memory (dense: one bulk copy per tensor; varlen:
// one tiled copy per tensor of the chunk's rows of head h); then thread c < d sums
// channel c of K in token order into k_partials, while the second half of the CTA (with
// V) takes max |V| of the chunk into v_partials.  Dense input (len == nullptr): every
// sequence is N long.  kv_finalize_kernel forms the mean and the V exponent from these.
// d * sizeof(element) must be a multiple of 16; the block is 2 * ceil32(d) threads with V,
// ceil32(d) without.
template <sl8_dtype DT>
__global__ void kv_partials_kernel(const void* __restrict__ k, const void* __restrict__ v, bool varlen, int32_t Hkv,
                                   int32_t N, int32_t d, const int32_t* __restrict__ len,
                                   const int32_t* __restrict__ tok0, float* __restrict__ k_partials,
                                   float* __restrict__ v_partials, int32_t max_chunks,
                                   const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                                   uint64_t limit_ns, DeviceStatus* st) {
  extern __shared__ __align__(128) uint8_t stage[];
  __shared__ uint64_t bar;
  __shared__ float s_max[32];
  constexpr int ES = DT == SL8_F32 ? 4 : 2;
  grid_dependency_wait();
  grid_dependents_launch();
  const int ch = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int half = (d + 31) / 32 * 32;  // threads per role
  const bool v_role = v_partials && static_cast<int>(threadIdx.x) >= half;
  const int c = v_role ? threadIdx.x - half : threadIdx.x;
  const int L = len ? len[s] : N;
  const int t0 = ch * kMeanChunk;
  if (t0 >= L) return;
  const int n = min(kMeanChunk, L - t0);
  const int32_t base = varlen ? tok0[s] : 0;
  const uint32_t row_bytes = static_cast<uint32_t>(d) * ES;  // K rows; V rows are bf16
  const uint32_t v_row_bytes = static_cast<uint32_t>(d) * 2;
  uint8_t* sk = stage;
  uint8_t* sv = stage + kMeanChunk * row_bytes;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // dense: the chunk's rows are contiguous (one bulk copy); varlen: one tiled copy of the
    // chunk's 64 token rows of head h (rows past the sequence are read and ignored, rows
    // past the tensors zero-filled)
    const uint32_t rows = varlen ? static_cast<uint32_t>(kMeanChunk) : static_cast<uint32_t>(n);
    const uint32_t tx = rows * ((k_partials ? row_bytes : 0u) + (v_partials ? v_row_bytes : 0u));
    mbar_arrive_expect_tx(&bar, tx);
    if (!varlen) {
      const int64_t e0 = row_offset(false, s, h, t0, Hkv, N, d, 0);
      if (k_partials) bulk_load(sk, static_cast<const uint8_t*>(k) + e0 * ES, n * row_bytes, &bar);
      if (v_partials) bulk_load(sv, static_cast<const uint8_t*>(v) + e0 * 2, n * v_row_bytes, &bar);
    } else {
      if (k_partials) tma_load_3d(sk, &map_k, &bar, 0, h, base + t0);
      if (v_partials) tma_load_3d(sv, &map_v, &bar, 0, h, base + t0);
    }
  }
  const bool ok = mbar_wait(&bar, 0, limit_ns, st, 903);
  const int64_t slot = (static_cast<int64_t>(s) * Hkv + h) * max_chunks + ch;
  if (!v_role) {
    // channel c of K, summed in token order (16 rows' loads in flight at a time)
    if (k_partials && ok && c < d) {
      float part = 0.0f;
      for (int i0 = 0; i0 < n; i0 += 16) {
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          x[i] = 0.0f;
          if (i0 + i < n) {
            const uint8_t* p = sk + (i0 + i) * row_bytes + c * ES;
            x[i] = DT == SL8_F32 ? *reinterpret_cast<const float*>(p)
                 : DT == SL8_BF16 ? bf16_bits_to_float(*reinterpret_cast<const uint16_t*>(p))
                                  : f16_bits_to_float(*reinterpret_cast<const uint16_t*>(p));
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i0 + i < n) part = __fadd_rn(part, x[i]);
      }
      k_partials[slot * d + c] = part;
    }
  } else {
    // max |V| of the chunk: channel c of every row, then over the role's threads
    float m = 0.0f;
    if (ok && c < d)
      for (int i = 0; i < n; ++i)
        m = fmaxf(m, fabsf(bf16_bits_to_float(*reinterpret_cast<const uint16_t*>(sv + i * v_row_bytes + c * 2))));
    m = warp_max(m);
    if ((c & 31) == 0) s_max[c / 32] = m;
    named_bar_sync(1, half);
    if (c == 0) {
      for (int w = 1; w < half / 32; ++w) m = fmaxf(m, s_max[w]);
      v_partials[slot] = m;
    }
  }
}

cudaError_t launch_kv_partials(const void* k, sl8_dtype dt, const void* v, bool varlen, int32_t nseq, int32_t Hkv,
                               int32_t N, int32_t d, const int32_t* len, const int32_t* tok0, float* k_partials,
                               float* v_partials, int32_t max_chunks, int64_t total_tokens, cudaStream_t s) {
  TraceScope tr("kv_partials", s);
  const int es = dt == SL8_F32 ? 4 : 2;
  const size_t smem = static_cast<size_t>(kMeanChunk) * d * es * (v_partials ? 2 : 1);
  const int half = (d + 31) / 32 * 32;
  const dim3 grid(max_chunks, Hkv, nseq), block(v_partials ? 2 * half : half);
  CUtensorMap mk, mv;
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  if (varlen) {  // [T][Hkv][d]: 64 token rows of one head per copy
    bool ok = true;
    const uint64_t T = static_cast<uint64_t>(total_tokens), dd = static_cast<uint64_t>(d);
    const CUtensorMapDataType et = es == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
    if (k_partials) mk = make_tmap_3d(k, et, dd, Hkv, T, dd * es, dd * es * Hkv, d, 1, kMeanChunk, &ok, false);
    if (v_partials)
      mv = make_tmap_3d(v, CU_TENSOR_MAP_DATA_TYPE_UINT16, dd, Hkv, T, dd * 2, dd * 2 * Hkv, d, 1, kMeanChunk, &ok,
                        false);
    if (!ok) return cudaErrorInvalidValue;
  }
  auto go = [&](auto kern) {
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, grid, block, smem, s, k, v, varlen, Hkv, N, d, len, tok0, k_partials, v_partials,
                      max_chunks, mk, mv, spin_limit_ns(), device_status_ptr());
  };
  switch (dt) {
    case SL8_BF16: return go(kv_partials_kernel<SL8_BF16>);
    case SL8_F16: return go(kv_partials_kernel<SL8_F16>);
    default: return go(kv_partials_kernel<SL8_F32>);
  }
}

// ---------------------------------------------------------------- prefill codes
// Arguments of the prefill quantiser (Q and K rows in one launch).  Rows live in the padded
// code workspace [H][t_pad][d]; padded rows past a sequence's end are written as zeros.
// For K rows with v16 set (V bf16, or head dim 32 run as 64), the same rows of V are
// written as fp16 scaled by the sequence/head's 2^-v_exp (exact) into v16 [Hkv][t_pad][d].

struct QuantQK {
  const void* q;
  const void* k;
  bool varlen;
  int32_t nseq, Hq, Hkv, N;
  int32_t q_off;            // dense query chunk: q holds positions q_off .. N-1
  int32_t q_row0;           // dense: the first position whose Q row the attention reads (a
                            // multiple of 64 <= q_off); Q blocks before it are not written
  int32_t d_io;             // values per input row (<= D; the code rows are zero past them)
  bool v_f16;               // V is fp16 (copied as is) rather than bf16
  int64_t total_tokens;
  SeqTable t;
  int64_t t_pad_max;
  const float* k_partials;  // [nseq][Hkv][max_chunks][d] K chunk sums (nullable: no smoothing)
  const float* v_partials;  // [nseq][Hkv][max_chunks] V chunk abs-max (with v16)
  int32_t max_chunks;
  int32_t* v_exp_out;       // [nseq][Hkv] written by the first K CTA of each (s, h)
  uint16_t* q_codes;
  float* q_scales;
  uint16_t* k_codes;
  float* k_scales;
  const void* v;            // bf16 V when v16 is set
  uint16_t* v16;
  // grouped scales (attn_w8a8_fwd): rows [g*G, (g+1)*G) of a sequence share one scale,
  // G a power of two <= 64; Q rows above q_tau x their group's lower median max|x| keep
  // their own (q_tau 0: no outlier test).  Only the kGroups instantiation reads these.
  int32_t q_group, k_group;
  float q_tau;
};

// ---------------------------------------------------------------- K mean and V exponent
// One CTA per (sequence, kv head): the K mean = (the chunk sums of k_partials added in
// chunk order) / L per channel, and the V exponent e >= 0 with max|V| * 2^-e <= 2^15
// from the chunk maxima of v_partials (e = 0 without them).  Both are read by the K units
// of the quantiser and v_exp by the attention kernel.
__global__ void __launch_bounds__(128) kv_finalize_kernel(bool varlen, int32_t Hkv, int32_t N, int32_t d_io,
                                                          const int32_t* __restrict__ len,
                                                          const float* __restrict__ k_partials,
                                                          const float* __restrict__ v_partials, int32_t max_chunks,
                                                          float* __restrict__ mean, int32_t* __restrict__ v_exp) {
  __shared__ float s_max[4];
  // Let the quantiser launch at once, so that its Q blocks run alongside the chunk kernel.
  // That is safe: this kernel starts only after the chunk kernel has passed its own wait,
  // i.e. after every earlier kernel (the previous attention reading the code workspace)
  // completed; and the quantiser waits for this kernel before it reads the mean.
  grid_dependents_launch();
  grid_dependency_wait();
  const int h = blockIdx.x, s = blockIdx.y, tid = threadIdx.x;
  const int L = varlen ? len[s] : N;
  const int nch = (L + kMeanChunk - 1) / kMeanChunk;
  const int64_t row = static_cast<int64_t>(s) * Hkv + h;
  if (k_partials) {
    for (int c = tid; c < d_io; c += blockDim.x) {
      const float* p = k_partials + row * max_chunks * d_io + c;
      float total = 0.0f;
      // 64 chunk sums in flight per round trip (a 4096-token sequence in one), added in order
      for (int cb = 0; cb < nch; cb += 64) {
        float x[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = cb + i < nch ? p[static_cast<int64_t>(cb + i) * d_io] : 0.0f;
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (cb + i < nch) total = __fadd_rn(total, x[i]);
      }
      mean[row * d_io + c] = L > 0 ? __fdiv_rn(total, static_cast<float>(L)) : 0.0f;
    }
  }
  float m = 0.0f;
  if (v_partials)
    for (int cb = tid; cb < nch; cb += blockDim.x) m = fmaxf(m, v_partials[row * max_chunks + cb]);
  m = warp_max(m);
  if ((tid & 31) == 0) s_max[tid / 32] = m;
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < 4; ++w) m = fmaxf(m, s_max[w]);
    int e = 0;
    if (m > 0.0f) {
      int k2 = 0;
      frexpf(m, &k2);  // m < 2^k2
      e = k2 > 15 ? k2 - 15 : 0;
    }
    v_exp[row] = e;
  }
}

// ---------------------------------------------------------------- prefill codes, pipelined
// Persistent CTAs walk the 64-row blocks ("units") of the code workspace: first those of
// every Q head, then those of every kv head, a K unit followed by the V unit of the same
// rows when V is converted.  A producer warp stages each unit's input rows in shared
// memory with bulk copies, kStages units ahead; eight consumer warps turn a staged unit
// into codes and scales (a V unit: into fp16 V), eight lanes per row, while the next
// units load.  Every unit moves the same bytes, so the last units end together.  K and V
// units read the K mean and the V exponent that kv_finalize_kernel wrote (they wait for
// it, and through it for the K/V chunk kernel, before their first unit), so Q units
// overlap those kernels.
// The arithmetic is that of the per-row reading: s = max|x| / 127 (IEEE division), codes
// RNE(x / s) formed as x * (1/s) and checked against the half-integer boundaries (the
// exact quotient is formed for the few values near one), smoothed K = K - mean in fp32.
constexpr int kQpRows = 64;       // rows per unit (a unit never straddles two sequences)
constexpr int kQpConsumers = 8;   // consumer warps: 8 rows each, two passes of four

// Run-time claiming: CTA c takes unit c first, then the next unclaimed unit from a
// per-launch counter.  A launch uses the counter pair g_qp_claim[ticket] ([0] next unit -
// grid, [1] CTAs done); the last CTA to finish zeroes the pair for the next launch that
// draws the same ticket (tickets rotate over kQpTickets launches).
constexpr int kQpTickets = 64;
__device__ uint32_t g_qp_claim[kQpTickets][2];

// The unit's place, decoded once by the producer and handed to the consumers in the
// unit's shared-memory stage.
constexpr int32_t kQpDone = -1, kQpQ = 0, kQpK = 1, kQpV = 2;  // QpUnit::kind
struct QpUnit {
  int32_t kind, h, s, L, tk, t0, vexp, pad;
  int64_t row0;
};

template <int D>
struct QpCfg {
  static constexpr int kUnitBytes = kQpRows * D * 2;       // staged rows of <= D 16-bit values
  static constexpr int kStages = D == 256 ? 3 : (D == 128 ? 4 : 6);
  static constexpr int kMeanOff = kUnitBytes;              // input rows, K mean row
  static constexpr int kInfoOff = kMeanOff + D * 4;
  static constexpr int kStageBytes = kInfoOff + 128;
  static constexpr int kSmem = kStages * kStageBytes + 128;
  static constexpr int kThreads = (kQpConsumers + 1) * 32;
  static constexpr int kCtasPerSm = D == 256 ? 2 : 3;
  static_assert(kCtasPerSm * (kSmem + 1024) <= 232448, "quantiser shared memory");
  static_assert(kStageBytes % 16 == 0 && sizeof(QpUnit) <= 128, "stage layout");
};

// A Q or K unit's codes and scales (K smoothed by the staged mean): the eight lanes of a row
// hold its vectors part + 8 j (8 values each), so that they read 128 consecutive bytes of
// shared memory.  s_am, s_med, s_sc: the grouped scales' shared scratch (kGroups).
template <sl8_dtype DT, int D, bool kGroups>
__device__ __forceinline__ void qp_codes(const QuantQK& a, const QpUnit& x, const uint8_t* sx, uint32_t row_bytes,
                                         int lane, float* s_am, float* s_med, float* s_sc) {
  using C = QpCfg<D>;
  constexpr int LPR = 8, NV = D / 64, RPP = 32 / LPR, P = kQpRows / kQpConsumers / RPP;
  const int warp = threadIdx.x / 32, rsub = lane / LPR, part = lane % LPR;
  const bool smooth = x.kind == kQpK && a.k_partials;
  uint16_t* codes = x.kind == kQpK ? a.k_codes : a.q_codes;
  float* scales = x.kind == kQpK ? a.k_scales : a.q_scales;
  // the lane's values of each pass (widened, smoothed) and the validity of the pass's row
  float v[P][NV][8];
  bool valid[P];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const int r = warp * (kQpRows / kQpConsumers) + p * RPP + rsub;
    const int t = x.t0 + r;
    valid[p] = t < x.L && (x.kind == kQpK || t >= a.q_off);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int c = 8 * (part + 8 * j);
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (valid[p] && c < a.d_io) w = *reinterpret_cast<const uint4*>(sx + r * row_bytes + c * 2);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (DT == SL8_BF16) {
          v[p][j][2 * e] = __uint_as_float(ww[e] << 16);
          v[p][j][2 * e + 1] = __uint_as_float(ww[e] & 0xffff0000u);
        } else {
          v[p][j][2 * e] = f16_bits_to_float(ww[e] & 0xffffu);
          v[p][j][2 * e + 1] = f16_bits_to_float(ww[e] >> 16);
        }
      }
      if (smooth && valid[p] && c < a.d_io) {
        const float4 m0 = *reinterpret_cast<const float4*>(sx + C::kMeanOff + c * 4);
        const float4 m1 = *reinterpret_cast<const float4*>(sx + C::kMeanOff + c * 4 + 16);
        const float mu[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
        for (int e = 0; e < 8; e += 2)
          q_upk2(q_sub2(q_pk2(v[p][j][e], v[p][j][e + 1]), q_pk2(mu[e], mu[e + 1])), v[p][j][e],
                 v[p][j][e + 1]);
      }
    }
  }
  // per-row max |x| over the row's eight lanes
  float am[P];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < NV; ++j)
#pragma unroll
      for (int e = 0; e < 8; e += 2) m = q_max3(m, fabsf(v[p][j][e]), fabsf(v[p][j][e + 1]));
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    am[p] = m;
  }
  float scale[P];
  if constexpr (kGroups) {
    // grouped scales: rows [g0, g0 + G) of the unit share one (see QuantQK); the unit's 64
    // rows are positions t0 .. t0 + 63 and t0 is a multiple of 64, so groups are
    // unit-local.  Rows that take no part hold -1.
#pragma unroll
    for (int p = 0; p < P; ++p)
      if (part == 0) s_am[warp * (kQpRows / kQpConsumers) + p * RPP + rsub] = valid[p] ? am[p] : -1.0f;
    named_bar_sync(1, kQpConsumers * 32);
    const int G = x.kind == kQpK ? a.k_group : a.q_group;
    const float tau = x.kind == kQpK ? 0.0f : a.q_tau;
    // four consecutive threads per row r, each scanning a quarter of r's group
    const int r = threadIdx.x >> 2, jq = threadIdx.x & 3, g0 = r & ~(G - 1);
    const int per = (G + 3) >> 2, c0 = g0 + jq * per, c1 = min(c0 + per, g0 + G);
    const float m = s_am[r];
    if (tau > 0.0f) {
      int n = 0, rank = 0;
      for (int i2 = c0; i2 < c1; ++i2) {
        const float c = s_am[i2];
        const bool in = c >= 0.0f;
        n += in ? 1 : 0;
        rank += (in && (c < m || (c == m && i2 < r))) ? 1 : 0;
      }
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        n += __shfl_xor_sync(0xffffffffu, n, o);
        rank += __shfl_xor_sync(0xffffffffu, rank, o);
      }
      if (jq == 0 && m >= 0.0f && rank == (n - 1) / 2) s_med[g0] = m;
      named_bar_sync(1, kQpConsumers * 32);
    }
    const float thr = tau > 0.0f ? __fmul_rn(tau, s_med[g0]) : INFINITY;
    float top = 0.0f;
    for (int i2 = c0; i2 < c1; ++i2) {
      const float c = s_am[i2];
      if (c >= 0.0f && !(c > thr)) top = fmaxf(top, c);
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) top = fmaxf(top, __shfl_xor_sync(0xffffffffu, top, o));
    if (jq == 0) s_sc[r] = m < 0.0f ? 0.0f : __fdiv_rn(m > thr ? m : top, 127.0f);
    named_bar_sync(1, kQpConsumers * 32);
#pragma unroll
    for (int p = 0; p < P; ++p) scale[p] = s_sc[warp * (kQpRows / kQpConsumers) + p * RPP + rsub];
    // the shared arrays are rewritten by the next unit only after every consumer has
    // passed this unit's last barrier
    named_bar_sync(1, kQpConsumers * 32);
  } else {
#pragma unroll
    for (int p = 0; p < P; ++p) scale[p] = valid[p] ? __fdiv_rn(am[p], 127.0f) : 0.0f;
  }
  // codes: y = x * (1/s) (an approximate reciprocal is close enough: y is within 2e-5 of the
  // correctly rounded quotient), rounded half-even by the 1.5 * 2^23 addition; a value whose
  // y lies within 1e-4 of a half-integer takes the IEEE quotient
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const int r = warp * (kQpRows / kQpConsumers) + p * RPP + rsub;
    const int64_t pr = x.row0 + r;
    const float rs = scale[p] == 0.0f ? 0.0f : (scale[p] >= 1.0e-37f ? rcp_approx(scale[p]) : __frcp_rn(scale[p]));
    const uint64_t rs2 = q_pk2(rs, rs), mg2 = q_pk2(12582912.0f, 12582912.0f);
    uint16_t* crow = codes + (static_cast<int64_t>(x.h) * a.t_pad_max + pr) * D;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      float cf[8];
      float dev = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const uint64_t y2 = q_mul2(q_pk2(v[p][j][e], v[p][j][e + 1]), rs2);
        const uint64_t c2 = q_sub2(q_add2(y2, mg2), mg2);
        float d0, d1;
        q_upk2(q_sub2(y2, c2), d0, d1);
        q_upk2(c2, cf[e], cf[e + 1]);
        dev = q_max3(dev, fabsf(d0), fabsf(d1));
      }
      if (dev > 0.4999f) {
#pragma unroll
        for (int e = 0; e < 8; ++e) cf[e] = quant_code_rcp(v[p][j][e], scale[p], rs);
      }
      // the codes are small integers: their bf16 bits are the float's upper half (one
      // byte permute per pair)
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = __byte_perm(__float_as_uint(cf[2 * e]), __float_as_uint(cf[2 * e + 1]), 0x7632);
      *reinterpret_cast<uint4*>(crow + 8 * (part + 8 * j)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (part == 0) scales[static_cast<int64_t>(x.h) * a.t_pad_max + pr] = scale[p];
  }
}

// A V unit: fp16 V * 2^-e of its rows (zeros past the sequence and past d_io).
template <int D>
__device__ __forceinline__ void qp_convert_v(const QuantQK& a, const QpUnit& x, const uint8_t* sx, uint32_t row_bytes,
                                             int lane) {
  constexpr int LPR = 8, NV = D / 64, RPP = 32 / LPR, P = kQpRows / kQpConsumers / RPP;
  const int warp = threadIdx.x / 32, rsub = lane / LPR, part = lane % LPR;
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const int r = warp * (kQpRows / kQpConsumers) + p * RPP + rsub;
    const bool valid = x.t0 + r < x.L;
    const float vscale = valid ? __int_as_float((127 - x.vexp) << 23) : 0.0f;
    const uint64_t vs2 = q_pk2(vscale, vscale);
    uint16_t* vrow = a.v16 + (static_cast<int64_t>(x.h) * a.t_pad_max + x.row0 + r) * D;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int c = 8 * (part + 8 * j);
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (valid && c < a.d_io) w = *reinterpret_cast<const uint4*>(sx + r * row_bytes + c * 2);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float v0 = a.v_f16 ? f16_bits_to_float(ww[e] & 0xffffu) : bf16_bits_to_float(ww[e] & 0xffffu);
        const float v1 = a.v_f16 ? f16_bits_to_float(ww[e] >> 16) : bf16_bits_to_float(ww[e] >> 16);
        float s0, s1;
        q_upk2(q_mul2(q_pk2(v0, v1), vs2), s0, s1);
        const __half2 h2 = __floats2half2_rn(s0, s1);
        o[e] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(vrow + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

template <sl8_dtype DT, int D, bool kGroups>
__global__ void __launch_bounds__(QpCfg<D>::kThreads, QpCfg<D>::kCtasPerSm)
    quant_qk_pipe_kernel(const QuantQK a, const float* __restrict__ k_mean, const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                         uint32_t ticket, DeviceStatus* st, uint64_t limit_ns) {
  using C = QpCfg<D>;
  extern __shared__ __align__(128) uint8_t qp_smem[];
  __shared__ uint64_t full[C::kStages], empty[C::kStages];
  __shared__ __align__(16) float s_am[kQpRows];
  __shared__ float s_med[kQpRows], s_sc[kQpRows];
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  // without the K/V chunk kernels before it, this kernel is the first to touch the
  // workspace after the previous attention launch read it: every unit waits
  const bool chained = a.k_partials || a.v_partials;
  if (!chained) grid_dependency_wait();
  grid_dependents_launch();
  if (blockIdx.x == 0 && threadIdx.x == 0) a.t.counts[2] = 0;  // the attention kernel's item counter
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kQpConsumers);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const int32_t seq_rows = (a.N + kQTile - 1) / kQTile * kPadRows;
  const int64_t rows_all = a.varlen ? static_cast<int64_t>(a.t.counts[1]) : static_cast<int64_t>(a.nseq) * seq_rows;
  const int64_t rows_used = rows_all < a.t_pad_max ? rows_all : a.t_pad_max;
  const int32_t nblk = static_cast<int32_t>((rows_used + kQpRows - 1) / kQpRows);
  const bool convert_v = a.v16 != nullptr;
  // dense Q blocks: those of each sequence from row q_row0 on (varlen: every block)
  const int32_t nqb = (seq_rows - a.q_row0) / kQpRows;
  const int32_t n_q_units = a.varlen ? a.Hq * nblk : a.Hq * a.nseq * nqb;
  const int32_t n_units = n_q_units + (a.k ? a.Hkv * nblk * (convert_v ? 2 : 1) : 0);  // k null: Q rows only
  const uint32_t row_bytes = static_cast<uint32_t>(a.d_io) * 2;

  if (warp == kQpConsumers) {
    // ------------------------------------------------------------ producer
    bool ok = true, waited = !chained;
    int stg = 0;
    uint32_t phase = 0;
    for (int32_t i = 0;; ++i) {
      if (i >= C::kStages)
        ok = __all_sync(0xffffffffu, mbar_wait(&empty[stg], phase ^ 1u, limit_ns, st, 911));
      if (!ok) break;
      int32_t u = static_cast<int32_t>(blockIdx.x);
      if (i > 0) {
        uint32_t c = 0;
        if (lane == 0) c = atomicAdd(&g_qp_claim[ticket][0], 1u);
        u = static_cast<int32_t>(gridDim.x + __shfl_sync(0xffffffffu, c, 0));
      }
      if (u >= n_units) {
        // no more units: tell the consumers through the stage
        if (lane == 0) {
          reinterpret_cast<QpUnit*>(qp_smem + stg * C::kStageBytes + C::kInfoOff)->kind = kQpDone;
          mbar_arrive(&full[stg]);
        }
        break;
      }
      QpUnit x;
      x.pad = 0;
      int32_t v = u;
      x.kind = kQpQ;
      x.h = -1;
      if (u < n_q_units && !a.varlen) {
        // dense Q block: head, sequence, block from row q_row0 of the sequence
        x.h = v / (a.nseq * nqb);
        const int32_t rem = v - x.h * (a.nseq * nqb), sq = rem / nqb;
        x.row0 = static_cast<int64_t>(sq) * seq_rows + a.q_row0 + static_cast<int64_t>(rem - sq * nqb) * kQpRows;
      }
      if (u >= n_q_units) {
        v = u - n_q_units;
        x.kind = kQpK;
        if (convert_v) {
          x.kind = (v & 1) ? kQpV : kQpK;
          v >>= 1;
        }
      }
      const bool kv = x.kind != kQpQ;
      if (x.h < 0) {  // varlen Q blocks and every K / V block: block v of the head's rows
        x.h = v / nblk;
        x.row0 = static_cast<int64_t>(v - x.h * nblk) * kQpRows;
      }
      int64_t pstart;
      if (!a.varlen) {
        x.s = static_cast<int32_t>(x.row0 / seq_rows);
        pstart = static_cast<int64_t>(x.s) * seq_rows;
        x.L = a.N;
        x.tk = 0;
      } else {
        int lo = 0, hi = a.nseq - 1;  // the last s with pstart[s] <= row0
        while (lo < hi) {
          const int mid = (lo + hi + 1) / 2;
          if (a.t.pstart[mid] <= x.row0) lo = mid; else hi = mid - 1;
        }
        x.s = lo;
        pstart = a.t.pstart[lo];
        x.L = a.t.len[lo];
        x.tk = a.t.tok0[lo];
      }
      x.t0 = static_cast<int32_t>(x.row0 - pstart);
      const bool smooth = x.kind == kQpK && a.k_partials;
      const int64_t srow = static_cast<int64_t>(x.s) * a.Hkv + x.h;
      if (kv && !waited) {
        grid_dependency_wait();  // the K mean and the V exponent of kv_finalize_kernel
        waited = true;
      }
      // the V exponent: from kv_finalize_kernel when the chunk kernels ran (bf16 V), else 0,
      // published here for the attention kernel by the unit holding the sequence's first rows
      x.vexp = 0;
      if (x.kind == kQpV) {
        if (chained) x.vexp = a.v_exp_out[srow];
        else if (x.t0 == 0 && lane == 0) a.v_exp_out[srow] = 0;
      }
      // the unit's rows with input: positions [ta, tb) (a query chunk's before q_off have none)
      int tb = min(x.t0 + kQpRows, x.L);
      if (a.varlen && static_cast<int64_t>(x.tk) + tb > a.total_tokens) {  // a length past the tensors
        if (lane == 0) record_status(st, kStatusBadArg, 901);
        tb = static_cast<int>(a.total_tokens - x.tk > x.t0 ? a.total_tokens - x.tk : x.t0);
        x.L = tb;  // rows past the tensors count as past the sequence
      }
      const int ta = max(x.t0, kv ? 0 : a.q_off);
      const int n = max(0, tb - ta);
      uint8_t* sx = qp_smem + stg * C::kStageBytes;
      const int H = kv ? a.Hkv : a.Hq;
      const void* src = x.kind == kQpV ? a.v : (kv ? a.k : a.q);
      // varlen rows are one tiled copy of the unit's 64 token rows (rows past the sequence
      // are read and ignored; past the tensors they are zero-filled), dense rows one bulk
      // copy of the rows with input
      const uint32_t rows_copied = n > 0 ? static_cast<uint32_t>(a.varlen ? kQpRows : n) : 0u;
      if (lane == 0) {
        *reinterpret_cast<QpUnit*>(sx + C::kInfoOff) = x;
        const uint32_t bytes = rows_copied * row_bytes + (smooth ? static_cast<uint32_t>(a.d_io) * 4u : 0u);
        if (bytes) mbar_arrive_expect_tx(&full[stg], bytes); else mbar_arrive(&full[stg]);
        if (smooth) bulk_load(sx + C::kMeanOff, k_mean + srow * a.d_io, a.d_io * 4, &full[stg]);
      }
      __syncwarp();
      if (n > 0) {
        if (!a.varlen) {
          if (lane == 0) {
            const int64_t e0 = kv ? row_offset(false, x.s, x.h, ta, H, a.N, a.d_io, 0)
                                  : row_offset(false, x.s, x.h, ta - a.q_off, H, a.N - a.q_off, a.d_io, 0);
            bulk_load(sx + (ta - x.t0) * row_bytes, static_cast<const uint16_t*>(src) + e0, n * row_bytes, &full[stg]);
          }
        } else if (lane == 0) {
          const CUtensorMap* map = x.kind == kQpV ? &map_v : (kv ? &map_k : &map_q);
          tma_load_3d(sx, map, &full[stg], 0, x.h, x.tk + x.t0);
        }
      }
      if (++stg == C::kStages) {
        stg = 0;
        phase ^= 1u;
      }
    }
    // this CTA claims no more; the last CTA of the launch resets the ticket's counters
    if (lane == 0) {
      __threadfence();
      if (atomicAdd(&g_qp_claim[ticket][1], 1u) == gridDim.x - 1) {
        atomicExch(&g_qp_claim[ticket][0], 0u);
        atomicExch(&g_qp_claim[ticket][1], 0u);
      }
    }
    return;
  }
  // ------------------------------------------------------------ consumers
  int stg = 0;
  uint32_t phase = 0;
  for (;;) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[stg], phase, limit_ns, st, 912));
    if (!ok) break;
    const uint8_t* sx = qp_smem + stg * C::kStageBytes;
    const QpUnit x = *reinterpret_cast<const QpUnit*>(sx + C::kInfoOff);
    if (x.kind == kQpDone) break;
    if (x.kind == kQpV) {
      qp_convert_v<D>(a, x, sx, row_bytes, lane);
    } else {
      qp_codes<DT, D, kGroups>(a, x, sx, row_bytes, lane, s_am, s_med, s_sc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stg]);
    if (++stg == C::kStages) {
      stg = 0;
      phase ^= 1u;
    }
  }
}

template <sl8_dtype DT, int D, bool kGroups>
static cudaError_t launch_quant_pipe(const QuantQK& a, const float* k_mean, cudaStream_t s) {
  using C = QpCfg<D>;
  auto kern = quant_qk_pipe_kernel<DT, D, kGroups>;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), C::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t units =
      static_cast<int64_t>(a.Hq + (a.k ? a.Hkv * (a.v16 ? 2 : 1) : 0)) * ((a.t_pad_max + kQpRows - 1) / kQpRows);
  const int64_t slots = static_cast<int64_t>(num_sms()) * C::kCtasPerSm;
  const int grid = static_cast<int>(units < slots ? units : slots);
  if (grid <= 0) return cudaSuccess;
  // varlen input: each unit's 64 token rows of one head as a tiled copy of [T][H][d_io]
  CUtensorMap mq, mk, mv;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  if (a.varlen) {
    bool ok = true;
    const uint64_t T = static_cast<uint64_t>(a.total_tokens), dio = static_cast<uint64_t>(a.d_io);
    mq = make_tmap_3d(a.q, CU_TENSOR_MAP_DATA_TYPE_UINT16, dio, a.Hq, T, dio * 2, dio * 2 * a.Hq, a.d_io, 1, kQpRows,
                      &ok, false);
    if (a.k)
      mk = make_tmap_3d(a.k, CU_TENSOR_MAP_DATA_TYPE_UINT16, dio, a.Hkv, T, dio * 2, dio * 2 * a.Hkv, a.d_io, 1,
                        kQpRows, &ok, false);
    if (a.v16)
      mv = make_tmap_3d(a.v, CU_TENSOR_MAP_DATA_TYPE_UINT16, dio, a.Hkv, T, dio * 2, dio * 2 * a.Hkv, a.d_io, 1,
                        kQpRows, &ok, false);
    if (!ok) return cudaErrorInvalidValue;
  }
  static std::atomic<uint32_t> next_ticket{0};
  const uint32_t ticket = next_ticket.fetch_add(1, std::memory_order_relaxed) % kQpTickets;
  return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmem, s, a, k_mean, mq, mk, mv, ticket,
                    device_status_ptr(), spin_limit_ns());
}

template <sl8_dtype DT, bool kGroups>
static cudaError_t launch_quant_pipe_dt(const QuantQK& a, const float* k_mean, int32_t d, cudaStream_t s) {
  switch (d) {
    case 64: return launch_quant_pipe<DT, 64, kGroups>(a, k_mean, s);
    case 128: return launch_quant_pipe<DT, 128, kGroups>(a, k_mean, s);
    default: return launch_quant_pipe<DT, 256, kGroups>(a, k_mean, s);
  }
}

cudaError_t launch_kv_finalize(bool varlen, int32_t nseq, int32_t Hkv, int32_t N, int32_t d_io, const int32_t* len,
                               const float* k_partials, const float* v_partials, int32_t max_chunks, float* mean,
                               int32_t* v_exp, cudaStream_t s) {
  TraceScope tr("kv_finalize", s);
  return launch_pdl(kv_finalize_kernel, dim3(Hkv, nseq), dim3(128), 0, s, varlen, Hkv, N, d_io, len, k_partials,
                    v_partials, max_chunks, mean, v_exp);
}

cudaError_t launch_quant_qk(const void* q, const void* k, sl8_dtype dt, bool varlen, int32_t nseq, int32_t Hq,
                            int32_t Hkv, int32_t N, int32_t d, int64_t total_tokens, const SeqTable& t,
                            int64_t t_pad_max, const float* k_partials, const float* v_partials,
                            int32_t max_chunks, uint16_t* q_codes, float* q_scales, uint16_t* k_codes,
                            float* k_scales, const void* v, int32_t* v_exp, uint16_t* v16, cudaStream_t s,
                            int32_t q_off, int32_t d_io, bool v_f16, const QuantGroups& groups,
                            const float* k_mean) {
  // a chunk's Q blocks start at the first row of the attention's first item
  const int32_t item_rows = prefill_item_rows(d, Hq / Hkv);
  const int32_t q_row0 = varlen ? 0 : q_off / item_rows * item_rows;
  QuantQK a{q, k, varlen, nseq, Hq, Hkv, N, q_off, q_row0, d_io > 0 ? d_io : d, v_f16, total_tokens, t, t_pad_max,
            k_partials,
            v_partials, max_chunks, v_exp,
            q_codes, q_scales, k_codes, k_scales, v, v16, groups.q_group, groups.k_group, groups.q_tau};
  TraceScope tr("quant_qk", s);
  if (groups.q_group > 1 || groups.k_group > 1 || groups.q_tau > 0.0f)
    return dt == SL8_BF16 ? launch_quant_pipe_dt<SL8_BF16, true>(a, k_mean, d, s)
                          : launch_quant_pipe_dt<SL8_F16, true>(a, k_mean, d, s);
  return dt == SL8_BF16 ? launch_quant_pipe_dt<SL8_BF16, false>(a, k_mean, d, s)
                        : launch_quant_pipe_dt<SL8_F16, false>(a, k_mean, d, s);
}

// ---------------------------------------------------------------- codes from an int8 cache
// The V exponent of each (sequence, kv head) of a dense int8 cache: e >= 0 the least with
// max(v_scale) < 2^(e + 8), so that |code * scale| <= 127 * max(v_scale) < 2^15 after the
// 2^-e and fp16 cannot overflow (the exponent the bf16-V path would choose, or one more).
// One CTA per (kv head, sequence).
__global__ void __launch_bounds__(256) cache_vexp_kernel(const float* __restrict__ v_scale, int32_t Hkv, int32_t N,
                                                         int32_t Lmax, int32_t* __restrict__ v_exp) {
  __shared__ float s_max[8];
  grid_dependency_wait();
  grid_dependents_launch();
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const float* vs = v_scale + (static_cast<int64_t>(b) * Hkv + h) * Lmax;
  float m0 = 0.0f, m1 = 0.0f, m2 = 0.0f, m3 = 0.0f;
  int t = tid;
  for (; t + 768 < N; t += 1024) {  // four loads in flight per round
    m0 = fmaxf(m0, vs[t]);
    m1 = fmaxf(m1, vs[t + 256]);
    m2 = fmaxf(m2, vs[t + 512]);
    m3 = fmaxf(m3, vs[t + 768]);
  }
  for (; t < N; t += 256) m0 = fmaxf(m0, vs[t]);
  float m = warp_max(fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)));
  if ((tid & 31) == 0) s_max[tid >> 5] = m;
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < 8; ++w) m = fmaxf(m, s_max[w]);
    int e = 0;
    if (m > 0.0f) {
      int km = 0;
      frexpf(m, &km);  // m < 2^km
      e = km > 8 ? km - 8 : 0;
    }
    v_exp[static_cast<int64_t>(b) * Hkv + h] = e;
  }
}

// K and V rows of the cache into the code workspace: one CTA per (64-row block of a
// sequence's padded rows, kv head, sequence); each thread turns 16 codes of a row of K
// and of V at a time.  Launched as a programmatic dependent of cache_vexp_kernel, whose
// exponent it reads.
__global__ void __launch_bounds__(256) cache_codes_kernel(const int8_t* __restrict__ k_cache,
                                                          const float* __restrict__ k_scale,
                                                          const int8_t* __restrict__ v_cache,
                                                          const float* __restrict__ v_scale, int32_t Hkv, int32_t N,
                                                          int32_t Lmax, int32_t d, int32_t d_io, int32_t seq_rows,
                                                          int64_t t_pad_max, uint16_t* __restrict__ k_codes,
                                                          float* __restrict__ k_scales, uint16_t* __restrict__ v16,
                                                          const int32_t* __restrict__ v_exp) {
  const int h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int64_t src_row0 = (static_cast<int64_t>(b) * Hkv + h) * Lmax;  // token 0 of (b, h) in the cache
  const int vec = d / 16;                                               // 16-code vectors per code row
  const int t0 = blockIdx.x * 64;
  grid_dependency_wait();
  grid_dependents_launch();
  const int e = v_exp[static_cast<int64_t>(b) * Hkv + h];
  const float vmul = __int_as_float((127 - e) << 23);  // 2^-e
  for (int i = tid; i < 64 * vec; i += blockDim.x) {
    const int r = i / vec, c = (i - r * vec) * 16, t = t0 + r;
    const int64_t dst = static_cast<int64_t>(h) * t_pad_max + static_cast<int64_t>(b) * seq_rows + t;
    const bool valid = t < N && c < d_io;
    uint4 kw = make_uint4(0u, 0u, 0u, 0u), vw = kw;
    float vs = 0.0f;
    if (valid) {
      kw = *reinterpret_cast<const uint4*>(k_cache + (src_row0 + t) * d_io + c);
      vw = *reinterpret_cast<const uint4*>(v_cache + (src_row0 + t) * d_io + c);
      vs = __fmul_rn(v_scale[src_row0 + t], vmul);
    }
    const uint32_t kb[4] = {kw.x, kw.y, kw.z, kw.w}, vb[4] = {vw.x, vw.y, vw.z, vw.w};
    uint32_t ko[8], vo[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      // codes 2j and 2j+1 of the vector, sign-extended from their bytes
      const int c0 = static_cast<int8_t>((kb[j >> 1] >> (16 * (j & 1))) & 0xffu);
      const int c1 = static_cast<int8_t>((kb[j >> 1] >> (16 * (j & 1) + 8)) & 0xffu);
      ko[j] = (__float_as_uint(static_cast<float>(c0)) >> 16) | (__float_as_uint(static_cast<float>(c1)) & 0xffff0000u);
      const int v0 = static_cast<int8_t>((vb[j >> 1] >> (16 * (j & 1))) & 0xffu);
      const int v1 = static_cast<int8_t>((vb[j >> 1] >> (16 * (j & 1) + 8)) & 0xffu);
      const __half2 h2 = __floats2half2_rn(__fmul_rn(static_cast<float>(v0), vs), __fmul_rn(static_cast<float>(v1), vs));
      vo[j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    uint4* kd = reinterpret_cast<uint4*>(k_codes + dst * d + c);
    uint4* vd = reinterpret_cast<uint4*>(v16 + dst * d + c);
    kd[0] = make_uint4(ko[0], ko[1], ko[2], ko[3]);
    kd[1] = make_uint4(ko[4], ko[5], ko[6], ko[7]);
    vd[0] = make_uint4(vo[0], vo[1], vo[2], vo[3]);
    vd[1] = make_uint4(vo[4], vo[5], vo[6], vo[7]);
    if (c == 0) k_scales[static_cast<int64_t>(h) * t_pad_max + static_cast<int64_t>(b) * seq_rows + t] =
        t < N ? k_scale[src_row0 + t] : 0.0f;
  }
}

cudaError_t launch_cache_codes(const int8_t* k_cache, const float* k_scale, const int8_t* v_cache,
                               const float* v_scale, int32_t nseq, int32_t Hkv, int32_t N, int32_t Lmax, int32_t d,
                               int32_t d_io, int64_t t_pad_max, uint16_t* k_codes, float* k_scales, uint16_t* v16,
                               int32_t* v_exp, cudaStream_t s) {
  TraceScope tr("cache_codes", s);
  const int32_t seq_rows = (N + kQTile - 1) / kQTile * kPadRows;
  cudaError_t e = launch_pdl(cache_vexp_kernel, dim3(Hkv, nseq), dim3(256), 0, s, v_scale, Hkv, N, Lmax, v_exp);
  if (e != cudaSuccess) return e;
  return launch_pdl(cache_codes_kernel, dim3(seq_rows / 64, Hkv, nseq), dim3(256), 0, s, k_cache, k_scale, v_cache,
                    v_scale, Hkv, N, Lmax, d, d_io, seq_rows, t_pad_max, k_codes, k_scales, v16,
                    static_cast<const int32_t*>(v_exp));
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
  const float rs = s == 0.0f ? 0.0f : __frcp_rn(s);
  int8_t* q = q_out + row * cols;
  for (int c = lane; c < cols; c += 32) {
    float v = load_elem<DT>(x, base + c);
    if (mu) v = __fsub_rn(v, mu[c]);
    q[c] = s == 0.0f ? 0 : static_cast<int8_t>(static_cast<int>(quant_code_rcp(v, s, rs)));
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
                                    int32_t nseq, int32_t H, int32_t N, int32_t d, int32_t d_io, SeqTable t,
                                    int64_t t_pad_max, int8_t* __restrict__ codes_out,
                                    float* __restrict__ scales_out) {
  const int s = blockIdx.y, h = blockIdx.z;
  const int32_t L = t.len[s];
  const int32_t tok = blockIdx.x;
  if (tok >= L) return;
  const int64_t src = static_cast<int64_t>(h) * t_pad_max + t.pstart[s] + tok;
  const int64_t dst_row = varlen ? (static_cast<int64_t>(t.tok0[s]) + tok) * H + h
                                 : (static_cast<int64_t>(s) * H + h) * N + tok;
  for (int c = threadIdx.x; c < d_io; c += blockDim.x) {
    const float v = __bfloat162float(__ushort_as_bfloat16(codes[src * d + c]));
    codes_out[dst_row * d_io + c] = static_cast<int8_t>(__float2int_rn(v));
  }
  if (threadIdx.x == 0) scales_out[dst_row] = scales[src];
}

cudaError_t launch_export_codes(const uint16_t* codes, const float* scales, bool varlen, int32_t nseq, int32_t H,
                                int32_t N, int32_t d, const SeqTable& t, int64_t t_pad_max, int8_t* codes_out,
                                float* scales_out, cudaStream_t s, int32_t d_io) {
  TraceScope tr("export_codes", s);
  export_codes_kernel<<<dim3(N, nseq, H), 64, 0, s>>>(codes, scales, varlen, nseq, H, N, d, d_io > 0 ? d_io : d, t,
                                                       t_pad_max, codes_out, scales_out);
  return cudaGetLastError();
}

}  // namespace sl8
