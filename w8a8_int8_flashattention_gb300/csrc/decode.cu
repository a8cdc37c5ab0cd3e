// Split-KV decode over an int8 KV cache, and its combine step, for sm_103a.
//
// Operation: the "SuperL8" README (github.com/jajmangold/superl8), "Attention
// kernels" table, attn_decode row (split-KV decode with an int8 KV cache; the int8-V
// variant).  Reading taken: q [B, Hq, d] is quantised per (b, hq) row like prefill
// (s = max|x| / 127, round-half-even, clamp to +-127); the cache holds int8 codes
// [B, Hkv, Lmax, d] with one fp32 scale per (b, hkv, token) for K and for V; for
// query head hq (kv head hq / (Hq / Hkv)) and tokens t < L_b:
//   x_t = int32(q_i8 . k_i8[t]) * s_q * s_k[t] / sqrt(d),  p = softmax(x),
//   O = sum_t p_t * s_v[t] * v_i8[t].
// The key range is cut into contiguous splits of split_size tokens.  Each split
// writes its normalised partial O and its log-sum-exp (natural log; -inf for an
// empty split); the combine kernel merges the partials of a row with weights
// exp(lse_s - max lse).
//
// GB300 design: HBM streaming is the bound.  One CTA per (split, kv head, batch):
// the split's K and V codes are contiguous in the cache, so each is fetched with
// one bulk async copy (TMA, cp.async.bulk) into shared memory; the G query rows
// of the kv group are quantised in the CTA and the int32 dots run on dp4a with
// 8 threads (16 bytes each) per key row, conflict-free shared-memory reads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sl8_internal.h"

namespace sl8 {

namespace {

constexpr int kThreads = 256;

template <int D>
struct DCfg {
  static constexpr int kChunk = 32768 / D;  // tokens per sub-chunk (32 KB of K codes)
  static constexpr int kTPR = D / 16;       // threads per key row (16 codes each)
  static constexpr int kRowsPerPass = kThreads / kTPR;
};

template <int D, int GT>
struct DSmem {
  static constexpr int kK = 0;
  static constexpr int kV = kK + DCfg<D>::kChunk * D;
  static constexpr int kKs = kV + DCfg<D>::kChunk * D;
  static constexpr int kVs = kKs + DCfg<D>::kChunk * 4;
  static constexpr int kScore = kVs + DCfg<D>::kChunk * 4;          // [GT][chunk] floats
  static constexpr int kQ = kScore + GT * DCfg<D>::kChunk * 4;      // [GT][D] int8
  static constexpr int kQs = kQ + GT * D;                           // [GT] floats
  static constexpr int kRowStat = kQs + GT * 4 + 16;                // [GT][2] floats (m, l of the sub-chunk)
  // [8 warps][GT][D] floats for the final P.V reduction: reuses the K chunk once it
  // is consumed when it fits there
  static constexpr bool kRedInK = 8 * GT * D * 4 <= DCfg<D>::kChunk * D;
  static constexpr int kTail = (kRowStat + GT * 8 + 127) / 128 * 128;
  static constexpr int kRed = kRedInK ? kK : kTail;
  static constexpr int kBar = kRedInK ? kTail : kTail + 8 * GT * D * 4;
  static constexpr int kBytes = kBar + 64 + 128;
};

__device__ __forceinline__ float bf16_bits(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ float f16_bits(uint32_t b) { return __half2float(__ushort_as_half(static_cast<unsigned short>(b))); }

__device__ __forceinline__ float warp_max_f(float a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  return a;
}
__device__ __forceinline__ float warp_sum_f(float a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
  return a;
}

// int8 byte k of w (sign-extended) as float
__device__ __forceinline__ float i8_to_f(uint32_t w, int k) {
  return static_cast<float>(static_cast<int8_t>((w >> (8 * k)) & 0xFFu));
}

// An empty split: lse = -inf and a zero partial O for the G rows of the group.
__device__ __forceinline__ void write_empty_split(const DecodeArgs& a, int64_t part_row0, int split, int G, int D) {
  for (int i = threadIdx.x; i < G * D; i += kThreads) {
    const int g = i / D, c = i % D;
    a.o_partial[((part_row0 + g) * a.num_splits + split) * D + c] = 0.0f;
  }
  if (threadIdx.x < G) a.lse_partial[(part_row0 + threadIdx.x) * a.num_splits + split] = -INFINITY;
}

template <int D, int GT>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const DecodeArgs a, DeviceStatus* st, uint64_t limit_ns) {
  using C = DCfg<D>;
  using S = DSmem<D, GT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  int8_t* sk = reinterpret_cast<int8_t*>(smem + S::kK);
  int8_t* sv = reinterpret_cast<int8_t*>(smem + S::kV);
  float* sks = reinterpret_cast<float*>(smem + S::kKs);
  float* svs = reinterpret_cast<float*>(smem + S::kVs);
  float* score = reinterpret_cast<float*>(smem + S::kScore);
  int8_t* sq = reinterpret_cast<int8_t*>(smem + S::kQ);
  float* sqs = reinterpret_cast<float*>(smem + S::kQs);
  float* red = reinterpret_cast<float*>(smem + S::kRed);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + S::kBar);

  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int G = a.Hq / a.Hkv;
  int L = a.seqlens[b];
  if (L < 0 || L > a.Lmax) {
    if (tid == 0) record_status(st, kStatusBadArg, 700);
    L = L < 0 ? 0 : a.Lmax;
  }
  const int t_begin = split * a.split_size;
  const int t_end = min(t_begin + a.split_size, L);
  const int64_t part_row0 = (static_cast<int64_t>(b) * a.Hq + hkv * G);  // first (b, hq) row of this group
  const bool empty = t_begin >= t_end;
  if (empty && !(split == 0 && a.q_codes)) {
    write_empty_split(a, part_row0, split, G, D);
    return;
  }

  // ---- quantise the G query rows of this kv group (warp per row)
  for (int g = warp; g < GT; g += kThreads / 32) {
    float v[D / 32];
    const int64_t qrow = (static_cast<int64_t>(b) * a.Hq + hkv * G + g) * D;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      const int c = lane * (D / 32) + e;
      float x = 0.0f;
      if (g < G) {
        if (a.q_dtype == SL8_BF16) x = bf16_bits(static_cast<const uint16_t*>(a.q)[qrow + c]);
        else if (a.q_dtype == SL8_F16) x = f16_bits(static_cast<const uint16_t*>(a.q)[qrow + c]);
        else x = static_cast<const float*>(a.q)[qrow + c];
      }
      v[e] = x;
    }
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
    amax = warp_max_f(amax);
    const float s = __fdiv_rn(amax, 127.0f);
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      int code = 0;
      if (s != 0.0f) {
        code = __float2int_rn(__fdiv_rn(v[e], s));
        code = code > 127 ? 127 : (code < -127 ? -127 : code);
      }
      sq[g * D + lane * (D / 32) + e] = static_cast<int8_t>(code);
      if (split == 0 && g < G && a.q_codes) a.q_codes[qrow + lane * (D / 32) + e] = static_cast<int8_t>(code);
    }
    if (lane == 0) {
      sqs[g] = s;
      if (split == 0 && g < G && a.q_scales) a.q_scales[qrow / D] = s;
    }
  }
  if (empty) {  // split 0 of an empty sequence: only the q codes were asked for
    write_empty_split(a, part_row0, split, G, D);
    return;
  }

  // thread roles for the dot products and P.V: 8 threads (for d = 128) per key row
  const int sub = tid % C::kTPR;           // 16-byte column slice of the row
  const int rsub = tid / C::kTPR;          // row within a pass
  const float log2e_over_sqrtd = 1.4426950408889634f / sqrtf(static_cast<float>(D));

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncthreads();

  // running statistics over the sub-chunks of this split (per q row g; every thread
  // keeps the copy for all g, identical across threads)
  float run_m[GT], run_l[GT];
  float acc[GT][16];
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    run_m[g] = -INFINITY;
    run_l[g] = 0.0f;
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[g][c] = 0.0f;
  }
  // this thread's 16 q codes per row, as 4 words
  uint32_t qw[GT][4];
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    const uint4 w = *reinterpret_cast<const uint4*>(sq + g * D + sub * 16);
    qw[g][0] = w.x; qw[g][1] = w.y; qw[g][2] = w.z; qw[g][3] = w.w;
  }
  float qsc[GT];
#pragma unroll
  for (int g = 0; g < GT; ++g) qsc[g] = sqs[g] * log2e_over_sqrtd;

  const int64_t cache_row0 = (static_cast<int64_t>(b) * a.Hkv + hkv) * a.Lmax;
  uint32_t phase = 0;
  bool ok = true;
  for (int c0 = t_begin; c0 < t_end; c0 += C::kChunk) {
    const int n = min(C::kChunk, t_end - c0);
    if (tid == 0) {
      const uint32_t bytes = static_cast<uint32_t>(n) * D;
      mbar_arrive_expect_tx(bar, 2 * bytes);
      bulk_load(sk, a.k_cache + (cache_row0 + c0) * D, bytes, bar);
      bulk_load(sv, a.v_cache + (cache_row0 + c0) * D, bytes, bar);
    }
    for (int i = tid; i < n; i += kThreads) {
      sks[i] = a.k_scale[cache_row0 + c0 + i];
      svs[i] = a.v_scale[cache_row0 + c0 + i];
    }
    ok = mbar_wait(bar, phase, limit_ns, st, 40);
    phase ^= 1;
    if (!__syncthreads_and(ok)) break;  // also publishes the scales

    // ---- scores: x2[g][t] = S * s_q * s_k[t] * log2(e) / sqrt(d)
    for (int r0 = 0; r0 < n; r0 += C::kRowsPerPass) {
      const int t = r0 + rsub;
      uint4 kw = make_uint4(0, 0, 0, 0);
      if (t < n) kw = *reinterpret_cast<const uint4*>(sk + t * D + sub * 16);
      int dot[GT];
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        int s = 0;
        s = __dp4a(static_cast<int>(kw.x), static_cast<int>(qw[g][0]), s);
        s = __dp4a(static_cast<int>(kw.y), static_cast<int>(qw[g][1]), s);
        s = __dp4a(static_cast<int>(kw.z), static_cast<int>(qw[g][2]), s);
        s = __dp4a(static_cast<int>(kw.w), static_cast<int>(qw[g][3]), s);
#pragma unroll
        for (int o = 1; o < C::kTPR; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        dot[g] = s;
      }
      if (sub == 0 && t < n) {
        const float kscale = sks[t];
#pragma unroll
        for (int g = 0; g < GT; ++g) {
          if (a.logits && g < G)
            a.logits[(part_row0 + g) * a.Lmax + c0 + t] = dot[g];
          score[g * C::kChunk + t] = static_cast<float>(dot[g]) * kscale * qsc[g];
        }
      }
    }
    __syncthreads();

    // ---- sub-chunk softmax statistics (warp per row g), weights w = p * s_v
    float* rowstat = reinterpret_cast<float*>(smem + S::kRowStat);
    for (int g = warp; g < GT; g += kThreads / 32) {
      float mx = -INFINITY;
      for (int t = lane; t < n; t += 32) mx = fmaxf(mx, score[g * C::kChunk + t]);
      mx = warp_max_f(mx);
      const float m_new = fmaxf(run_m[g], mx);
      float sum = 0.0f;
      for (int t = lane; t < n; t += 32) {
        const float p = exp2f(score[g * C::kChunk + t] - m_new);
        sum += p;
        score[g * C::kChunk + t] = p * svs[t];
      }
      sum = warp_sum_f(sum);
      if (lane == 0) {
        rowstat[2 * g] = m_new;
        rowstat[2 * g + 1] = sum;
      }
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      const float m_new = rowstat[2 * g];
      const float corr = run_m[g] == -INFINITY ? 0.0f : exp2f(run_m[g] - m_new);
      run_l[g] = run_l[g] * corr + rowstat[2 * g + 1];
      run_m[g] = m_new;
#pragma unroll
      for (int c = 0; c < 16; ++c) acc[g][c] *= corr;
    }

    // ---- P.V: each thread accumulates its 16 channels over rows t = rsub (mod rows per pass)
    for (int t = rsub; t < n; t += C::kRowsPerPass) {
      const uint4 vw = *reinterpret_cast<const uint4*>(sv + t * D + sub * 16);
      float vf[16];
      const uint32_t wds[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int k = 0; k < 4; ++k) vf[q * 4 + k] = i8_to_f(wds[q], k);
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        const float wt = score[g * C::kChunk + t];
#pragma unroll
        for (int c = 0; c < 16; ++c) acc[g][c] = fmaf(wt, vf[c], acc[g][c]);
      }
    }
    __syncthreads();  // score / sk / sv are rewritten by the next sub-chunk
  }

  if (!ok) return;
  // ---- reduce acc over the row slots: within a warp (lanes with equal sub), then across warps
#pragma unroll
  for (int g = 0; g < GT; ++g)
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float v = acc[g][c];
#pragma unroll
      for (int o = C::kTPR; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc[g][c] = v;
    }
  if (lane < C::kTPR) {
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
      for (int c = 0; c < 16; ++c) red[(warp * GT + g) * D + sub * 16 + c] = acc[g][c];
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += kThreads) {
    const int g = i / D, c = i % D;
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) v += red[(w * GT + g) * D + c];
    a.o_partial[((part_row0 + g) * a.num_splits + split) * D + c] = v / run_l[g];
  }
  if (tid < G) {
    a.lse_partial[(part_row0 + tid) * a.num_splits + split] = (run_m[tid] + log2f(run_l[tid])) * 0.6931471805599453f;
  }
}

// One warp per (b, hq): merge the non-empty splits of the row.
template <int D>
__global__ void decode_combine_kernel(const float* __restrict__ o_partial, const float* __restrict__ lse_partial,
                                      const int32_t* __restrict__ seqlens, int32_t B, int32_t Hq, int32_t num_splits,
                                      int32_t split_size, void* out, sl8_dtype out_dtype, float* lse_out) {
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= B * Hq) return;
  const int b = row / Hq;
  const int L = max(0, seqlens[b]);
  const int ns = min(num_splits, (L + split_size - 1) / split_size);
  const float* lse = lse_partial + static_cast<int64_t>(row) * num_splits;
  float m = -INFINITY;
  for (int s = lane; s < ns; s += 32) m = fmaxf(m, lse[s]);
  m = warp_max_f(m);
  constexpr int E = D / 32;
  float o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.0f;
  float wsum = 0.0f;
  if (m != -INFINITY) {
    for (int s = 0; s < ns; ++s) {
      const float ls = lse[s];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - m);
      wsum += w;
      const float* op = o_partial + (static_cast<int64_t>(row) * num_splits + s) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = fmaf(w, op[e], o[e]);
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float v = o[e] * inv;
    const int64_t idx = static_cast<int64_t>(row) * D + lane * E + e;
    if (out_dtype == SL8_F32) static_cast<float*>(out)[idx] = v;
    else if (out_dtype == SL8_BF16) static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else static_cast<__half*>(out)[idx] = __float2half_rn(v);
  }
  if (lse_out && lane == 0) lse_out[row] = m == -INFINITY ? -INFINITY : m + logf(wsum);
}

__global__ void timeout_selftest_kernel(uint64_t limit_ns, DeviceStatus* st) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // nothing ever arrives on this barrier: the bounded wait must give up and record it
  if (threadIdx.x == 0) mbar_wait(&bar, 0, limit_ns, st, 999);
}

template <int D, int GT>
cudaError_t launch_split_dg(const DecodeArgs& a, cudaStream_t s) {
  using S = DSmem<D, GT>;
  auto kern = decode_split_kernel<D, GT>;
  const int smem = S::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_splits, a.Hkv, a.B);
  kern<<<grid, kThreads, smem, s>>>(a, device_status_ptr(), spin_limit_ns());
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_split_d(const DecodeArgs& a, cudaStream_t s) {
  const int G = a.Hq / a.Hkv;
  if (G <= 1) return launch_split_dg<D, 1>(a, s);
  if (G <= 2) return launch_split_dg<D, 2>(a, s);
  if (G <= 4) return launch_split_dg<D, 4>(a, s);
  return launch_split_dg<D, 8>(a, s);
}

}  // namespace

int decode_chunk_tokens(int d) { return 32768 / d; }  // DCfg<d>::kChunk

cudaError_t launch_decode_split(const DecodeArgs& a, cudaStream_t s) {
  TraceScope tr("decode_split", s);
  switch (a.d) {
    case 64: return launch_split_d<64>(a, s);
    case 128: return launch_split_d<128>(a, s);
    case 256: return launch_split_d<256>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_combine(const float* o_partial, const float* lse_partial, const int32_t* seqlens, int32_t B,
                                  int32_t Hq, int32_t d, int32_t num_splits, int32_t split_size, void* out,
                                  sl8_dtype out_dtype, float* lse_out, cudaStream_t s) {
  TraceScope tr("decode_combine", s);
  const int rows = B * Hq;
  const int grid = (rows + 7) / 8;
  switch (d) {
    case 64: decode_combine_kernel<64><<<grid, 256, 0, s>>>(o_partial, lse_partial, seqlens, B, Hq, num_splits, split_size, out, out_dtype, lse_out); break;
    case 128: decode_combine_kernel<128><<<grid, 256, 0, s>>>(o_partial, lse_partial, seqlens, B, Hq, num_splits, split_size, out, out_dtype, lse_out); break;
    case 256: decode_combine_kernel<256><<<grid, 256, 0, s>>>(o_partial, lse_partial, seqlens, B, Hq, num_splits, split_size, out, out_dtype, lse_out); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_timeout_selftest(uint64_t limit_ns, cudaStream_t s) {
  timeout_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, device_status_ptr());
  return cudaGetLastError();
}

}  // namespace sl8
