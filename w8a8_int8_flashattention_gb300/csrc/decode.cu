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
// empty split, whose O is left unwritten); the combine kernel merges the partials
// of a row with weights exp(lse_s - max lse).
//
// GB300 design.  The kernel streams the cache once, so HBM is the bound; the work
// per byte must stay small enough that the compute warps of an SM keep up with it.
//  * A persistent CTA per SM walks a balanced list of (b, kv head, split) work slots
//    (full splits first, then the tails longest first), claiming each next slot from
//    a per-launch counter.  Warp 0 loads each split's K and V codes with tiled TMA
//    copies (128-byte swizzle for d >= 128) in stages of 16 tokens per compute warp,
//    with their scales and the group's raw q rows, into shared-memory rings that run
//    ahead across splits.
//  * Each compute warp (ten for d <= 128, eight for d = 256) takes 16 tokens of every
//    stage and keeps its own online-softmax state; compute warp r < G also quantises
//    q row r of each split as its raw rows land.  Warp 1 merges the warps' states of
//    the previous split into the split's partial O and LSE, so the compute warps never
//    meet at a CTA barrier.
//  * Both contractions run on the tensor cores as m16n8k16 fp16 MMAs with fp32
//    accumulation (the int8 tensor rate of this part is low).  Codes become fp16
//    exactly (|c| <= 127), so q.k is the exact integer dot (|sum| < 2^24).
//      S^T[16 tokens x 8 q] = K[16 x d] . Q^T    (the G <= 8 query rows of the group)
//      O^T[d x 8 q]        += V^T[d x 16] . P'^T  (P' = p * s_v * 2^-E, fp16)
//    Putting tokens and head dims on the M side keeps the padded query columns
//    cheap and gives every lane the same two query columns in S^T and O^T, so the
//    rescales of the online softmax stay inside the lane.
//  * Rescaling is lazy: the running max moves only when a tile exceeds it by more
//    than 2^8 (p then stays below 256), and the power-of-two V range E only when a
//    token's V scale exceeds 2^E; both keep P' inside the fp16 range.
#include <cuda_bf16.h>
#include <atomic>
#include <type_traits>
#include <cuda_fp16.h>

#include "sl8_internal.h"

namespace sl8 {

namespace {

constexpr int kFirstCompute = 2;                // warp 0: loads, warp 1: merges
constexpr int kUnit = 16;                       // tokens per compute warp per stage
constexpr int kQSlots = 2;                      // q-row buffers (one per split in flight)
constexpr float kLazy = 8.0f;                   // log2 headroom of the lazy max

constexpr int kSchedMaxB = 512;
struct Slot {
  int split, b, hkv, t0, t1;  // b < 0: no more slots
};
constexpr int kSlotRing = 8;   // slots announced by the loader ahead of the compute warps
struct Sched {
  int32_t len[kSchedMaxB];       // sequence lengths clamped to [0, Lmax]
  int32_t pf[kSchedMaxB + 1];    // prefix over b of the full slots (full splits x Hkv)
  uint32_t key[kSchedMaxB];      // sorted: (split_size - tail) << 16 | b, then 0xffffffff
  int32_t n_full, n_tail;        // slots of each kind
  Slot ring[kSlotRing];          // slot n of this CTA in ring[n % kSlotRing]
  Slot merge;                    // the slot whose warp states wait in the merge buffer
};
// Dynamic claims: CTA c takes slot c first, then the next unclaimed slot from a
// per-launch counter.  A launch uses counter pair g_claim[ticket] ([0] next slot - grid,
// [1] CTAs done); the last CTA to finish zeroes the pair for the next launch that draws
// the same ticket (tickets rotate over kTickets launches, so up to kTickets launches may
// run at the same time).
constexpr int kTickets = 64;
__device__ uint32_t g_claim[kTickets][2];
static_assert(kSchedMaxB <= 65536, "b fits the key");

template <int D, bool kV16 = false>
struct DCfg {
  // ten compute warps (eight for d = 256, whose tiles and merge buffer are twice as
  // large); registers are granted to the CTA in steps of four warps, so the loader and
  // merging warps come free with them
  static constexpr int kNW = D == 256 ? 8 : 10;
  static constexpr int kCT = kNW * 32;
  static constexpr int kThreads = kCT + 32 * kFirstCompute;
  static constexpr int kChunk = kNW * kUnit;     // tokens per stage
  static constexpr int kBW = D < 128 ? D : 128;  // bytes in one row of a TMA box
  static constexpr int kBoxes = D / kBW;
  static constexpr bool kSwz = D >= 128;         // 128-byte swizzled tiles
  static constexpr int kTile = kChunk * D;       // one stage of K codes
  // V: int8 codes like K, or (kV16) fp16 values in 128-byte rows of 64 dims
  static constexpr int kTileV = kV16 ? 2 * kTile : kTile;
  static constexpr int kBoxesV = kV16 ? D / 64 : kBoxes;
  static constexpr int kStages = kV16 ? (D == 64 ? 4 : 2) : (D <= 64 ? 8 : (D == 128 ? 3 : 2));
  static constexpr int kSK = 0;
  static constexpr int kSV = kTile;
  static constexpr int kSKs = kTile + kTileV;
  static constexpr int kSVs = kSKs + kChunk * 4;
  static constexpr int kStageBytes = (kSVs + kChunk * 4 + 1023) / 1024 * 1024;
  static constexpr int kQBytes = 8 * D * 4;                    // 8 raw q rows, fp32 at most
  static constexpr int kQ = kStages * kStageBytes;             // [2] raw q rows
  static constexpr int kRed = kQ + kQSlots * kQBytes;          // [warp][d][8 q] floats
  static constexpr int kStat = kRed + kNW * D * 8 * 4;         // [warp][8 q][4] floats
  static constexpr int kQcBytes = 8 * D + 64;                  // 8 code rows, 8 scales, 8 code sums
  static constexpr int kQc = kStat + kNW * 8 * 16;             // [2] quantised q rows
  static constexpr int kSched = kQc + kQSlots * kQcBytes;      // Sched
  static constexpr int kBar = (kSched + static_cast<int>(sizeof(Sched)) + 15) / 16 * 16;
  static constexpr int kNumBars = 2 * kStages + 4 * kQSlots + 3;
  static constexpr int kBytes = kBar + kNumBars * 8 + 1024;    // + alignment slack
  static_assert(kStageBytes % 1024 == 0 && kTile % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(!kV16 || (D >= 64 && D <= 128), "fp16 V: 64 <= d <= 128");
  static_assert(kBytes <= 232448, "smem budget");
};

// Byte offset of (row r, 16-byte chunk c of the row) in a stage tile made of kBoxes
// boxes of kChunk rows x kBW bytes, with the 128-byte swizzle when it applies.
template <int D>
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  using C = DCfg<D>;
  constexpr int cpb = C::kBW / 16;
  const int b = c / cpb, cc = c % cpb;
  return static_cast<uint32_t>(b * (C::kChunk * C::kBW) + r * C::kBW + 16 * (C::kSwz ? (cc ^ (r & 7)) : cc));
}

__device__ __forceinline__ float bf16_bits(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ float f16_bits(uint32_t b) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
}
__device__ __forceinline__ float warp_max_f(float a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  return a;
}
// max / sum over the 8 lanes of one thread-in-group column (lanes t, t+4, ..., t+28)
__device__ __forceinline__ float col_max(float a) {
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
  return fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
}
__device__ __forceinline__ float col_sum(float a) {
  a += __shfl_xor_sync(0xffffffffu, a, 4);
  a += __shfl_xor_sync(0xffffffffu, a, 8);
  return a + __shfl_xor_sync(0xffffffffu, a, 16);
}
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns, DeviceStatus* st,
                                          int site) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, limit_ns, st, site));
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 2^n as a float for -126 <= n <= 127, 0 below.
__device__ __forceinline__ float pow2i(int n) {
  return n < -126 ? 0.0f : __uint_as_float(static_cast<uint32_t>(n + 127) << 23);
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// Two int8 codes, already offset by 128 (byte ^ 0x80), picked from ub by sel (0x4140:
// bytes 0 and 1; 0x4342: bytes 2 and 3) and widened exactly to an fp16 pair: each byte
// u becomes the mantissa of 1024 + u, and subtracting 1152 leaves u - 128.
__device__ __forceinline__ uint32_t codes_f16x2(uint32_t ub, uint32_t sel) {
  const uint32_t h = prmt(ub, 0x64646464u, sel);
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
  return r;
}
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Four transposed 8x8 fp16 matrices from shared memory: lanes 8i .. 8i+7 give the row
// addresses of matrix i; register i of thread T holds its rows 2 (T % 4) and 2 (T % 4) + 1
// in column T / 4.
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// Transpose of an 8x8 fp16 matrix held one register per lane (lane l: row l / 4,
// columns 2 (l % 4) and 2 (l % 4) + 1), into the same layout.
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Quantise one q row of D values (f16/bf16/f32) held by a warp, D / 32 per lane.
template <int D>
__device__ __forceinline__ float quant_row_warp(const float (&v)[D / 32], int8_t (&code)[D / 32]) {
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < D / 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
  amax = warp_max_f(amax);
  const float sc = __fdiv_rn(amax, 127.0f);
#pragma unroll
  for (int e = 0; e < D / 32; ++e) {
    int c = 0;
    if (sc != 0.0f) {
      c = __float2int_rn(__fdiv_rn(v[e], sc));
      c = c > 127 ? 127 : (c < -127 ? -127 : c);
    }
    code[e] = static_cast<int8_t>(c);
  }
  return sc;
}

__device__ __forceinline__ float load_q_elem(const void* base, sl8_dtype dt, int64_t idx) {
  return dt == SL8_BF16 ? bf16_bits(static_cast<const uint16_t*>(base)[idx])
       : dt == SL8_F16 ? f16_bits(static_cast<const uint16_t*>(base)[idx])
                       : static_cast<const float*>(base)[idx];
}

// ---- work schedule
// A work slot is one (b, kv head, split).  With B <= kSchedMaxB the launch's slot list
// is: the full splits (split_size tokens), then the sequences' partial last splits,
// longest first; empty splits are handled up front and never listed.  Above
// kSchedMaxB the list is every slot in split-major order (empty ones are skipped).

// The cache sequence of (virtual) sequence b: b itself, or b / verify_ng when verifying.
__device__ __forceinline__ int cache_seq(const DecodeArgs& a, int b) { return a.verify_T ? b / a.verify_ng : b; }

// Query column c (< 8) of a slot of sequence v, kv head hkv: its (b, hq) row of the
// partials and whether it holds a query (the G heads, or verify_dps drafts x G heads;
// drafts past verify_T are dead columns).
template <bool kVerify>
__device__ __forceinline__ int64_t col_row(const DecodeArgs& a, int v, int hkv, int c, int G, bool& live) {
  if constexpr (!kVerify) {
    live = c < G;
    return static_cast<int64_t>(v) * a.Hq + hkv * G + c;
  }
  const int t = (v % a.verify_ng) * a.verify_dps + c / G;
  live = c < a.verify_dps * G && t < a.verify_T;
  return (static_cast<int64_t>(v / a.verify_ng) * a.verify_T + t) * a.Hq + hkv * G + c % G;
}

__device__ __forceinline__ int clamp_len(const DecodeArgs& a, int b, DeviceStatus* st, bool report) {
  int L = a.seqlens[cache_seq(a, b)];
  if (L < 0 || L > a.Lmax) {
    if (report) record_status(st, kStatusBadArg, 700);
    L = L < 0 ? 0 : a.Lmax;
  }
  return L;
}

// Lengths, tail keys (unsorted) and the prefix of the full slots; one warp.
__device__ void sched_prefix_warp(const DecodeArgs& a, Sched* sc, DeviceStatus* st) {
  const int lane = threadIdx.x & 31;
  int n2 = 32;
  while (n2 < a.B) n2 <<= 1;
  // lane owns b = lane * per .. : lengths, tail keys, full-slot counts
  const int per = (a.B + 31) / 32, b0 = lane * per, b1 = min(b0 + per, a.B);
  int sum = 0, tails = 0;
  for (int b = b0; b < b1; ++b) {
    const int L = clamp_len(a, b, st, blockIdx.x == 0);
    sc->len[b] = L;
    const int nf = min(L / a.split_size, a.num_splits);
    const int tail = L - nf * a.split_size;
    sc->key[b] = tail > 0 ? (static_cast<uint32_t>(a.split_size - tail) << 16) | static_cast<uint32_t>(b) : 0xffffffffu;
    sum += nf * a.Hkv;
    tails += tail > 0;
  }
  for (int b = a.B + lane; b < n2; b += 32) sc->key[b] = 0xffffffffu;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tails += __shfl_xor_sync(0xffffffffu, tails, o);
  int run = incl - sum;
  for (int b = b0; b < b1; ++b) {
    sc->pf[b] = run;
    run += min(sc->len[b] / a.split_size, a.num_splits) * a.Hkv;
  }
  if (lane == 31) {
    sc->pf[a.B] = incl;
    sc->n_full = incl;
  }
  if (lane == 0) sc->n_tail = tails * a.Hkv;
  __syncwarp();
}

// Bitonic sort of the tail keys, ascending (longest tail first); one warp.
__device__ void sched_sort_warp(const DecodeArgs& a, Sched* sc) {
  const int lane = threadIdx.x & 31;
  int n2 = 32;
  while (n2 < a.B) n2 <<= 1;
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = lane; i < n2 / 2; i += 32) {
        const int lo = (i / stride) * 2 * stride + (i % stride), hi = lo + stride;
        const uint32_t x = sc->key[lo], y = sc->key[hi];
        if ((x > y) == ((lo & size) == 0)) {
          sc->key[lo] = y;
          sc->key[hi] = x;
        }
      }
      __syncwarp();
    }
  }
}

// Number of entries in the launch's slot list.
__device__ __forceinline__ int64_t slot_count(const DecodeArgs& a, const Sched* sc, bool balanced) {
  return balanced ? static_cast<int64_t>(sc->n_full) + sc->n_tail
                  : static_cast<int64_t>(a.num_splits) * a.B * a.Hkv;
}

// Entry j of the slot list; false if it is empty (split-major order only).  Tail
// entries (j >= n_full) need the sorted keys.
__device__ __forceinline__ bool slot_at(const DecodeArgs& a, const Sched* sc, bool balanced, int64_t j, Slot& s) {
  if (!balanced) {
    const int64_t per = static_cast<int64_t>(a.B) * a.Hkv;
    s.split = static_cast<int>(j / per);
    const int64_t r = j - s.split * per;
    s.b = static_cast<int>(r / a.Hkv);
    s.hkv = static_cast<int>(r - static_cast<int64_t>(s.b) * a.Hkv);
    int L = a.seqlens[cache_seq(a, s.b)];
    L = L < 0 ? 0 : (L > a.Lmax ? a.Lmax : L);
    s.t0 = s.split * a.split_size;
    s.t1 = min(s.t0 + a.split_size, L);
    return s.t0 < s.t1;
  }
  if (j < sc->n_full) {
    const int jj = static_cast<int>(j);
    int lo = 0, hi = a.B;  // last b with pf[b] <= j
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sc->pf[mid] <= jj) lo = mid;
      else hi = mid;
    }
    const int r = jj - sc->pf[lo];
    s.b = lo;
    s.split = r / a.Hkv;
    s.hkv = r - s.split * a.Hkv;
    s.t0 = s.split * a.split_size;
    s.t1 = s.t0 + a.split_size;
    return true;
  }
  const int i = static_cast<int>(j - sc->n_full);
  s.b = static_cast<int>(sc->key[i / a.Hkv] & 0xffffu);
  s.hkv = i % a.Hkv;
  const int L = sc->len[s.b];
  s.split = min(L / a.split_size, a.num_splits);
  s.t0 = s.split * a.split_size;
  s.t1 = L;
  return true;
}

// Tensor maps of the two caches.  Contiguous cache: [0] only, boxes of one stage
// (kChunk rows).  Paged cache: boxes of 16 << i rows (i < kPageBoxes), so that a stage's
// rows inside one page go in a few large copies.
constexpr int kPageBoxes = 4;
struct CacheMaps {
  CUtensorMap k[kPageBoxes], v[kPageBoxes];
};

// kVerify: the speculative-verify form (a.verify_T > 0), built apart so that plain decode
// carries none of its per-column masks.
template <int D, bool kV16, bool kVerify>
__global__ void __launch_bounds__(DCfg<D, kV16>::kThreads, 1)
    decode_split_kernel(const DecodeArgs a, const __grid_constant__ CacheMaps maps, uint32_t ticket,
                        DeviceStatus* st, uint64_t limit_ns) {
  using C = DCfg<D, kV16>;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBar);  // stage ring
  uint64_t* empty = full + kStages;
  uint64_t* raw_full = empty + kStages;  // raw q rows (loader -> q warp)
  uint64_t* raw_empty = raw_full + kQSlots;
  uint64_t* qc_full = raw_empty + kQSlots;  // quantised q rows (q warp -> compute warps)
  uint64_t* qc_empty = qc_full + kQSlots;
  uint64_t* red_full = qc_empty + kQSlots;  // per-warp split states (compute warps -> merging warp)
  uint64_t* red_empty = red_full + 1;
  uint64_t* sched_sorted = red_empty + 1;  // tail keys sorted (merging warp -> loader)
  Sched* sc = reinterpret_cast<Sched*>(smem + C::kSched);
  float* stat = reinterpret_cast<float*>(smem + C::kStat);  // [warp][8 q][m, l, -, -]
  float* red = reinterpret_cast<float*>(smem + C::kRed);    // [warp][d][8 q]

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int G = a.Hq / a.Hkv;
  const int GC = kVerify ? a.verify_dps * G : G;  // query columns of a slot
  const bool balanced = a.B <= kSchedMaxB;
  const int q_elem = a.q_dtype == SL8_F32 ? 4 : 2;
  // scales ride the bulk copies when every stage's range is 16-byte aligned
  const bool scales_bulk = (a.Lmax % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.k_scale) |
                                                  reinterpret_cast<uintptr_t>(a.v_scale)) & 15u) == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], C::kNW);
    }
    for (int i = 0; i < kQSlots; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], GC);  // the warps quantising the rows
      mbar_init(&qc_full[i], GC);
      mbar_init(&qc_empty[i], C::kNW);
    }
    mbar_init(red_full, C::kNW);
    mbar_init(red_empty, 1);
    mbar_init(sched_sorted, 1);
    fence_barrier_init();
  }
  // the loader's warp lays out the slot list before anyone uses it; the merging warp
  // sorts the tail keys in the background
  if (balanced && warp == 0) sched_prefix_warp(a, sc, st);
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      for (int i = 0; i < (a.block_table ? kPageBoxes : 1); ++i) {
        prefetch_tensormap(&maps.k[i]);
        prefetch_tensormap(&maps.v[i]);
      }
    }
    // Slot n + 1 is claimed (and its q rows requested) before the stages of slot n, so
    // that its q rows are quantised while slot n streams; the claim of slot n + 2 is in
    // flight meanwhile.
    const int64_t total = slot_count(a, sc, balanced);
    uint32_t* counter = &g_claim[ticket][0];
    uint32_t k = 0, n = 0;  // stages issued, current slot
    bool ok = true, sorted = !balanced;
    // the next entry of the slot list for this CTA: entry blockIdx.x first, then claims
    int64_t first = blockIdx.x;
    uint32_t pending = 0;  // claim in flight (valid when claiming)
    bool claiming = false, exhausted = static_cast<int64_t>(blockIdx.x) >= total;
    auto next_entry = [&](Slot& x) {
      while (!exhausted) {
        int64_t j;
        if (first >= 0) {
          j = first;
          first = -1;
        } else {
          if (!claiming) {
            if (lane == 0) pending = atomicAdd(counter, 1u);
            claiming = true;
          }
          j = static_cast<int64_t>(__shfl_sync(0xffffffffu, pending, 0)) + gridDim.x;
          claiming = false;
        }
        if (j >= total) {
          exhausted = true;
          break;
        }
        // start the following claim now; its result is read at the next call
        if (lane == 0) pending = atomicAdd(counter, 1u);
        claiming = true;
        if (balanced && j >= sc->n_full && !sorted) {
          sorted = warp_wait(sched_sorted, 0, limit_ns, st, 48);
          if (!sorted) {
            ok = false;
            exhausted = true;
            break;
          }
        }
        if (slot_at(a, sc, balanced, j, x)) return true;
      }
      x.b = -1;  // no more slots
      return false;
    };
    // announce slot i (or the end) to the compute warps and request its q rows
    auto announce = [&](const Slot& x, uint32_t i) {
      const uint32_t qs = i % kQSlots;
      if (i >= kQSlots && !warp_wait(&raw_empty[qs], ((i / kQSlots) - 1) & 1, limit_ns, st, 42)) return false;
      if (lane == 0) {
        sc->ring[i % kSlotRing] = x;
        if (x.b >= 0) {
          // the G rows of each live group of columns (one group unless verifying)
          const uint32_t q_bytes = static_cast<uint32_t>(G * D * q_elem);
          int groups = 0;
          for (int c = 0; c < GC; c += G) {
            bool live;
            col_row<kVerify>(a, x.b, x.hkv, c, G, live);
            groups += live ? 1 : 0;
          }
          mbar_arrive_expect_tx(&raw_full[qs], q_bytes * groups);
          for (int c = 0; c < GC; c += G) {
            bool live;
            const int64_t row = col_row<kVerify>(a, x.b, x.hkv, c, G, live);
            if (live)
              bulk_load(smem + C::kQ + qs * C::kQBytes + c * D * q_elem,
                        static_cast<const uint8_t*>(a.q) + row * D * q_elem, q_bytes, &raw_full[qs]);
          }
        } else {
          mbar_arrive(&raw_full[qs]);
        }
      }
      return true;
    };
    const bool paged = !kV16 && a.block_table != nullptr;
    Slot cur, nxt;
    bool has_cur = next_entry(cur);
    ok = ok && announce(cur, 0);
    while (ok && has_cur) {
      const bool has_nxt = next_entry(nxt);
      if (!ok || !announce(nxt, n + 1)) break;
      const int64_t row0 = (static_cast<int64_t>(cache_seq(a, cur.b)) * (a.Hkv / a.kv_groups) + cur.hkv / a.kv_groups) *
                           a.Lmax;
      for (int c0 = cur.t0; c0 < cur.t1 && ok; c0 += C::kChunk, ++k) {
        const int nt = min(C::kChunk, cur.t1 - c0);
        const uint32_t stg = k % kStages;
        uint8_t* base = smem + stg * C::kStageBytes;
        // paged cache: the page of this lane's unit, read before the wait for the stage
        // so that the wait covers the load's latency
        const int t = c0 + lane * kUnit;
        const int units = (nt + kUnit - 1) / kUnit;
        int pg = 0;
        if (paged && lane < units) pg = a.block_table[static_cast<int64_t>(cur.b) * a.max_blocks + t / a.page_size];
        if (k >= kStages) ok = warp_wait(&empty[stg], ((k / kStages) - 1) & 1, limit_ns, st, 41);
        if (!ok) break;
        if (paged) {
          // paged cache: the stage's 16-token units (page_size is a multiple of 16; units
          // past the split's end are not loaded, their compute warps skip them) fall into
          // pieces that each lie in one page; the lane of a piece's first unit loads the
          // piece in boxes of 128/64/32/16 rows and its scales in one bulk copy each
          if (lane == 0)
            mbar_arrive_expect_tx(&full[stg], static_cast<uint32_t>(units * 2 * kUnit * (D + 4)));
          __syncwarp();
          if (lane < units && (lane == 0 || t % a.page_size == 0)) {
            const int rows = min(a.page_size - t % a.page_size, (units - lane) * kUnit);
            if (pg < 0 || pg >= a.num_pages) {
              record_status(st, kStatusBadArg, 49);
              pg = 0;
            }
            const int64_t prow = (static_cast<int64_t>(pg) * (a.Hkv / a.kv_groups) + cur.hkv / a.kv_groups) * a.page_size +
                                 t % a.page_size;
            for (int r = 0; r < rows;) {
              const int left = rows - r;
              const int i = left >= 128 ? 3 : left >= 64 ? 2 : left >= 32 ? 1 : 0;
#pragma unroll
              for (int b = 0; b < C::kBoxes; ++b) {
                const uint32_t dst = static_cast<uint32_t>(b * C::kChunk * C::kBW + (lane * kUnit + r) * C::kBW);
                tma_load_3d(base + C::kSK + dst, &maps.k[i], &full[stg], b * C::kBW, static_cast<int>(prow + r), 0);
                tma_load_3d(base + C::kSV + dst, &maps.v[i], &full[stg], b * C::kBW, static_cast<int>(prow + r), 0);
              }
              r += kUnit << i;
            }
            bulk_load(base + C::kSKs + lane * kUnit * 4, a.k_scale + prow, static_cast<uint32_t>(rows * 4), &full[stg]);
            bulk_load(base + C::kSVs + lane * kUnit * 4, a.v_scale + prow, static_cast<uint32_t>(rows * 4), &full[stg]);
          }
          continue;
        }
        if (!scales_bulk) {
          for (int j = lane; j < nt; j += 32) {
            reinterpret_cast<float*>(base + C::kSKs)[j] = a.k_scale[row0 + c0 + j];
            if (!kV16) reinterpret_cast<float*>(base + C::kSVs)[j] = a.v_scale[row0 + c0 + j];
          }
          __syncwarp();
        }
        if (lane == 0) {
          const uint32_t sc_bytes = scales_bulk ? static_cast<uint32_t>((nt + 3) / 4 * 16) : 0u;
          mbar_arrive_expect_tx(&full[stg], C::kTile + C::kTileV + (kV16 ? 1 : 2) * sc_bytes);
          const int y = static_cast<int>(row0 + c0);
#pragma unroll
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(base + C::kSK + b * C::kChunk * C::kBW, &maps.k[0], &full[stg], b * C::kBW, y, 0);
#pragma unroll
          for (int b = 0; b < C::kBoxesV; ++b)  // V16: boxes of 64 fp16 dims
            tma_load_3d(base + C::kSV + b * C::kChunk * (kV16 ? 128 : C::kBW), &maps.v[0], &full[stg],
                        b * (kV16 ? 64 : C::kBW), y, 0);
          if (scales_bulk) {
            bulk_load(base + C::kSKs, a.k_scale + row0 + c0, sc_bytes, &full[stg]);
            if (!kV16) bulk_load(base + C::kSVs, a.v_scale + row0 + c0, sc_bytes, &full[stg]);
          }
        }
      }
      cur = nxt;
      has_cur = has_nxt;
      ++n;
    }
    // This CTA claims no more; a claim still in flight is part of the count.  The last
    // CTA of the launch resets the ticket's counters.
    if (lane == 0) {
      if (claiming) {
        volatile uint32_t settled = pending;  // the claim in flight has completed
        (void)settled;
      }
      __threadfence();
      if (atomicAdd(&g_claim[ticket][1], 1u) == gridDim.x - 1) {
        atomicExch(&g_claim[ticket][0], 0u);
        atomicExch(&g_claim[ticket][1], 0u);
      }
    }
    return;  // nothing waits on the loader beyond the rings
  }

  if (warp == 1) {
    // ------------------------------------------------------------ merges
    bool ok = true;
    uint32_t n = 0;
    auto merge = [&](const Slot& m, uint32_t mi) {
      // lane q < GC: the split's max and sum of query column q over the warps
      bool lane_live;
      const int64_t lane_row = col_row<kVerify>(a, m.b, m.hkv, lane & 7, G, lane_live);
      float M = -INFINITY, L = 0.0f;
      if (lane < GC) {
#pragma unroll
        for (int w = 0; w < C::kNW; ++w) M = fmaxf(M, stat[(w * 8 + lane) * 4]);
#pragma unroll
        for (int w = 0; w < C::kNW; ++w) {
          const float mw = stat[(w * 8 + lane) * 4];
          if (mw != -INFINITY) L += stat[(w * 8 + lane) * 4 + 1] * ex2(mw - M);
        }
        if (lane_live) a.lse_partial[lane_row * a.num_splits + m.split] = (M + log2f(L)) * 0.6931471805599453f;
      }
      // weight of warp w's state for query q: 2^(m_w - M) / L
      const int nq4 = GC > 4 ? 2 : 1;  // float4 groups of query columns
      const float rL = lane < GC ? 1.0f / L : 0.0f;
      float wt[C::kNW][8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float Mq = __shfl_sync(0xffffffffu, M, q), rLq = __shfl_sync(0xffffffffu, rL, q);
#pragma unroll
        for (int w = 0; w < C::kNW; ++w) {
          const float mw = stat[(w * 8 + q) * 4];
          wt[w][q] = mw == -INFINITY ? 0.0f : ex2(mw - Mq) * rLq;
        }
      }
      // lane: dims lane + 32 i, all query columns of the group
      for (int dim = lane; dim < D; dim += 32) {
        float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int w = 0; w < C::kNW; ++w) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h < nq4) {
              const float4 r4 = *reinterpret_cast<const float4*>(red + (w * D + dim) * 8 + 4 * h);
              acc[4 * h] = fmaf(r4.x, wt[w][4 * h], acc[4 * h]);
              acc[4 * h + 1] = fmaf(r4.y, wt[w][4 * h + 1], acc[4 * h + 1]);
              acc[4 * h + 2] = fmaf(r4.z, wt[w][4 * h + 2], acc[4 * h + 2]);
              acc[4 * h + 3] = fmaf(r4.w, wt[w][4 * h + 3], acc[4 * h + 3]);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          bool live;
          const int64_t row = col_row<kVerify>(a, m.b, m.hkv, q, G, live);
          if (live) a.o_partial[(row * a.num_splits + m.split) * D + dim] = acc[q];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(red_empty);
      return true;
    };
    if (balanced) {
      sched_sort_warp(a, sc);
      if (lane == 0) mbar_arrive(sched_sorted);
    }
    // the compute warps hand over slot n with red_full; a slot with b < 0 ends the list
    while (ok) {
      if (!warp_wait(red_full, n & 1, limit_ns, st, 45)) break;
      const Slot m = sc->merge;
      if (m.b < 0) break;
      ok = merge(m, n);
      ++n;
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  const int ct = threadIdx.x - 32 * kFirstCompute;  // 0 .. 255
  const int cw = ct / 32;                            // compute warp 0 .. 7
  const int g = lane >> 2, t = lane & 3;
  const int u0 = kUnit * cw;  // this warp's rows in every stage
  // S^T row r (and r + 8) holds unit token tok(r) (and tok(r) + 8).  The permutation keeps
  // the K reads (row tok(g), 16-byte chunk t; 8-byte piece t at d = 32) and the V reads
  // (rows tok(2t), tok(2t + 1), + 8) free of bank conflicts, or at two ways for the
  // 64-byte rows of d = 64.
  auto tok = [](int r) {
    if constexpr (C::kSwz) return (r >> 1) + 4 * (r & 1);
    if constexpr (D == 32) return (r & 1) ? 4 + (((r >> 1) + 2) & 3) : (r >> 1);
    return (r & 1) ? 4 + ((r >> 1) ^ 1) : (r >> 1);
  };
  const int pi = tok(g);
  // V^T rows of this lane: 16-byte chunk (8-byte piece for d = 64) pi of each V row
  const int cg = pi;
  // stage-tile offsets of this lane's reads, the same for every stage
  constexpr int kKH = D >= 64 ? D / 64 : 1;  // 64-dim parts of a K row (d = 32: one 32-byte row)
  uint32_t offk[kKH][2];
  if constexpr (D == 32) {
    offk[0][0] = static_cast<uint32_t>((u0 + pi) * 32 + 8 * t);
    offk[0][1] = static_cast<uint32_t>((u0 + pi + 8) * 32 + 8 * t);
  } else {
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      offk[h][0] = tile_off<D>(u0 + pi, 4 * h + t);
      offk[h][1] = tile_off<D>(u0 + pi + 8, 4 * h + t);
    }
  }
  // V rows: the k columns 2t, 2t+1, 2t+8, 2t+9 of P'^T are the S^T rows 2t, 2t+1 of the
  // two 8-row halves (movm_t transposes each half), i.e. unit tokens tok(2t), tok(2t+1)
  // and the same + 8
  uint32_t offv[C::kBoxes][4];
#pragma unroll
  for (int b = 0; b < C::kBoxes; ++b)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int row = u0 + tok(2 * t + (c & 1)) + 8 * (c >> 1);
      offv[b][c] = D == 32   ? static_cast<uint32_t>(row * 32 + 4 * cg)
                 : D == 64 ? static_cast<uint32_t>(row * 64 + 8 * cg)
                           : tile_off<D>(row, 8 * b + cg);
    }
  // fp16 V: this lane's ldmatrix row address for m-tile j (dims 16 j ..): it serves matrix
  // i = lane / 8 (dims + 8 (i % 2); k columns 8 (i / 2) ..) and its row r = lane % 8, the
  // token at k column 8 (i / 2) + r: tok(r) + 8 (i / 2)
  uint32_t offv16[kV16 ? D / 16 : 1];
  if constexpr (kV16) {
    const int i = lane >> 3, r = lane & 7;
    const int row = u0 + 8 * (i >> 1) + tok(r);
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      const int chunk = 2 * j + (i & 1);
      offv16[j] = static_cast<uint32_t>((chunk >> 3) * (C::kChunk * 128) + row * 128 + 16 * ((chunk & 7) ^ (row & 7)));
    }
  }
  const float log2e_over_sqrtd = 1.4426950408889634f / sqrtf(static_cast<float>(D));

  // ---- empty splits, up front: lse = -inf (their O is never read), and the q codes of
  // an empty sequence when asked; sequences b = blockIdx.x + k * gridDim.x
  for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
    const int L = clamp_len(a, b, st, !balanced && ct == 0);
    const int ns = (L + a.split_size - 1) / a.split_size;
    // the rows of sequence b: its Hq heads, or (verify) those of its drafts
    const int nd = kVerify ? min(a.verify_dps, a.verify_T - (b % a.verify_ng) * a.verify_dps) : 1;
    const int n_empty = (a.num_splits - ns) * nd * a.Hq;
    for (int e = ct; e < n_empty; e += C::kCT) {
      const int split = ns + e / (nd * a.Hq), r = e % (nd * a.Hq);
      const int64_t row = kVerify ? (static_cast<int64_t>(b / a.verify_ng) * a.verify_T +
                                        (b % a.verify_ng) * a.verify_dps + r / a.Hq) * a.Hq + r % a.Hq
                                     : static_cast<int64_t>(b) * a.Hq + r;
      a.lse_partial[row * a.num_splits + split] = -INFINITY;
    }
    if (L == 0 && a.q_codes) {
      for (int hq = cw; hq < a.Hq; hq += C::kNW) {
        const int64_t row = static_cast<int64_t>(b) * a.Hq + hq;
        float v[D / 32];
        int8_t code[D / 32];
#pragma unroll
        for (int e = 0; e < D / 32; ++e) v[e] = load_q_elem(a.q, a.q_dtype, row * D + lane * (D / 32) + e);
        const float scq = quant_row_warp<D>(v, code);
#pragma unroll
        for (int e = 0; e < D / 32; ++e) a.q_codes[row * D + lane * (D / 32) + e] = code[e];
        if (lane == 0) a.q_scales[row] = scq;
      }
    }
  }

  // compute warp r < G quantises q row r of each split into qc[split % 2], one split
  // ahead (split 0 before the loop)
  auto quant_row = [&](uint32_t i) {
    const uint32_t qs = i % kQSlots;
    if (!warp_wait(&raw_full[qs], (i / kQSlots) & 1, limit_ns, st, 43)) return false;
    if (i >= kQSlots && !warp_wait(&qc_empty[qs], ((i / kQSlots) - 1) & 1, limit_ns, st, 44)) return false;
    const Slot x = sc->ring[i % kSlotRing];
    if (x.b < 0) {  // the list has ended: nothing to quantise
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&raw_empty[qs]);
        mbar_arrive(&qc_full[qs]);
      }
      return true;
    }
    const uint8_t* raw = smem + C::kQ + qs * C::kQBytes + cw * D * q_elem;
    bool col_live;
    col_row<kVerify>(a, x.b, x.hkv, cw, G, col_live);  // dead verify columns quantise zeros
    int8_t* qc = reinterpret_cast<int8_t*>(smem + C::kQc + qs * C::kQcBytes);
    float* qinfo = reinterpret_cast<float*>(qc + 8 * D);  // [8] scales, [8] code sums
    float v[D / 32];
    int8_t code[D / 32];
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      const int idx = lane * (D / 32) + e;
      v[e] = !col_live ? 0.0f
           : a.q_dtype == SL8_F32 ? reinterpret_cast<const float*>(raw)[idx]
           : a.q_dtype == SL8_BF16 ? bf16_bits(reinterpret_cast<const uint16_t*>(raw)[idx])
                                   : f16_bits(reinterpret_cast<const uint16_t*>(raw)[idx]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&raw_empty[qs]);
    const float scq = quant_row_warp<D>(v, code);
    int csum = 0;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      qc[cw * D + lane * (D / 32) + e] = code[e];
      csum += code[e];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) csum += __shfl_xor_sync(0xffffffffu, csum, o);
    if (lane == 0) {
      qinfo[cw] = scq;
      qinfo[8 + cw] = static_cast<float>(csum);
    }
    if (a.q_codes && x.split == 0) {
      const int64_t row = static_cast<int64_t>(x.b) * a.Hq + x.hkv * G + cw;
#pragma unroll
      for (int e = 0; e < D / 32; ++e) a.q_codes[row * D + lane * (D / 32) + e] = code[e];
      if (lane == 0) a.q_scales[row] = scq;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&qc_full[qs]);
    return true;
  };

  uint32_t k = 0, n = 0;
  bool ok = true;
  Slot s;
  if (cw < GC) ok = quant_row(0);
  while (ok) {
    // ---- slot n, as announced by the loader (b < 0: the list has ended)
    const uint32_t qs = n % kQSlots;
    if (!warp_wait(&qc_full[qs], (n / kQSlots) & 1, limit_ns, st, 46)) {
      ok = false;
      break;
    }
    s = sc->ring[n % kSlotRing];
    if (s.b < 0) break;
    const int64_t part_row0 = static_cast<int64_t>(s.b) * a.Hq + s.hkv * G;  // first (b, hq) row
    // ---- B fragments of Q^T from the quantised rows: k-step 4h + j holds dims
    // 64h + 16t + 4j + {0, 1} | {2, 3} of query row g (exact fp16 integers); zero past G
    const int8_t* qc = reinterpret_cast<const int8_t*>(smem + C::kQc + qs * C::kQcBytes);
    const float* qinfo = reinterpret_cast<const float*>(qc + 8 * D);
    uint32_t qb[D / 16][2];
    if constexpr (D == 32) {
      // k-step j holds dims 8t + 4j + {0, 1} | {2, 3}
      uint2 w = make_uint2(0u, 0u);
      if (g < GC) w = *reinterpret_cast<const uint2*>(qc + g * D + 8 * t);
      const uint32_t ww[2] = {w.x, w.y};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t u = ww[j] ^ 0x80808080u;
        qb[j][0] = g < GC ? codes_f16x2(u, 0x4140) : 0u;
        qb[j][1] = g < GC ? codes_f16x2(u, 0x4342) : 0u;
      }
    }
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (g < GC) w = *reinterpret_cast<const uint4*>(qc + g * D + 64 * h + 16 * t);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t u = ww[j] ^ 0x80808080u;
        qb[4 * h + j][0] = g < GC ? codes_f16x2(u, 0x4140) : 0u;
        qb[4 * h + j][1] = g < GC ? codes_f16x2(u, 0x4342) : 0u;
      }
    }
    // query columns qa = 2t, qb = 2t + 1: dequantisation factors (log2 units) and the
    // offset of the biased K codes, -128 * sum(q codes)
    const float qsa = 2 * t < GC ? qinfo[2 * t] * log2e_over_sqrtd : 0.0f;
    const float qsb = 2 * t + 1 < GC ? qinfo[2 * t + 1] * log2e_over_sqrtd : 0.0f;
    const float offa = 2 * t < GC ? -128.0f * qinfo[8 + 2 * t] : 0.0f;
    const float offb = 2 * t + 1 < GC ? -128.0f * qinfo[8 + 2 * t + 1] : 0.0f;
    __syncwarp();
    if (lane == 0) mbar_arrive(&qc_empty[qs]);
    if (cw < GC && !quant_row(n + 1)) {
      ok = false;
      break;
    }

    // ---- per-warp online softmax state for the two query columns
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.0f, l_b = 0.0f;
    float tha = -INFINITY, thb = -INFINITY;  // m + lazy headroom
    int E = -126;                            // P' carries s_v * 2^-E
    float vlim = pow2i(-126), inv = pow2i(126);
    float o[D / 16][4], osum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < D / 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
    // verify: the slot's draft tokens start at v_tail; mask_a / mask_b say which of them
    // the lane's query columns 2t and 2t + 1 see
    int v_tail = 0;
    uint32_t mask_a = 0, mask_b = 0;
    if constexpr (kVerify) {
      v_tail = (balanced ? sc->len[s.b] : clamp_len(a, s.b, st, false)) - a.verify_T;
      bool la, lb;
      const int64_t ra_ = col_row<kVerify>(a, s.b, s.hkv, 2 * t, G, la), rb_ = col_row<kVerify>(a, s.b, s.hkv, 2 * t + 1, G, lb);
      if (la) mask_a = a.tree_mask[ra_ / a.Hq];
      if (lb) mask_b = a.tree_mask[rb_ / a.Hq];
    }
    for (int c0 = s.t0; c0 < s.t1 && ok; c0 += C::kChunk, ++k) {
      const int ntok = min(C::kChunk, s.t1 - c0);
      const uint32_t stg = k % kStages;
      const uint8_t* base = smem + stg * C::kStageBytes;
      if (!warp_wait(&full[stg], (k / kStages) & 1, limit_ns, st, 40)) {
        ok = false;
        break;
      }
      const int nv = ntok - u0;  // valid tokens of this warp's unit
      auto unit = [&](auto full_tag) {
        constexpr bool kFull = decltype(full_tag)::value;
        const uint8_t* sk = base + C::kSK;
        const uint8_t* sv = base + C::kSV;
        const float* sks = reinterpret_cast<const float*>(base + C::kSKs);
        const float* svs = reinterpret_cast<const float*>(base + C::kSVs);
        // ---- S'^T = K_biased . Q^T: K codes + 128 enter as fp16 subnormals (u * 2^-24), so
        // S = 2^24 S' - 128 sum(q) exactly (two accumulation chains)
        float s0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if constexpr (D == 32) {
          const uint2 wa = *reinterpret_cast<const uint2*>(sk + offk[0][0]);
          const uint2 wb = *reinterpret_cast<const uint2*>(sk + offk[0][1]);
          const uint32_t A[2] = {wa.x, wa.y}, Bw[2] = {wb.x, wb.y};
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t ua = A[j] ^ 0x80808080u, ub = Bw[j] ^ 0x80808080u;
            mma_f16(j & 1 ? s1 : s0, prmt(ua, 0u, 0x4140), prmt(ub, 0u, 0x4140), prmt(ua, 0u, 0x4342),
                    prmt(ub, 0u, 0x4342), qb[j][0], qb[j][1]);
          }
        }
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          const uint4 wa = *reinterpret_cast<const uint4*>(sk + offk[h][0]);
          const uint4 wb = *reinterpret_cast<const uint4*>(sk + offk[h][1]);
          const uint32_t A[4] = {wa.x, wa.y, wa.z, wa.w}, Bw[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t ua = A[j] ^ 0x80808080u, ub = Bw[j] ^ 0x80808080u;
            mma_f16(j & 1 ? s1 : s0, prmt(ua, 0u, 0x4140), prmt(ub, 0u, 0x4140), prmt(ua, 0u, 0x4342),
                    prmt(ub, 0u, 0x4342), qb[4 * h + j][0], qb[4 * h + j][1]);
          }
        }
        constexpr float k2p24 = 16777216.0f;
        const float d00 = fmaf(s0[0] + s1[0], k2p24, offa), d01 = fmaf(s0[1] + s1[1], k2p24, offb);
        const float d10 = fmaf(s0[2] + s1[2], k2p24, offa), d11 = fmaf(s0[3] + s1[3], k2p24, offb);
        const int rA = u0 + pi, rB = rA + 8;
        const bool vA = kFull || pi < nv, vB = kFull || pi + 8 < nv;
        // per query column: verify shows the draft tokens from v_tail on as the masks say
        bool vAa = vA, vAb = vA, vBa = vB, vBb = vB;
        if (kVerify && !kFull) {
          const int tA = c0 + rA, tB = c0 + rB;
          if (tA >= v_tail) {
            vAa = vAa && ((mask_a >> (tA - v_tail)) & 1u);
            vAb = vAb && ((mask_b >> (tA - v_tail)) & 1u);
          }
          if (tB >= v_tail) {
            vBa = vBa && ((mask_a >> (tB - v_tail)) & 1u);
            vBb = vBb && ((mask_b >> (tB - v_tail)) & 1u);
          }
        }
        if (a.logits) {
          int32_t* lg = a.logits + c0;
          if (2 * t < G) {
            if (vA) lg[(part_row0 + 2 * t) * a.Lmax + rA] = static_cast<int32_t>(d00);
            if (vB) lg[(part_row0 + 2 * t) * a.Lmax + rB] = static_cast<int32_t>(d10);
          }
          if (2 * t + 1 < G) {
            if (vA) lg[(part_row0 + 2 * t + 1) * a.Lmax + rA] = static_cast<int32_t>(d01);
            if (vB) lg[(part_row0 + 2 * t + 1) * a.Lmax + rB] = static_cast<int32_t>(d11);
          }
        }
        // ---- online softmax (log2 units), lazily rescaled
        const float ksA = vA ? sks[rA] : 0.0f, ksB = vB ? sks[rB] : 0.0f;
        const float vsA = vA ? (kV16 ? 1.0f : svs[rA]) : 0.0f, vsB = vB ? (kV16 ? 1.0f : svs[rB]) : 0.0f;
        const float ka = ksA * qsa, kb = ksA * qsb, kc = ksB * qsa, kd = ksB * qsb;
        const float xa0 = vAa ? d00 * ka : -INFINITY, xa1 = vAb ? d01 * kb : -INFINITY;
        const float xb0 = vBa ? d10 * kc : -INFINITY, xb1 = vBb ? d11 * kd : -INFINITY;
        const bool grow = (fmaxf(xa0, xb0) > tha) || (fmaxf(xa1, xb1) > thb) || (fmaxf(vsA, vsB) > vlim);
        if (__any_sync(0xffffffffu, grow)) {
          const float ma = col_max(fmaxf(xa0, xb0)), mb = col_max(fmaxf(xa1, xb1));
          const float vm = col_max(fmaxf(vsA, vsB));
          float fa = 1.0f, fb = 1.0f;
          if (ma > tha) {
            fa = m_a == -INFINITY ? 0.0f : ex2(m_a - ma);
            l_a *= fa;
            m_a = ma;
            tha = ma + kLazy;
          }
          if (mb > thb) {
            fb = m_b == -INFINITY ? 0.0f : ex2(m_b - mb);
            l_b *= fb;
            m_b = mb;
            thb = mb + kLazy;
          }
          if (vm > vlim) {  // uniform: vm is the unit's max over all lanes
            int e = static_cast<int>((__float_as_uint(vm) >> 23) & 0xffu) - 126;  // vm < 2^e
            e = e > 126 ? 126 : e;
            const float fe = pow2i(E - e);
            fa *= fe;
            fb *= fe;
            E = e;
            vlim = pow2i(e);
            inv = pow2i(-e);
          }
#pragma unroll
          for (int j = 0; j < D / 16; ++j) {
            o[j][0] *= fa;
            o[j][2] *= fa;
            o[j][1] *= fb;
            o[j][3] *= fb;
          }
          osum[0] *= fa;
          osum[2] *= fa;
          osum[1] *= fb;
          osum[3] *= fb;
        }
        // a column with no visible token yet (verify masks can hide a warp's whole first
        // unit) keeps m = -inf: its p must be 0, not exp(-inf - -inf)
        const float ra = m_a == -INFINITY ? 0.0f : m_a, rb = m_b == -INFINITY ? 0.0f : m_b;
        const float pa0 = ex2(xa0 - ra), pa1 = ex2(xa1 - rb), pb0 = ex2(xb0 - ra), pb1 = ex2(xb1 - rb);
        l_a += pa0 + pb0;
        l_b += pa1 + pb1;
        const float wA = vsA * inv, wB = vsB * inv;
        // ---- P'^T as B fragments: the fp16 S^T layout of P', each 8-row half transposed
        const uint32_t pb0r = movm_t(f16x2_of(pa0 * wA, pa1 * wA));
        const uint32_t pb1r = movm_t(f16x2_of(pb0 * wB, pb1 * wB));
        // ---- O'^T += V_biased^T . P'^T (V codes + 128 as fp16 subnormals), and the row
        // sums of P' from an all-ones A for the offset; fp16 V: O'^T += V^T . P'^T with the
        // A fragments read transposed from the [token][dim] tile
        if constexpr (kV16) {
          const uint32_t svb = smem_u32(sv);
#pragma unroll
          for (int j = 0; j < D / 16; ++j) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(svb + offv16[j], v0, v1, v2, v3);
            mma_f16(o[j], v0, v1, v2, v3, pb0r, pb1r);
          }
        } else if constexpr (D == 32) {
          // one 4-byte piece (dims 4 cg .. 4 cg + 3) of each of the four V rows
          uint32_t w[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const uint32_t*>(sv + offv[0][c]);
          const uint32_t x01 = prmt(w[0], w[1], 0x5140) ^ 0x80808080u, y01 = prmt(w[0], w[1], 0x7362) ^ 0x80808080u;
          const uint32_t x23 = prmt(w[2], w[3], 0x5140) ^ 0x80808080u, y23 = prmt(w[2], w[3], 0x7362) ^ 0x80808080u;
          mma_f16(o[0], prmt(x01, 0u, 0x4140), prmt(x01, 0u, 0x4342), prmt(x23, 0u, 0x4140), prmt(x23, 0u, 0x4342),
                  pb0r, pb1r);
          mma_f16(o[1], prmt(y01, 0u, 0x4140), prmt(y01, 0u, 0x4342), prmt(y23, 0u, 0x4140), prmt(y23, 0u, 0x4342),
                  pb0r, pb1r);
        } else if constexpr (D == 64) {
          uint2 w[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const uint2*>(sv + offv[0][c]);
#pragma unroll
          for (int ii = 0; ii < 2; ++ii) {
            const uint32_t w0 = ii ? w[0].y : w[0].x, w1 = ii ? w[1].y : w[1].x;
            const uint32_t w2 = ii ? w[2].y : w[2].x, w3 = ii ? w[3].y : w[3].x;
            const uint32_t x01 = prmt(w0, w1, 0x5140) ^ 0x80808080u, y01 = prmt(w0, w1, 0x7362) ^ 0x80808080u;
            const uint32_t x23 = prmt(w2, w3, 0x5140) ^ 0x80808080u, y23 = prmt(w2, w3, 0x7362) ^ 0x80808080u;
            mma_f16(o[2 * ii], prmt(x01, 0u, 0x4140), prmt(x01, 0u, 0x4342), prmt(x23, 0u, 0x4140),
                    prmt(x23, 0u, 0x4342), pb0r, pb1r);
            mma_f16(o[2 * ii + 1], prmt(y01, 0u, 0x4140), prmt(y01, 0u, 0x4342), prmt(y23, 0u, 0x4140),
                    prmt(y23, 0u, 0x4342), pb0r, pb1r);
          }
        } else {
#pragma unroll
          for (int b = 0; b < C::kBoxes; ++b) {
            uint4 w[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const uint4*>(sv + offv[b][c]);
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
              const uint32_t w0 = ii == 0 ? w[0].x : ii == 1 ? w[0].y : ii == 2 ? w[0].z : w[0].w;
              const uint32_t w1 = ii == 0 ? w[1].x : ii == 1 ? w[1].y : ii == 2 ? w[1].z : w[1].w;
              const uint32_t w2 = ii == 0 ? w[2].x : ii == 1 ? w[2].y : ii == 2 ? w[2].z : w[2].w;
              const uint32_t w3 = ii == 0 ? w[3].x : ii == 1 ? w[3].y : ii == 2 ? w[3].z : w[3].w;
              const uint32_t x01 = prmt(w0, w1, 0x5140) ^ 0x80808080u, y01 = prmt(w0, w1, 0x7362) ^ 0x80808080u;
              const uint32_t x23 = prmt(w2, w3, 0x5140) ^ 0x80808080u, y23 = prmt(w2, w3, 0x7362) ^ 0x80808080u;
              mma_f16(o[8 * b + 2 * ii], prmt(x01, 0u, 0x4140), prmt(x01, 0u, 0x4342), prmt(x23, 0u, 0x4140),
                      prmt(x23, 0u, 0x4342), pb0r, pb1r);
              mma_f16(o[8 * b + 2 * ii + 1], prmt(y01, 0u, 0x4140), prmt(y01, 0u, 0x4342),
                      prmt(y23, 0u, 0x4140), prmt(y23, 0u, 0x4342), pb0r, pb1r);
            }
          }
        }
        if constexpr (!kV16) mma_f16(osum, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, pb0r, pb1r);
      };
      if (nv >= kUnit && !(kVerify && c0 + u0 + kUnit > v_tail)) {
        unit(std::true_type{});
      } else if (nv > 0) {
        unit(std::false_type{});
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stg]);  // 8 arrivals (one per compute warp) free the stage
    }
    if (!ok) break;
    // ---- hand this warp's state to the merging warp: per query column its max and
    // sum, and O = (2^24 O' - 128 rowsum(P')) * 2^E
    l_a = col_sum(l_a);
    l_b = col_sum(l_b);
    if (n > 0 && !warp_wait(red_empty, (n - 1) & 1, limit_ns, st, 47)) {
      ok = false;
      break;
    }
    if (g == 0) {
      float* sa = stat + (cw * 8 + 2 * t) * 4;
      sa[0] = m_a;
      sa[1] = l_a;
      sa[4] = m_b;
      sa[5] = l_b;
    }
    const float pe = pow2i(E);
    constexpr float k2p24 = 16777216.0f;
    const float ca = -128.0f * osum[0], cb = -128.0f * osum[1];
    if constexpr (kV16) {
      // fp16 V: O = O' 2^E; rows g and g + 8 of m-tile j are dims 16 j + g and 16 j + g + 8
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        *reinterpret_cast<float2*>(red + (cw * D + 16 * j + g) * 8 + 2 * t) = make_float2(o[j][0] * pe, o[j][1] * pe);
        *reinterpret_cast<float2*>(red + (cw * D + 16 * j + g + 8) * 8 + 2 * t) =
            make_float2(o[j][2] * pe, o[j][3] * pe);
      }
    }
#pragma unroll
    for (int j = 0; j < (kV16 ? 0 : D / 16); ++j) {
      // physical dims of rows g and g + 8 of m-tile j
      int dim;
      if constexpr (D == 32) {
        dim = 4 * cg + 2 * j;
      } else if constexpr (D == 64) {
        dim = 8 * cg + 4 * (j >> 1) + 2 * (j & 1);
      } else {
        dim = 128 * (j >> 3) + 16 * cg + 4 * ((j & 7) >> 1) + 2 * (j & 1);
      }
      *reinterpret_cast<float2*>(red + (cw * D + dim) * 8 + 2 * t) =
          make_float2(fmaf(o[j][0], k2p24, ca) * pe, fmaf(o[j][1], k2p24, cb) * pe);
      *reinterpret_cast<float2*>(red + (cw * D + dim + 1) * 8 + 2 * t) =
          make_float2(fmaf(o[j][2], k2p24, ca) * pe, fmaf(o[j][3], k2p24, cb) * pe);
    }
    if (cw == 0 && lane == 0) sc->merge = s;
    __syncwarp();
    if (lane == 0) mbar_arrive(red_full);
    ++n;
  }
  // hand the end of the list to the merging warp
  if (ok && n > 0 && !warp_wait(red_empty, (n - 1) & 1, limit_ns, st, 47)) ok = false;
  if (ok) {
    if (cw == 0 && lane == 0) sc->merge.b = -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(red_full);
  }
}

// One warp per (b, hq): merge the non-empty splits of the row.
template <int D>
__global__ void decode_combine_kernel(const float* __restrict__ o_partial, const float* __restrict__ lse_partial,
                                      const int32_t* __restrict__ seqlens, int32_t B, int32_t Hq, int32_t num_splits,
                                      int32_t split_size, void* out, sl8_dtype out_dtype, float* lse_out,
                                      int32_t seq_div) {
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= B * Hq) return;
  const int b = row / Hq;
  const int L = max(0, seqlens[b / seq_div]);
  const float* lse = lse_partial + static_cast<int64_t>(row) * num_splits;
  const float* op = o_partial + static_cast<int64_t>(row) * num_splits * D + lane * (D / 32);
  constexpr int E = D / 32, K = 8;
  float o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.0f;
  float m = -INFINITY, wsum = 0.0f;
  // K splits at a time: their LSEs (the same word for every lane) and partial rows are
  // all loaded before any is used, together with the length.  An empty split (past the
  // length, or lse = -inf) gets weight 0 and its unwritten row is never multiplied.
  for (int s0 = 0; s0 < num_splits; s0 += K) {
    float ls[K], pre[K][E];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const bool in = s0 + k < num_splits;
      ls[k] = in ? lse[s0 + k] : -INFINITY;
#pragma unroll
      for (int e = 0; e < E; ++e) pre[k][e] = in ? op[static_cast<int64_t>(s0 + k) * D + e] : 0.0f;
    }
    const int ns = min(num_splits, (L + split_size - 1) / split_size);
    float m_new = m;
#pragma unroll
    for (int k = 0; k < K; ++k)
      if (s0 + k < ns) m_new = fmaxf(m_new, ls[k]);
    if (m_new == -INFINITY) continue;  // every split so far is empty
    const float c = m == -INFINITY ? 0.0f : expf(m - m_new);
    wsum *= c;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] *= c;
    m = m_new;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const float w = (s0 + k < ns && ls[k] != -INFINITY) ? expf(ls[k] - m) : 0.0f;
      if (w == 0.0f) continue;
      wsum += w;
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = fmaf(w, pre[k][e], o[e]);
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

template <int D, bool kV16, bool kVerify = false>
cudaError_t launch_split_d(const DecodeArgs& a, cudaStream_t s) {
  using C = DCfg<D, kV16>;
  auto kern = decode_split_kernel<D, kV16, kVerify>;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), C::kBytes);
  if (e != cudaSuccess) return e;
  // each cache as a 2-D [B * Hkv * Lmax rows][d bytes] tensor, loaded in boxes of
  // C::kChunk rows x kBW bytes; a paged cache as [num_pages * Hkv * page_size rows][d],
  // loaded in boxes of one 16-token unit
  const bool paged = a.block_table != nullptr;
  const uint64_t hkv_cache = static_cast<uint64_t>(a.Hkv / a.kv_groups);  // kv heads the cache holds
  const uint64_t rows = paged ? static_cast<uint64_t>(a.num_pages) * hkv_cache * a.page_size
                              : static_cast<uint64_t>(a.B) * hkv_cache * a.Lmax;
  bool ok = true;
  CacheMaps maps;
  memset(&maps, 0, sizeof(maps));
  for (int i = 0; i < (paged ? kPageBoxes : 1); ++i) {
    // a box taller than the whole pool is never used (a piece lies in one page)
    const uint32_t box_rows = paged ? static_cast<uint32_t>(std::min<uint64_t>(static_cast<uint64_t>(kUnit) << i, rows / kUnit * kUnit))
                                    : C::kChunk;
    maps.k[i] = make_tmap_3d(a.k_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, D, rows, 1, D, rows * D, C::kBW, box_rows, 1,
                             &ok, C::kSwz);
    if (kV16)  // [rows][d] fp16, boxes of 64 dims (128 bytes, swizzled)
      maps.v[i] = make_tmap_3d(a.v_cache, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, D, rows, 1, 2 * D, rows * D * 2, 64,
                               box_rows, 1, &ok, true);
    else
      maps.v[i] = make_tmap_3d(a.v_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, D, rows, 1, D, rows * D, C::kBW, box_rows,
                               1, &ok, C::kSwz);
  }
  if (!ok) return cudaErrorInvalidValue;
  const int64_t slots = static_cast<int64_t>(a.num_splits) * a.B * a.Hkv;
  const int grid = static_cast<int>(slots < num_sms() ? slots : num_sms());
  static std::atomic<uint32_t> next_ticket{0};
  const uint32_t ticket = next_ticket.fetch_add(1, std::memory_order_relaxed) % kTickets;
  kern<<<grid, C::kThreads, C::kBytes, s>>>(a, maps, ticket, device_status_ptr(), spin_limit_ns());
  return cudaGetLastError();
}

}  // namespace

int decode_chunk_tokens(int d) {
  return d == 256 ? DCfg<256>::kChunk : d == 128 ? DCfg<128>::kChunk : d == 64 ? DCfg<64>::kChunk : DCfg<32>::kChunk;
}

cudaError_t launch_decode_split(const DecodeArgs& a, cudaStream_t s) {
  TraceScope tr("decode_split", s);
  if (a.verify_T) {
    switch (a.d) {
      case 32: return launch_split_d<32, false, true>(a, s);
      case 64: return launch_split_d<64, false, true>(a, s);
      case 128: return launch_split_d<128, false, true>(a, s);
      case 256: return launch_split_d<256, false, true>(a, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (a.v16) {
    switch (a.d) {
      case 64: return launch_split_d<64, true>(a, s);
      case 128: return launch_split_d<128, true>(a, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.d) {
    case 32: return launch_split_d<32, false>(a, s);
    case 64: return launch_split_d<64, false>(a, s);
    case 128: return launch_split_d<128, false>(a, s);
    case 256: return launch_split_d<256, false>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_combine(const float* o_partial, const float* lse_partial, const int32_t* seqlens, int32_t B,
                                  int32_t Hq, int32_t d, int32_t num_splits, int32_t split_size, void* out,
                                  sl8_dtype out_dtype, float* lse_out, cudaStream_t s, int32_t seq_div) {
  TraceScope tr("decode_combine", s);
  const int rows = B * Hq;
  const int grid = (rows + 7) / 8;
  switch (d) {
    case 32: decode_combine_kernel<32><<<grid, 256, 0, s>>>(o_partial, lse_partial, seqlens, B, Hq, num_splits, split_size, out, out_dtype, lse_out, seq_div); break;
    case 64: decode_combine_kernel<64><<<grid, 256, 0, s>>>(o_partial, lse_partial, seqlens, B, Hq, num_splits, split_size, out, out_dtype, lse_out, seq_div); break;
    case 128: decode_combine_kernel<128><<<grid, 256, 0, s>>>(o_partial, lse_partial, seqlens, B, Hq, num_splits, split_size, out, out_dtype, lse_out, seq_div); break;
    case 256: decode_combine_kernel<256><<<grid, 256, 0, s>>>(o_partial, lse_partial, seqlens, B, Hq, num_splits, split_size, out, out_dtype, lse_out, seq_div); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_timeout_selftest(uint64_t limit_ns, cudaStream_t s) {
  timeout_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, device_status_ptr());
  return cudaGetLastError();
}

}  // namespace sl8
