// W8A8 INT8 FlashAttention prefill for sm_103a (dense and varlen, causal or not,
// GQA/MQA, head dim 64/128/256).
//
// Operation: the "SuperL8" README (github.com/jajmangold/superl8), "Attention
// kernels" table -- attn_int8_fwd (W8A8 FlashAttention-2; causal, GQA/MQA, head
// dims 32/64/128/256) and attn_varlen_fwd (ragged prefill) -- with the layouts
// of its "Quick start" section.  Per (sequence, query head):
//   S = int32(Q_i8 . K_i8^T);  x = S * s_q * s_k / sqrt(d);  causal mask (key j
//   allowed for query i iff j <= i, top-left aligned);  online softmax
//   (FlashAttention-2);  O = P . V with fp32 accumulation.
//
// GB300 design (not the pages' DP4A CUDA-core design):
//   * sm_103a has no tcgen05 kind::i8 MMA.  The int8 codes are held as bf16 (every
//     integer in [-127, 127] is exact in bf16) and QK^T runs as tcgen05 kind::f16
//     with fp32 accumulation in TMEM.  Every partial sum is an integer of
//     magnitude <= 256 * 127^2 < 2^24, so S is the exact int32 dot.
//   * P.V runs in fp16 (P in [0, 2^8], V fp16 or a bf16 V re-expressed in fp16 with a
//     per-(sequence, kv head) power-of-two scale that the epilogue undoes).
//   * Persistent CTAs walk a longest-first list of (sequence, row block, head) items
//     built on the device.  One warp issues TMA loads (Q and K as 128B-swizzled code
//     tiles from the workspace, V), one thread issues tcgen05.mma, and softmax
//     warpgroups (one thread per query row = one TMEM lane) load S from TMEM,
//     dequantise, mask, run the online softmax, write P back over S in TMEM and
//     scale O in place when the running max grows by more than 2^8.
//   * d <= 128: two 128-row Q tiles per CTA, one softmax warpgroup each, so the tensor
//     core runs one tile's MMAs while the other tile's softmax runs (TMEM: S and O of
//     both tiles, 4 x 128 columns) and each K/V tile serves 256 query rows.
//   * d = 256: one Q tile per CTA with two S buffers (TMEM: 2 x 64 + 256 columns).
//   * Every mbarrier wait is bounded in time; a timeout is recorded in the library's
//     status word and the CTA winds down with all threads leaving together.
#include <cfloat>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sl8_internal.h"

namespace sl8 {

namespace {

constexpr float kRescaleThreshold = 8.0f;  // log2 units: O is rescaled when the max grows by more
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_out2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  return pack_half2(lo, hi);
}

// Wait on an mbarrier phase with the result made uniform across the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns, DeviceStatus* st,
                                          int site) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, limit_ns, st, site));
}

// ------------------------------------------------------------------ work items
// An item is a block of consecutive 128-row Q tiles of one (sequence, query head), or
// (head pairs) one Q tile of two query heads that share a kv head.
struct Item {
  int32_t s, it, hq, hkv, L, pstart, tok0;
  int32_t part;  // key split of the item (PrefillArgs::kv_split), 0 without splits
};

// Query heads handled per (sequence, row block) entry of the work list.
__device__ __forceinline__ int item_heads(const PrefillArgs& a) { return a.head_pairs ? a.Hq / 2 : a.Hq; }

// Work item -> (sequence, item index, heads, extent).  Varlen input uses the scheduler's
// longest-first list; dense input (every sequence N long) needs no table: pair p is item
// index max_items - 1 - p / nseq of sequence p % nseq, which is the same order (a query
// chunk's items start at dense_first, the item holding its first position).  With
// head pairs, w.hq is the first of the item's two query heads.
// kSplit = false: the launch has no key splits (kv_split <= 1), known at compile time.
template <bool kSplit = false>
__device__ __forceinline__ Item decode_item(const PrefillArgs& a, int64_t item, int group) {
  Item w;
  w.part = 0;
  if (kSplit && a.kv_split > 1) {  // the parts of one item are consecutive items
    const int64_t base = item / a.kv_split;
    w.part = static_cast<int32_t>(item - base * a.kv_split);
    item = base;
  }
  const int hh = item_heads(a);
  const int64_t pair = item / hh;
  w.hq = static_cast<int32_t>(item - pair * hh) * (a.head_pairs ? 2 : 1);
  w.hkv = w.hq / group;
  if (a.varlen) {
    w.s = a.table.pair_seq[pair];
    w.it = a.table.pair_qt[pair];
    w.L = a.table.len[w.s];
    w.pstart = a.table.pstart[w.s];
    w.tok0 = a.table.tok0[w.s];
  } else {
    const int64_t level = pair / a.nseq;
    w.s = static_cast<int32_t>(pair - level * a.nseq);
    w.it = a.dense_first + a.dense_items - 1 - static_cast<int32_t>(level);
    w.L = a.N;
    w.pstart = w.s * ((a.N + kQTile - 1) / kQTile) * kPadRows;
    w.tok0 = w.s * a.N;
  }
  return w;
}
// Number of work items (pairs x query heads, or x head pairs, x key splits).
template <bool kSplit = false>
__device__ __forceinline__ int64_t count_items(const PrefillArgs& a) {
  return (a.varlen ? static_cast<int64_t>(a.table.counts[0]) : static_cast<int64_t>(a.nseq) * a.dense_items) *
         item_heads(a) * (kSplit && a.kv_split > 1 ? a.kv_split : 1);
}

// Key tiles [jb, je) a Q tile with nkv_t key tiles visits in item part w.part: all of them
// without splits, else part w.part of the item's longest range (nkv_max tiles) cut into
// kv_split equal parts (je <= jb: none).
template <bool kSplit>
__device__ __forceinline__ void part_range(const PrefillArgs& a, const Item& w, int nkv_t, int nkv_max, int& jb,
                                           int& je) {
  if (!kSplit || a.kv_split <= 1) {
    jb = 0;
    je = nkv_t;
    return;
  }
  const int per = (nkv_max + a.kv_split - 1) / a.kv_split;
  jb = w.part * per;
  je = min(jb + per, nkv_t);
  if (je < jb) je = jb;
}

// Q tile t (0, 1) of a two-tile item: its tile index in the sequence and its query head.
__device__ __forceinline__ int tile_qt(const PrefillArgs& a, const Item& w, int t) {
  return a.head_pairs ? w.it : 2 * w.it + t;
}
__device__ __forceinline__ Item tile_item(const PrefillArgs& a, const Item& w, int t) {
  Item x = w;
  if (a.head_pairs) x.hq = w.hq + t;
  return x;
}

// Key tiles of BN keys that Q tile qt (128 rows) visits; 0 if the tile is past the end.
template <int BN>
__device__ __forceinline__ int tile_nkv(int qt, int L, bool causal, int q_off) {
  // past the end, or (query chunk) wholly before its first position
  if (qt * kQTile >= L || (qt + 1) * kQTile <= q_off) return 0;
  const int kend = causal ? min(L, (qt + 1) * kQTile) : L;
  return (kend + BN - 1) / BN;
}

// ------------------------------------------------------------------ softmax step
// A softmax warp over TMEM lanes 32w..32w+31 works in the 16-lane fragment layout: its
// thread (g = lane / 4, q = lane % 4) holds query rows 32w + {g, 8 + g, 16 + g, 24 + g}
// (slot s = 2h + j: lane half h, low / high row j) and, of every 8-key group, keys 2q and
// 2q + 1.  The quad (the four q of one g) together holds whole rows, so a row's max takes
// two shuffles, and each thread needs only a quarter of the tile's K scales.
struct QuadRows {
  float m[4];      // running max, log2 units (times alpha)
  float l[4];      // this thread's share of the running sum
  float alpha[4];  // s_q log2(e) / sqrt(d)
  int row[4];      // position of the row in its sequence
};

// Slot s of this thread: the row's offset within the warp's 32 lanes.
__device__ __forceinline__ int quad_row(int s) {
  return 16 * (s >> 1) + 8 * (s & 1) + ((threadIdx.x & 31) >> 2);
}

// This thread's K scales of a key tile (tile_ks: the tile's first key): ks[2i + e] = scale
// of key 8i + 2q + e.  Read through the read-only path: every warp of the CTA reads the
// same 4 * BN bytes, so all but the first hit L1.
template <int BN>
__device__ __forceinline__ void load_ks(const float* tile_ks, float (&ks)[BN / 4]) {
  const int q = threadIdx.x & 3;
#pragma unroll
  for (int i = 0; i < BN / 8; ++i) {
    const float2 v = __ldg(reinterpret_cast<const float2*>(tile_ks + 8 * i + 2 * q));
    ks[2 * i] = v.x;
    ks[2 * i + 1] = v.y;
  }
}

// One online-softmax step over a BN-key S tile in TMEM (s_taddr: the warp's lane base and
// the tile's first column): dequantise (S * s_k[key], alpha folded into the exponent),
// mask, update each row's max m and sum l, write P (fp16) over the S columns and, when a
// row's max grew by more than 2^8, scale the warp's O rows in TMEM.  o_bar (nullable):
// barrier to wait on before touching O.  Returns false on timeout.
template <int BN, int D>
__device__ __forceinline__ bool softmax_step(uint32_t s_taddr, uint32_t o_taddr, const float (&ks)[BN / 4],
                                             bool need_mask, int key0, int L, bool causal, bool first, QuadRows& rs,
                                             uint64_t* o_bar, uint32_t o_parity, uint64_t limit_ns,
                                             DeviceStatus* st) {
  constexpr int G = BN / 8;  // 8-key groups
  const int q = threadIdx.x & 3;
  float x[2][4 * G];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int c0 = 0; c0 < BN; c0 += 64) {
      uint32_t v[32];
      tmem_ld_q8(s_taddr + (static_cast<uint32_t>(16 * h) << 16) + c0, v);
#pragma unroll
      for (int k = 0; k < 32; ++k) x[h][c0 / 2 + k] = __uint_as_float(v[k]);
    }
  }
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < G; ++i) {
    const uint64_t k2 = pk2(ks[2 * i], ks[2 * i + 1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      upk2(mul2(pk2(x[h][4 * i], x[h][4 * i + 1]), k2), x[h][4 * i], x[h][4 * i + 1]);
      upk2(mul2(pk2(x[h][4 * i + 2], x[h][4 * i + 3]), k2), x[h][4 * i + 2], x[h][4 * i + 3]);
    }
  }
  if (need_mask) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < G; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int key = key0 + 8 * i + 2 * q + (c & 1), row = rs.row[2 * h + (c >> 1)];
          if (!(key < L && (!causal || key <= row))) x[h][4 * i + c] = -INFINITY;
        }
  }
  float mx[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int h = s >> 1, j = s & 1;
    float m0 = x[h][2 * j], m1 = x[h][2 * j + 1];
#pragma unroll
    for (int i = 1; i < G; i += 2) {
      m0 = max3(m0, x[h][4 * i + 2 * j], x[h][4 * i + 2 * j + 1]);
      if (i + 1 < G) m1 = max3(m1, x[h][4 * (i + 1) + 2 * j], x[h][4 * (i + 1) + 2 * j + 1]);
    }
    mx[s] = fmaxf(m0, m1);
  }
#pragma unroll
  for (int s = 0; s < 4; ++s) mx[s] = fmaxf(mx[s], __shfl_xor_sync(0xffffffffu, mx[s], 1));
#pragma unroll
  for (int s = 0; s < 4; ++s) mx[s] = fmaxf(mx[s], __shfl_xor_sync(0xffffffffu, mx[s], 2));
  float osc[4];
  bool rescale = false;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const float m_tile = mx[s] * rs.alpha[s];
    osc[s] = 1.0f;
    if (first) {
      rs.m[s] = m_tile;
    } else if (m_tile > rs.m[s] + kRescaleThreshold) {
      osc[s] = ex2(rs.m[s] - m_tile);
      rs.l[s] *= osc[s];
      rs.m[s] = m_tile;
      rescale = true;
    }
  }
  uint64_t acc[4][2] = {{0, 0}, {0, 0}, {0, 0}, {0, 0}};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint64_t a_lo = pk2(rs.alpha[2 * h], rs.alpha[2 * h]), a_hi = pk2(rs.alpha[2 * h + 1], rs.alpha[2 * h + 1]);
    const uint64_t n_lo = pk2(-rs.m[2 * h], -rs.m[2 * h]), n_hi = pk2(-rs.m[2 * h + 1], -rs.m[2 * h + 1]);
#pragma unroll
    for (int c0 = 0; c0 < BN; c0 += 64) {
      uint32_t pw[16];
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        const int i = c0 / 8 + ii;
        float t0, t1, t2, t3;
        upk2(fma2(pk2(x[h][4 * i], x[h][4 * i + 1]), a_lo, n_lo), t0, t1);
        upk2(fma2(pk2(x[h][4 * i + 2], x[h][4 * i + 3]), a_hi, n_hi), t2, t3);
        const float e0 = ex2(t0), e1 = ex2(t1), e2 = ex2(t2), e3 = ex2(t3);
        acc[2 * h][ii & 1] = add2(acc[2 * h][ii & 1], pk2(e0, e1));
        acc[2 * h + 1][ii & 1] = add2(acc[2 * h + 1][ii & 1], pk2(e2, e3));
        pw[2 * ii] = pack_half2(e0, e1);
        pw[2 * ii + 1] = pack_half2(e2, e3);
      }
      tmem_st_p8(s_taddr + (static_cast<uint32_t>(16 * h) << 16) + c0 / 2, pw);
    }
  }
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    float s0, s1, s2, s3;
    upk2(acc[s][0], s0, s1);
    upk2(acc[s][1], s2, s3);
    rs.l[s] += (s0 + s1) + (s2 + s3);
  }
  if (__any_sync(0xffffffffu, rescale)) {
    if (o_bar && !warp_wait(o_bar, o_parity, limit_ns, st, 31)) return false;
    tc_fence_after();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint64_t sc_lo = pk2(osc[2 * h], osc[2 * h]), sc_hi = pk2(osc[2 * h + 1], osc[2 * h + 1]);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 64) {
        const uint32_t ta = o_taddr + (static_cast<uint32_t>(16 * h) << 16) + c0;
        uint32_t v[32];
        tmem_ld_q8(ta, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float a0, a1, a2, a3;
          upk2(mul2(pk2(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1])), sc_lo), a0, a1);
          upk2(mul2(pk2(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])), sc_hi), a2, a3);
          v[4 * i] = __float_as_uint(a0);
          v[4 * i + 1] = __float_as_uint(a1);
          v[4 * i + 2] = __float_as_uint(a2);
          v[4 * i + 3] = __float_as_uint(a3);
        }
        tmem_st_q8(ta, v);
      }
    }
  }
  tmem_wait_st();
  return true;
}

// End of an item: complete each row's sum across its quad and give the thread on lane r
// the max and sum of row 32w + r (the epilogue reads O one row per thread).
__device__ __forceinline__ void quad_rows_to_lane(const QuadRows& rs, float& m, float& l) {
  const int lane = threadIdx.x & 31, src = 4 * (lane & 7), slot = lane >> 3;
  m = 0.0f;
  l = 0.0f;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    float ls = rs.l[s];
    ls += __shfl_xor_sync(0xffffffffu, ls, 1);
    ls += __shfl_xor_sync(0xffffffffu, ls, 2);
    const float mv = __shfl_sync(0xffffffffu, rs.m[s], src), lv = __shfl_sync(0xffffffffu, ls, src);
    if (s == slot) {
      m = mv;
      l = lv;
    }
  }
}

// Debug: write this row's exact int32 logits (S of the tile) for keys < L.
template <int BN>
__device__ __forceinline__ void logits_step(uint32_t s_taddr, const PrefillArgs& a, const Item& w, int row_abs,
                                            int key0) {
  float x[BN];
#pragma unroll
  for (int c0 = 0; c0 < BN; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(s_taddr + c0, v);
#pragma unroll
    for (int c = 0; c < 32; ++c) x[c0 + c] = __uint_as_float(v[c]);
  }
  tmem_wait_ld();
  if (row_abs >= a.row_begin && row_abs < a.row_end && row_abs < w.L) {
    int32_t* dst = a.logits + ((static_cast<int64_t>(w.s) * a.Hq + w.hq) * (a.row_end - a.row_begin) +
                               (row_abs - a.row_begin)) * a.N;
#pragma unroll
    for (int c = 0; c < BN; ++c)
      if (key0 + c < w.L) dst[key0 + c] = __float2int_rn(x[c]);
  }
}

// Output row index of position row_abs of item w's head (dense or varlen; a query chunk's
// output holds positions q_off .. N-1).
__device__ __forceinline__ int64_t out_row(const PrefillArgs& a, const Item& w, int row_abs) {
  return a.varlen ? (static_cast<int64_t>(w.tok0) + row_abs) * a.Hq + w.hq
                  : (static_cast<int64_t>(w.s) * a.Hq + w.hq) * (a.N - a.q_off) + row_abs - a.q_off;
}

// A key-split part with no keys for this row: log-sum-exp -inf (its O is never read).
__device__ __forceinline__ void store_empty_part(const PrefillArgs& a, const Item& w, int row_abs) {
  if (row_abs < w.L && row_abs >= a.q_off) {
    const int64_t rows = static_cast<int64_t>(a.nseq) * a.Hq * (a.N - a.q_off);
    a.lse_part[w.part * rows + out_row(a, w, row_abs)] = -INFINITY;
  }
}

// Normalised output row (and LSE) from O in TMEM; with key splits, the part's normalised
// fp32 row and log-sum-exp into the partials.
template <int D, bool kSplit = false>
__device__ __forceinline__ void store_row(uint32_t o_taddr, const PrefillArgs& a, const Item& w, int row_abs, float m,
                                          float l, float v_unscale) {
  const bool row_ok = row_abs < w.L && row_abs >= a.q_off;
  if (kSplit && a.kv_split > 1) {
    const int64_t rows = static_cast<int64_t>(a.nseq) * a.Hq * (a.N - a.q_off);
    const int64_t prow = w.part * rows + out_row(a, w, row_abs);
    const float sc = v_unscale / l;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 64) {
      uint32_t v[64];
      tmem_ld32(o_taddr + c0, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld32(o_taddr + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_wait_ld();
      if (row_ok) {
        float4* dst = reinterpret_cast<float4*>(a.o_part + prow * a.d_io + c0);
#pragma unroll
        for (int c = 0; c < 64; c += 4)
          if (c0 + c < a.d_io)
            dst[c / 4] = make_float4(__uint_as_float(v[c]) * sc, __uint_as_float(v[c + 1]) * sc,
                                     __uint_as_float(v[c + 2]) * sc, __uint_as_float(v[c + 3]) * sc);
      }
    }
    if (row_ok) a.lse_part[prow] = (m + __log2f(l)) * kLn2;
    return;
  }
  const float scale = v_unscale / l;
  const bool out_f32 = a.out_dtype == SL8_F32, out_bf16 = a.out_dtype == SL8_BF16;
  // a query chunk's output holds positions q_off .. N-1
  const int64_t orow = out_row(a, w, row_abs);
  // 64 columns per TMEM round trip
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 64) {
    uint32_t v[64];
    tmem_ld32(o_taddr + c0, *reinterpret_cast<uint32_t(*)[32]>(v));
    tmem_ld32(o_taddr + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
    tmem_wait_ld();
    if (row_ok) {
      if (out_f32) {
        // rows of the output hold d_io values (32 when head dim 32 runs as 64)
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow * a.d_io + c0);
#pragma unroll
        for (int c = 0; c < 64; c += 4)
          if (c0 + c < a.d_io)
            dst[c / 4] = make_float4(__uint_as_float(v[c]) * scale, __uint_as_float(v[c + 1]) * scale,
                                   __uint_as_float(v[c + 2]) * scale, __uint_as_float(v[c + 3]) * scale);
      } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + orow * a.d_io + c0);
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          if (c0 + c >= a.d_io) break;
          uint32_t p[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            p[e] = pack_out2(__uint_as_float(v[c + 2 * e]) * scale, __uint_as_float(v[c + 2 * e + 1]) * scale,
                             out_bf16);
          dst[c / 8] = make_uint4(p[0], p[1], p[2], p[3]);
        }
      }
    }
  }
  if (row_ok && a.lse) a.lse[orow] = (m + __log2f(l)) * kLn2;
}

// Issue the D/16 MMAs of S = Q . K^T (M = 128, N = BN) into TMEM column d_col.
template <int D, int BN>
// The descriptors of a tile's K-steps differ only in the start-address field, which holds
// address / 16 and cannot overflow its 14 bits for a shared-memory address: each is the
// first one plus a constant, so the issuing warp spends one add per descriptor.
__device__ __forceinline__ void issue_qk(uint32_t d_col, uint32_t qaddr, uint32_t kaddr) {
  constexpr uint32_t idesc = idesc_f16(kQTile, BN, true, false, false);
  const uint64_t da0 = desc_sw128(qaddr, 16, 1024), db0 = desc_sw128(kaddr, 16, 1024);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint64_t da = da0 + static_cast<uint64_t>(((k / 4) * (kQTile * 128) + (k % 4) * 32) >> 4);
    const uint64_t db = db0 + static_cast<uint64_t>(((k / 4) * (BN * 128) + (k % 4) * 32) >> 4);
    mma_ss(d_col, da, db, idesc, k > 0 ? 1u : 0u);
  }
}

// Issue the BN/16 MMAs of O (+)= P . V (M = 128, N = D), P fp16 in TMEM at p_col.
template <int D, int BN>
__device__ __forceinline__ void issue_pv(uint32_t o_col, uint32_t p_col, uint32_t vaddr, bool accumulate) {
  constexpr uint32_t idesc = idesc_f16(kQTile, D, false, false, true);  // fp16 P x fp16 V (MN-major)
  const uint64_t db0 = desc_sw128(vaddr, BN * 128, 1024);
#pragma unroll
  for (int k = 0; k < BN / 16; ++k)
    mma_ts(o_col, p_col + k * 8, db0 + static_cast<uint64_t>(k * (2048 >> 4)), idesc, (accumulate || k > 0) ? 1u : 0u);
}

__device__ __forceinline__ void load_q_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int boxes, int row,
                                            int head) {
  for (int b = 0; b < boxes; ++b) tma_load_3d(dst + b * (kQTile * 128), map, bar, b * 64, row, head);
}

// K and V tiles j of item w into one pipeline stage (V waits for its stage to drain).
template <int BN>
__device__ __forceinline__ void load_kv_tile(uint8_t* kdst, uint8_t* vdst, const CUtensorMap* map_k,
                                             const CUtensorMap* map_v, uint64_t* kbar, uint64_t* vbar, int boxes,
                                             const PrefillArgs& a, const Item& w, int j, uint32_t bytes,
                                             uint64_t* v_empty, uint32_t v_parity, bool wait_v, uint64_t limit_ns,
                                             DeviceStatus* st, bool* ok) {
  mbar_arrive_expect_tx(kbar, bytes);
  for (int b = 0; b < boxes; ++b) tma_load_3d(kdst + b * (BN * 128), map_k, kbar, b * 64, w.pstart + j * BN, w.hkv);
  if (wait_v && !mbar_wait(v_empty, v_parity, limit_ns, st, 12)) {
    *ok = false;
    return;
  }
  mbar_arrive_expect_tx(vbar, bytes);
  for (int b = 0; b < boxes; ++b) {
    if (a.v16)
      tma_load_3d(vdst + b * (BN * 128), map_v, vbar, b * 64, w.pstart + j * BN, w.hkv);
    else if (a.varlen)
      tma_load_3d(vdst + b * (BN * 128), map_v, vbar, b * 64, w.hkv, w.tok0 + j * BN);
    else
      tma_load_3d(vdst + b * (BN * 128), map_v, vbar, b * 64, j * BN, w.s * a.Hkv + w.hkv);
  }
}

// ==================================================================== d <= 128: two Q tiles per CTA
template <int D>
struct PairCfg {
  static constexpr int BN = 128;
  static constexpr int kBoxes = D / 64;
  static constexpr int kQBytes = kQTile * D * 2;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kStages = 2;
  static constexpr int kQOff = 0;                                   // 2 Q tiles
  static constexpr int kKOff = kQOff + 2 * kQBytes;
  static constexpr int kVOff = kKOff + kStages * kKVBytes;
  static constexpr int kBarOff = kVOff + kStages * kKVBytes;
  static constexpr int kUsed = kBarOff + 256 + 1024;
  // at least 116 KB so that a second CTA never shares the SM (each holds all 512 TMEM columns)
  static constexpr int kSmemBytes = kUsed > 118784 ? kUsed : 118784;
  // warps 0-3 / 4-7: softmax of tile 0 / 1; 8: TMA; 9: MMA; 10-11 idle.  Launched at 168
  // registers per thread (384 x 168 = 64512); then the TMA/MMA warpgroup moves to 104 and
  // the softmax warpgroups to 200: 8 x 32 x 200 + 4 x 32 x 104 = 64512, and per SMSP
  // (warps k, k+4, k+8) 200 + 200 + 104 = 504 <= 512 registers per lane slot.  The
  // attention instantiations compile without spills at this split; it ran about 5 %
  // faster than 216 / 72 and 208 / 88.
  static constexpr int kThreads = 384;
  static constexpr int kRegsSoftmax = 200;
  static constexpr int kRegsOther = 104;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(2 * (BN + D) <= 512, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "smem budget");
};

// Work items are claimed at run time (a counter in the workspace, after a first wave of
// blockIdx.x): the TMA warp claims the next item when it is about to load it and hands
// the index to the MMA warp and the softmax warps through a small ring.  Dense items are
// numbered longest first, so the claims approximate longest-processing-time scheduling.
constexpr int kItemRing = 4;

struct PairBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t item_full[kItemRing], item_empty[kItemRing];
  uint64_t drain;
  int32_t item_idx[kItemRing];  // -1: no more items
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(PairBars) <= 256, "pair kernel barrier block");

template <int D, bool kLogits, bool kSplit>
__global__ void __launch_bounds__(PairCfg<D>::kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v, const PrefillArgs a, DeviceStatus* st,
                        uint64_t limit_ns) {
  using C = PairCfg<D>;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairBars& bars = *reinterpret_cast<PairBars*>(smem + C::kBarOff);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const bool causal = kLogits ? false : a.causal;
  const int group = a.Hq / a.Hkv;
  const int64_t n_items = count_items<kSplit>(a);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 1);
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 4);  // one arrival per softmax warp
      mbar_init(&bars.o_done[i], 1);
    }
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(&bars.item_full[i], 1);
      mbar_init(&bars.item_empty[i], 9);  // the MMA warp and the 8 softmax warps
    }
    mbar_init(&bars.drain, 1);
    bars.abort = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars.tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  // launched as a programmatic dependent of the quantiser: the set-up above overlaps
  // its tail; everything below reads what it wrote
  grid_dependency_wait();
  const uint32_t tbase = bars.tmem_base;
  volatile int* abort_flag = &bars.abort;
  static_assert(8 * 32 * C::kRegsSoftmax + 4 * 32 * C::kRegsOther <= C::kThreads * 168, "register split");

  if (warp >= 8) {
    // warps 8-11: TMA producer, MMA issuer, two idle warps
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsOther));
    if (warp == 8 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      uint32_t g = 0;
      bool ok = true;
      for (uint32_t it = 0;; ++it) {
        // claim the next item and publish it (-1 ends every consumer's loop)
        const uint32_t slot = it % kItemRing;
        if (it >= kItemRing) ok = ok && mbar_wait(&bars.item_empty[slot], (it / kItemRing - 1) & 1, limit_ns, st, 13);
        int64_t item = it == 0 ? blockIdx.x : gridDim.x + atomicAdd(a.table.counts + 2, 1);
        if (item >= n_items || !ok || *abort_flag) item = -1;
        bars.item_idx[slot] = static_cast<int32_t>(item);
        mbar_arrive(&bars.item_full[slot]);
        if (item < 0) break;
        const Item w = decode_item<kSplit>(a, item, group);
        const int nkv0 = tile_nkv<BN>(tile_qt(a, w, 0), w.L, causal, a.q_off);
        const int nkv1 = tile_nkv<BN>(tile_qt(a, w, 1), w.L, causal, a.q_off);
        int jb, je0, je1;
        part_range<kSplit>(a, w, nkv0, max(nkv0, nkv1), jb, je0);
        part_range<kSplit>(a, w, nkv1, max(nkv0, nkv1), jb, je1);
        const int je = max(je0, je1);
        // both Q tiles are always loaded (a tile past the end reads rows no one uses)
        for (int t = 0; t < 2 && ok; ++t) {
          if (it >= 1) ok = mbar_wait(&bars.q_empty[t], (it - 1) & 1, limit_ns, st, 10);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars.q_full[t], C::kQBytes);
          load_q_tile(smem + C::kQOff + t * C::kQBytes, &map_q, &bars.q_full[t], C::kBoxes,
                      w.pstart + tile_qt(a, w, t) * kQTile, tile_item(a, w, t).hq);
        }
        for (int j = jb; j < je && ok; ++j, ++g) {
          const uint32_t stg = g % C::kStages, n = g / C::kStages;
          if (g >= C::kStages) ok = mbar_wait(&bars.k_empty[stg], (n - 1) & 1, limit_ns, st, 11);
          if (!ok || *abort_flag) break;
          load_kv_tile<BN>(smem + C::kKOff + stg * C::kKVBytes, smem + C::kVOff + stg * C::kKVBytes, &map_k, &map_v,
                           &bars.k_full[stg], &bars.v_full[stg], C::kBoxes, a, w, j, C::kKVBytes, &bars.v_empty[stg],
                           (n - 1) & 1, g >= C::kStages, limit_ns, st, &ok);
        }
      }
      if (!ok) *abort_flag = 1;
    } else if (warp == 9) {
      // ---------------------------------------------------------- MMA issuer (whole warp, one lane issues)
      // Per key tile j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1): while one tile's softmax
      // runs, the tensor core works on the other tile.
      uint32_t g = 0, np[2] = {0, 0};
      bool ok = true, issued = false;
      for (uint32_t it = 0; ok && !*abort_flag; ++it) {
        const uint32_t slot = it % kItemRing;
        ok = warp_wait(&bars.item_full[slot], (it / kItemRing) & 1, limit_ns, st, 25);
        if (!ok) break;
        const int32_t item = bars.item_idx[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.item_empty[slot]);
        if (item < 0) break;
        const Item w = decode_item<kSplit>(a, item, group);
        // key tiles of each Q tile in this item (part), counted from the part's first, jb
        const int nkv0 = tile_nkv<BN>(tile_qt(a, w, 0), w.L, causal, a.q_off);
        const int nkv1 = tile_nkv<BN>(tile_qt(a, w, 1), w.L, causal, a.q_off);
        int jb, je0, je1;
        part_range<kSplit>(a, w, nkv0, max(nkv0, nkv1), jb, je0);
        part_range<kSplit>(a, w, nkv1, max(nkv0, nkv1), jb, je1);
        const int nkv_t[2] = {je0 - jb, je1 - jb};
        const int nkv = max(nkv_t[0], nkv_t[1]);
        ok = warp_wait(&bars.q_full[0], it & 1, limit_ns, st, 20) &&
             warp_wait(&bars.q_full[1], it & 1, limit_ns, st, 20);
        if (ok && (!kSplit || nkv > 0)) ok = warp_wait(&bars.k_full[g % C::kStages], (g / C::kStages) & 1, limit_ns, st, 21);
        if (!ok) break;
        tc_fence_after();
        if (kSplit && nkv == 0) {
          // a key split with no key tiles for either Q tile: nothing to compute or load
          mma_commit(&bars.q_empty[0]);
          mma_commit(&bars.q_empty[1]);
          issued = true;
          continue;
        }
        {
          const uint32_t kaddr = smem_u32(smem + C::kKOff + (g % C::kStages) * C::kKVBytes);
          for (int t = 0; t < 2; ++t) {
            if (nkv_t[t] > 0) {
              issue_qk<D, BN>(tbase + t * 256, smem_u32(smem + C::kQOff + t * C::kQBytes), kaddr);
              mma_commit(&bars.s_full[t]);
            }
            if (nkv_t[t] <= 1) mma_commit(&bars.q_empty[t]);
          }
          issued = true;
          mma_commit(&bars.k_empty[g % C::kStages]);
        }
        for (int j = 0; j < nkv && ok; ++j) {
          const uint32_t gj = g + j, gn = g + j + 1;
          bool v_ready = false, k_ready = false;
          for (int t = 0; t < 2 && ok; ++t) {
            if (j >= nkv_t[t]) continue;
            ok = warp_wait(&bars.p_full[t], np[t] & 1, limit_ns, st, 22);
            ++np[t];
            if (ok && !v_ready)
              ok = warp_wait(&bars.v_full[gj % C::kStages], (gj / C::kStages) & 1, limit_ns, st, 23);
            if (!ok) break;
            v_ready = true;
            tc_fence_after();
            issue_pv<D, BN>(tbase + t * 256 + 128, tbase + t * 256,
                            smem_u32(smem + C::kVOff + (gj % C::kStages) * C::kKVBytes), j > 0);
            if (j == nkv_t[t] - 1) mma_commit(&bars.o_done[t]);
            if (j + 1 < nkv_t[t]) {
              if (!k_ready) {
                ok = warp_wait(&bars.k_full[gn % C::kStages], (gn / C::kStages) & 1, limit_ns, st, 21);
                if (!ok) break;
                k_ready = true;
                tc_fence_after();
              }
              issue_qk<D, BN>(tbase + t * 256, smem_u32(smem + C::kQOff + t * C::kQBytes),
                              smem_u32(smem + C::kKOff + (gn % C::kStages) * C::kKVBytes));
              mma_commit(&bars.s_full[t]);
              if (j + 1 == nkv_t[t] - 1) mma_commit(&bars.q_empty[t]);
            }
          }
          if (!ok) break;
          mma_commit(&bars.v_empty[gj % C::kStages]);
          if (k_ready) mma_commit(&bars.k_empty[gn % C::kStages]);
        }
        g += nkv;
      }
      if (!ok) *abort_flag = 1;
      if (issued) {
        mma_commit(&bars.drain);
        warp_wait(&bars.drain, 0, limit_ns, st, 24);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsSoftmax));
    const int t = warp / 4;                       // Q tile of this warpgroup
    const int r = threadIdx.x - t * 128;          // TMEM lane: the row this thread stores
    const int wrow = (warp & 3) * 32;             // the warp's first row in the tile
    const uint32_t lane_base = static_cast<uint32_t>(wrow) << 16;
    const uint32_t s_taddr = tbase + lane_base + t * 256;
    const uint32_t o_taddr = s_taddr + 128;
    const float qk_scale = kLog2e * rsqrtf(static_cast<float>(a.d_io));  // the true head dim (32 runs as 64)
    uint32_t ns = 0, no = 0;   // S tiles consumed, items finished (this tile)
    bool bad = false;
    // item index it from the ring (false on timeout)
    auto fetch = [&](uint32_t it, int32_t& item) -> bool {
      const uint32_t slot = it % kItemRing;
      if (!warp_wait(&bars.item_full[slot], (it / kItemRing) & 1, limit_ns, st, 35)) return false;
      item = bars.item_idx[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.item_empty[slot]);
      return true;
    };
    // The next item is read from the ring, and its q scales and V exponent loaded, before
    // this item's epilogue, so that their latency overlaps the epilogue.
    int32_t next_item = -1;
    bool have_next = false, have_scales = false;
    float qs_next[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int ve_next = 0;
    for (uint32_t it = 0; !bad; ++it) {
      int32_t item = next_item;
      if (!have_next && !fetch(it, item)) {
        bad = true;
        break;
      }
      have_next = false;
      if (item < 0) break;
      const Item w = tile_item(a, decode_item<kSplit>(a, item, group), t);  // this warpgroup's Q tile
      const int qt = tile_qt(a, w, t);
      const int nkv_full = tile_nkv<BN>(qt, w.L, causal, a.q_off);
      const bool scales_ready = have_scales;
      have_scales = false;
      if (nkv_full == 0) continue;  // this tile lies past the sequence's end (or before a chunk)
      const int row_abs = qt * kQTile + r;
      int jb, je;
      part_range<kSplit>(a, w, nkv_full, max(nkv_full, tile_nkv<BN>(tile_qt(a, w, 1 - t), w.L, causal, a.q_off)), jb, je);
      if (je <= jb) {  // a key split that reaches none of this tile's keys: an empty part
        store_empty_part(a, w, row_abs);
        continue;
      }
      QuadRows rs;
      const float* qs = a.q_scales + static_cast<int64_t>(w.hq) * a.t_pad_max + w.pstart + qt * kQTile + wrow;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        rs.m[s] = -INFINITY;
        rs.l[s] = 0.0f;
        rs.alpha[s] = fmaxf((scales_ready ? qs_next[s] : qs[quad_row(s)]) * qk_scale, FLT_MIN);
        rs.row[s] = qt * kQTile + wrow + quad_row(s);
      }
      const int ve = scales_ready ? ve_next : (a.v_exp ? a.v_exp[static_cast<int64_t>(w.s) * a.Hkv + w.hkv] : 0);
      const float v_unscale = __int_as_float((127 + ve) << 23);
      const float* ksrc = a.k_scales + static_cast<int64_t>(w.hkv) * a.t_pad_max + w.pstart;
      for (int j = jb; j < je; ++j, ++ns) {
        if (*abort_flag) {
          bad = true;
          break;
        }
        float ks[BN / 4];
        load_ks<BN>(ksrc + j * BN, ks);
        if (!warp_wait(&bars.s_full[t], ns & 1, limit_ns, st, 30)) {
          bad = true;
          break;
        }
        tc_fence_after();
        const int key0 = j * BN;
        if constexpr (kLogits) {
          logits_step<BN>(s_taddr, a, w, row_abs, key0);
        } else {
          const bool need_mask = (causal && key0 + BN - 1 > qt * kQTile) || (key0 + BN > w.L);
          // O_t is safe to touch: S_t(j) was issued after PV_t(j-1), and its commit covers it
          if (!softmax_step<BN, D>(s_taddr, o_taddr, ks, need_mask, key0, w.L, causal, j == jb, rs, nullptr, 0,
                                   limit_ns, st)) {
            bad = true;
            break;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[t]);
      }
      if (bad || *abort_flag) {
        bad = true;
        break;
      }
      // only when the next item is already published: never wait for it here
      const uint32_t nslot = (it + 1) % kItemRing;
      if (__all_sync(0xffffffffu, mbar_try_wait(&bars.item_full[nslot], ((it + 1) / kItemRing) & 1))) {
        if (!fetch(it + 1, next_item)) {
          bad = true;
          break;
        }
        have_next = true;
      }
      if (have_next && next_item >= 0) {
        const Item wn = tile_item(a, decode_item<kSplit>(a, next_item, group), t);
        const int qtn = tile_qt(a, wn, t);
        if (tile_nkv<BN>(qtn, wn.L, causal, a.q_off) > 0) {
          const float* qsn = a.q_scales + static_cast<int64_t>(wn.hq) * a.t_pad_max + wn.pstart + qtn * kQTile + wrow;
#pragma unroll
          for (int s = 0; s < 4; ++s) qs_next[s] = qsn[quad_row(s)];
          ve_next = a.v_exp ? a.v_exp[static_cast<int64_t>(wn.s) * a.Hkv + wn.hkv] : 0;
          have_scales = true;
        }
      }
      if (!warp_wait(&bars.o_done[t], no & 1, limit_ns, st, 32)) {
        bad = true;
      } else {
        tc_fence_after();
        if constexpr (!kLogits) {
          float m, l;
          quad_rows_to_lane(rs, m, l);
          store_row<D, kSplit>(o_taddr, a, w, row_abs, m, l, v_unscale);
        }
      }
      ++no;
    }
    if (bad) *abort_flag = 1;
  }
  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tbase, C::kTmemCols);
}

// ==================================================================== d = 256: one Q tile per CTA
// Item k of this CTA.  Items are numbered longest first; CTA c takes item c of every even
// round of gridDim.x items and item gridDim.x - 1 - c of every odd round ("snake" order),
// so that each CTA's long and short items even out (plain round robin gives CTA 0 the
// longest item of every round).  Past the last item, every later k is past it too.
__device__ __forceinline__ int64_t snake_item(int64_t k) {
  const int64_t base = k * gridDim.x;
  return (k & 1) ? base + gridDim.x - 1 - blockIdx.x : base + blockIdx.x;
}

template <int D>
struct SingleCfg {
  static constexpr int BN = 64;
  static constexpr int kBoxes = D / 64;
  static constexpr int kQBytes = kQTile * D * 2;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kStages = 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + kStages * kKVBytes;
  static constexpr int kBarOff = kVOff + kStages * kKVBytes;
  static constexpr int kUsed = kBarOff + 256 + 1024;
  static constexpr int kSmemBytes = kUsed > 118784 ? kUsed : 118784;
  static constexpr int kThreads = 192;  // warps 0-3 softmax; 4 TMA; 5 MMA
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 2 * BN;
  static_assert(kOCol + D <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "smem budget");
};

struct SingleBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <int D, bool kLogits>
__global__ void __launch_bounds__(SingleCfg<D>::kThreads, 1)
    prefill_single_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                          const __grid_constant__ CUtensorMap map_v, const PrefillArgs a, DeviceStatus* st,
                          uint64_t limit_ns) {
  using C = SingleCfg<D>;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SingleBars& bars = *reinterpret_cast<SingleBars*>(smem + C::kBarOff);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const bool causal = kLogits ? false : a.causal;
  const int group = a.Hq / a.Hkv;
  const int64_t n_items = count_items(a);

  if (threadIdx.x == 0) {
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 4);  // one arrival per softmax warp
      mbar_init(&bars.o_done[i], 1);
    }
    mbar_init(&bars.drain, 1);
    bars.abort = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars.tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  // launched as a programmatic dependent of the quantiser: the set-up above overlaps
  // its tail; everything below reads what it wrote
  grid_dependency_wait();
  const uint32_t tbase = bars.tmem_base;
  volatile int* abort_flag = &bars.abort;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      uint32_t g = 0, it = 0;
      bool ok = true;
      for (int64_t item = snake_item(0); item < n_items && ok && !*abort_flag; ++it, item = snake_item(it)) {
        const Item w = decode_item(a, item, group);
        const int nkv = tile_nkv<BN>(w.it, w.L, causal, a.q_off);
        if (it >= 1) ok = mbar_wait(&bars.q_empty, (it - 1) & 1, limit_ns, st, 10);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars.q_full, C::kQBytes);
        load_q_tile(smem + C::kQOff, &map_q, &bars.q_full, C::kBoxes, w.pstart + w.it * kQTile, w.hq);
        for (int j = 0; j < nkv && ok; ++j, ++g) {
          const uint32_t stg = g % C::kStages, n = g / C::kStages;
          if (g >= C::kStages) ok = mbar_wait(&bars.k_empty[stg], (n - 1) & 1, limit_ns, st, 11);
          if (!ok || *abort_flag) break;
          load_kv_tile<BN>(smem + C::kKOff + stg * C::kKVBytes, smem + C::kVOff + stg * C::kKVBytes, &map_k, &map_v,
                           &bars.k_full[stg], &bars.v_full[stg], C::kBoxes, a, w, j, C::kKVBytes, &bars.v_empty[stg],
                           (n - 1) & 1, g >= C::kStages, limit_ns, st, &ok);
        }
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // S tiles run one ahead of P.V: S_{g+1} is issued before PV_g (two S buffers).  The
    // whole warp runs this loop; one lane issues.
    {
      int64_t item_s = snake_item(0), item_p = item_s;
      uint32_t it_s = 0, it_p = 0, gs = 0, gp = 0;
      int j_s = 0, j_p = 0;
      int nkv_s = 0, nkv_p = 0;
      if (item_s < n_items) {
        const Item ws = decode_item(a, item_s, group);
        nkv_s = tile_nkv<BN>(ws.it, ws.L, causal, a.q_off);
        nkv_p = nkv_s;
      }
      bool ok = true, issued = false;
      while (ok && item_p < n_items && !*abort_flag) {
        while (ok && item_s < n_items && gs <= gp + 1) {
          if (j_s == 0) ok = warp_wait(&bars.q_full, it_s & 1, limit_ns, st, 20);
          const uint32_t stg = gs % C::kStages;
          if (ok) ok = warp_wait(&bars.k_full[stg], (gs / C::kStages) & 1, limit_ns, st, 21);
          if (!ok) break;
          tc_fence_after();
          issue_qk<D, BN>(tbase + (gs & 1) * BN, smem_u32(smem + C::kQOff),
                          smem_u32(smem + C::kKOff + stg * C::kKVBytes));
          issued = true;
          mma_commit(&bars.s_full[gs & 1]);
          mma_commit(&bars.k_empty[stg]);
          ++gs;
          if (++j_s == nkv_s) {
            mma_commit(&bars.q_empty);
            j_s = 0;
            ++it_s;
            item_s = snake_item(it_s);
            if (item_s < n_items) {
              const Item ws = decode_item(a, item_s, group);
              nkv_s = tile_nkv<BN>(ws.it, ws.L, causal, a.q_off);
            }
          }
        }
        if (!ok) break;
        ok = warp_wait(&bars.p_full[gp & 1], (gp >> 1) & 1, limit_ns, st, 22);
        const uint32_t stg = gp % C::kStages;
        if (ok) ok = warp_wait(&bars.v_full[stg], (gp / C::kStages) & 1, limit_ns, st, 23);
        if (!ok) break;
        tc_fence_after();
        issue_pv<D, BN>(tbase + C::kOCol, tbase + (gp & 1) * BN, smem_u32(smem + C::kVOff + stg * C::kKVBytes),
                        j_p > 0);
        mma_commit(&bars.o_done[gp & 1]);
        mma_commit(&bars.v_empty[stg]);
        ++gp;
        if (++j_p == nkv_p) {
          j_p = 0;
          item_p = snake_item(++it_p);
          if (item_p < n_items) {
            const Item wp = decode_item(a, item_p, group);
            nkv_p = tile_nkv<BN>(wp.it, wp.L, causal, a.q_off);
          }
        }
      }
      if (!ok) *abort_flag = 1;
      if (issued) {
        mma_commit(&bars.drain);
        warp_wait(&bars.drain, 0, limit_ns, st, 24);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroup (warps 0-3)
    const int r = threadIdx.x;                    // TMEM lane: the row this thread stores
    const int wrow = warp * 32;
    const uint32_t lane_base = static_cast<uint32_t>(wrow) << 16;
    const float qk_scale = kLog2e * rsqrtf(static_cast<float>(a.d_io));  // the true head dim (32 runs as 64)
    int64_t k_item = 0, item = snake_item(0);
    Item w{};
    uint32_t g = 0;
    // q scales of this thread's four softmax rows (the quad layout) for the next item
    float qs_next[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int ve_next = 0;
    auto load_qs = [&](const Item& x) {
      const float* qs = a.q_scales + static_cast<int64_t>(x.hq) * a.t_pad_max + x.pstart + x.it * kQTile;
#pragma unroll
      for (int s = 0; s < 4; ++s) qs_next[s] = qs[wrow + quad_row(s)];
    };
    if (item < n_items) {
      w = decode_item(a, item, group);
      load_qs(w);
      if (a.v_exp) ve_next = a.v_exp[static_cast<int64_t>(w.s) * a.Hkv + w.hkv];
    }
    bool bad = false;
    while (item < n_items) {
      const int nkv = tile_nkv<BN>(w.it, w.L, causal, a.q_off);
      const int row_abs = w.it * kQTile + r;
      QuadRows rs;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        rs.m[s] = -INFINITY;
        rs.l[s] = 0.0f;
        rs.alpha[s] = fmaxf(qs_next[s] * qk_scale, FLT_MIN);
        rs.row[s] = w.it * kQTile + wrow + quad_row(s);
      }
      const float v_unscale = __int_as_float((127 + ve_next) << 23);
      const int64_t item_n = snake_item(k_item + 1);
      Item wn{};
      if (item_n < n_items) wn = decode_item(a, item_n, group);
      const float* ksrc = a.k_scales + static_cast<int64_t>(w.hkv) * a.t_pad_max + w.pstart;
      for (int j = 0; j < nkv; ++j, ++g) {
        const uint32_t buf = g & 1;
        if (j + 1 == nkv && item_n < n_items) {
          load_qs(wn);
          if (a.v_exp) ve_next = a.v_exp[static_cast<int64_t>(wn.s) * a.Hkv + wn.hkv];
        }
        if (*abort_flag) {
          bad = true;
          break;
        }
        float ks[BN / 4];
        load_ks<BN>(ksrc + j * BN, ks);
        if (!warp_wait(&bars.s_full[buf], (g >> 1) & 1, limit_ns, st, 30)) {
          bad = true;
          break;
        }
        tc_fence_after();
        const uint32_t s_taddr = tbase + lane_base + buf * BN;
        const int key0 = j * BN;
        if constexpr (kLogits) {
          logits_step<BN>(s_taddr, a, w, row_abs, key0);
        } else {
          const bool need_mask = (causal && key0 + BN - 1 > w.it * kQTile) || (key0 + BN > w.L);
          // here S_g was issued after PV_{g-2} only: wait for PV_{g-1} before touching O
          const uint32_t gprev = g - 1;
          if (!softmax_step<BN, D>(s_taddr, tbase + lane_base + C::kOCol, ks, need_mask, key0, w.L, causal, j == 0,
                                   rs, &bars.o_done[gprev & 1], (gprev >> 1) & 1, limit_ns, st)) {
            bad = true;
            break;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[buf]);
      }
      if (bad || *abort_flag) {
        bad = true;
        break;
      }
      const uint32_t glast = g - 1;
      if (!warp_wait(&bars.o_done[glast & 1], (glast >> 1) & 1, limit_ns, st, 32)) {
        bad = true;
      } else {
        tc_fence_after();
        if constexpr (!kLogits) {
          float m, l;
          quad_rows_to_lane(rs, m, l);
          store_row<D>(tbase + lane_base + C::kOCol, a, w, row_abs, m, l, v_unscale);
        }
      }
      item = item_n;
      ++k_item;
      w = wn;
    }
    if (bad) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tbase, C::kTmemCols);
}

// ------------------------------------------------------------------ host side
template <int BN>
static bool make_maps(const PrefillArgs& a, int D, CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mv) {
  bool ok = true;
  *mq = make_tmap_3d(a.q_codes, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, a.t_pad_max, a.Hq, D * 2ull,
                     a.t_pad_max * D * 2ull, 64, kQTile, 1, &ok);
  *mk = make_tmap_3d(a.k_codes, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, a.t_pad_max, a.Hkv, D * 2ull,
                     a.t_pad_max * D * 2ull, 64, BN, 1, &ok);
  // P.V runs in fp16: V is either the caller's fp16 tensor or the fp16 copy of a bf16 V
  // in the padded workspace layout (same coordinates as K)
  if (a.v16)
    *mv = make_tmap_3d(a.v16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, D, a.t_pad_max, a.Hkv, D * 2ull, a.t_pad_max * D * 2ull,
                       64, BN, 1, &ok);
  else if (a.varlen)  // [T, Hkv, d]: dims (d, Hkv, T)
    *mv = make_tmap_3d(a.v, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, D, a.Hkv, a.total_tokens, D * 2ull,
                       static_cast<uint64_t>(a.Hkv) * D * 2ull, 64, 1, BN, &ok);
  else  // [nseq, Hkv, N, d]: dims (d, N, nseq*Hkv)
    *mv = make_tmap_3d(a.v, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, D, a.N, static_cast<uint64_t>(a.nseq) * a.Hkv, D * 2ull,
                       static_cast<uint64_t>(a.N) * D * 2ull, 64, BN, 1, &ok);
  return ok;
}

template <int D, bool kLogits, bool kSplit = false>
static cudaError_t launch_pair(const PrefillArgs& a, cudaStream_t s) {
  using C = PairCfg<D>;
  CUtensorMap mq, mk, mv;
  if (!make_maps<C::BN>(a, D, &mq, &mk, &mv)) return cudaErrorInvalidValue;
  auto kern = prefill_pair_kernel<D, kLogits, kSplit>;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t max_items = a.max_pairs * a.Hq * (kSplit ? a.kv_split : 1);
  const int grid = static_cast<int>(max_items < num_sms() ? max_items : num_sms());
  if (grid <= 0) return cudaSuccess;
  TraceScope tr(kLogits ? "prefill_logits" : "prefill_attn", s);
  return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, mq, mk, mv, a, device_status_ptr(),
                    spin_limit_ns());
}

template <int D, bool kLogits>
static cudaError_t launch_single(const PrefillArgs& a, cudaStream_t s) {
  using C = SingleCfg<D>;
  CUtensorMap mq, mk, mv;
  if (!make_maps<C::BN>(a, D, &mq, &mk, &mv)) return cudaErrorInvalidValue;
  auto kern = prefill_single_kernel<D, kLogits>;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t max_items = a.max_pairs * a.Hq;
  const int grid = static_cast<int>(max_items < num_sms() ? max_items : num_sms());
  if (grid <= 0) return cudaSuccess;
  TraceScope tr(kLogits ? "prefill_logits" : "prefill_attn", s);
  return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, mq, mk, mv, a, device_status_ptr(),
                    spin_limit_ns());
}

}  // namespace

// Merge of the key-split partials of a query chunk: one warp per output row; weights
// e^(lse_p - max lse) over the parts that saw a key (lse -inf parts are skipped).  Every
// part's LSE and row slice are loaded before any is used (at most kMaxKeySplit parts).
template <int EPL>
static __global__ void __launch_bounds__(256) prefill_combine_kernel(const float* __restrict__ o_part,
                                                              const float* __restrict__ lse_part, int64_t rows,
                                                              int d_io, int S, void* __restrict__ out,
                                                              sl8_dtype out_dtype, float* __restrict__ lse) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  float lp[kMaxKeySplit], x[kMaxKeySplit][EPL];
#pragma unroll
  for (int p = 0; p < kMaxKeySplit; ++p) {
    lp[p] = p < S ? lse_part[p * rows + row] : -INFINITY;
#pragma unroll
    for (int e = 0; e < EPL; ++e) x[p][e] = p < S ? o_part[(p * rows + row) * d_io + lane * EPL + e] : 0.0f;
  }
  float M = -INFINITY;
#pragma unroll
  for (int p = 0; p < kMaxKeySplit; ++p) M = fmaxf(M, lp[p]);
  float acc[EPL] = {};
  float wsum = 0.0f;
#pragma unroll
  for (int p = 0; p < kMaxKeySplit; ++p) {
    if (lp[p] == -INFINITY) continue;
    const float w = expf(lp[p] - M);
    wsum += w;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, x[p][e], acc[e]);
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
  const int64_t o = row * d_io + lane * EPL;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const float y = acc[e] * inv;
    if (out_dtype == SL8_F32) static_cast<float*>(out)[o + e] = y;
    else if (out_dtype == SL8_BF16) static_cast<__nv_bfloat16*>(out)[o + e] = __float2bfloat16_rn(y);
    else static_cast<__half*>(out)[o + e] = __float2half_rn(y);
  }
  if (lse && lane == 0) lse[row] = wsum > 0.0f ? M + logf(wsum) : -INFINITY;
}

cudaError_t launch_prefill_combine(const float* o_part, const float* lse_part, int64_t rows, int32_t d_io,
                                   int32_t kv_split, void* out, sl8_dtype out_dtype, float* lse, cudaStream_t s) {
  TraceScope tr("prefill_combine", s);
  if (rows <= 0) return cudaSuccess;
  if (kv_split > kMaxKeySplit) return cudaErrorInvalidValue;
  const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
  switch (d_io) {
    case 32: prefill_combine_kernel<1><<<grid, 256, 0, s>>>(o_part, lse_part, rows, d_io, kv_split, out, out_dtype, lse); break;
    case 64: prefill_combine_kernel<2><<<grid, 256, 0, s>>>(o_part, lse_part, rows, d_io, kv_split, out, out_dtype, lse); break;
    case 128: prefill_combine_kernel<4><<<grid, 256, 0, s>>>(o_part, lse_part, rows, d_io, kv_split, out, out_dtype, lse); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

bool prefill_head_pairs(int d, int group) { return d <= 128 && group % 2 == 0; }
int prefill_item_rows(int d, int group) { return d <= 128 && !prefill_head_pairs(d, group) ? 2 * kQTile : kQTile; }

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  const bool logits = a.logits != nullptr;
  switch (a.d) {
    // key splits (query chunks only) have an instantiation of their own, so that the
    // unsplit kernel compiles without the split bookkeeping
    case 64: return logits ? launch_pair<64, true>(a, s)
                           : (a.kv_split > 1 ? launch_pair<64, false, true>(a, s) : launch_pair<64, false>(a, s));
    case 128: return logits ? launch_pair<128, true>(a, s)
                            : (a.kv_split > 1 ? launch_pair<128, false, true>(a, s) : launch_pair<128, false>(a, s));
    case 256: return logits ? launch_single<256, true>(a, s) : launch_single<256, false>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sl8
