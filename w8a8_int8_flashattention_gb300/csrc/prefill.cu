// W8A8 INT8 FlashAttention prefill for sm_103a (dense and varlen, causal or not,
// GQA/MQA, head dim 64/128/256).
//
// Operation: the "SuperL8" README (github.com/jajmangold/superl8), "Attention
// kernels" table -- attn_int8_fwd (W8A8 FlashAttention-2; causal, GQA/MQA, head
// dims 32/64/128/256) and attn_varlen_fwd (ragged prefill) -- with the layouts
// of its "Quick start" section.  Per (sequence, query head):
//   S = int32(Q_i8 . K_i8^T);  x = S * s_q * s_k / sqrt(d);  causal mask (key j
//   allowed for query i iff j <= i, top-left aligned);  online softmax
//   (FlashAttention-2);  O = P . V with P rounded to V's dtype, fp32 accumulation.
//
// GB300 design (not the pages' DP4A CUDA-core design):
//   * sm_103a has no tcgen05 kind::i8 MMA.  The int8 codes are held as bf16 (every
//     integer in [-127, 127] is exact in bf16) and QK^T runs as tcgen05 kind::f16
//     with fp32 accumulation in TMEM.  Every partial sum is an integer of
//     magnitude <= 256 * 127^2 < 2^24, so S is the exact int32 dot.
//   * Persistent CTAs walk a longest-first list of (sequence, 128-row q-tile,
//     head) items built on the device.  Roles: warp 0 issues TMA loads of Q, K
//     (128B-swizzled code tiles from the workspace) and V (the caller's tensor);
//     warp 1 issues tcgen05.mma from one thread (S = Q K^T into one of two TMEM
//     buffers; O += P V with P read from TMEM); warps 4..7 (one thread per query
//     row) load S from TMEM, dequantise, mask, run the online softmax, write P
//     back over S in TMEM, rescale O when the running max grows by more than
//     2^8, and write the normalised output.
//   * Every mbarrier wait is bounded in time; a timeout is recorded in the
//     library's status word and the CTA winds down.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sl8_internal.h"

namespace sl8 {

namespace {

constexpr int kThreads = 256;
constexpr int kSoftmaxWarp0 = 4;  // warps 4..7: TMEM lanes 0..127
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Cfg {
  static constexpr int BN = D <= 128 ? 128 : 64;         // keys per KV tile
  static constexpr int kBoxes = D / 64;                    // 64-element (128 B) boxes along d
  static constexpr int kQBytes = kQTile * D * 2;
  static constexpr int kKBytes = BN * D * 2;
  static constexpr int kVBytes = BN * D * 2;
  static constexpr int kStages = 2;
  static constexpr int kQStages = D <= 128 ? 2 : 1;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQStages * kQBytes;
  static constexpr int kVOff = kKOff + kStages * kKBytes;
  static constexpr int kScaleOff = kVOff + kStages * kVBytes;  // 2 x BN floats
  static constexpr int kBarOff = kScaleOff + 2 * BN * 4;
  // + barriers + alignment slack; at least 116 KB so that a second CTA never shares the SM
  // (each CTA holds all 512 TMEM columns)
  static constexpr int kSmemBytes = kBarOff + 256 + 1024 > 118784 ? kBarOff + 256 + 1024 : 118784;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 2 * BN;
  static_assert(kOCol + D <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "smem budget");
};

struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct Item {
  int32_t s, qt, hq, hkv, L, pstart, tok0, nkv;
};

template <int D>
__device__ __forceinline__ Item decode_item(const PrefillArgs& a, int64_t item, int group, bool causal) {
  Item it;
  const int64_t pair = item / a.Hq;
  it.hq = static_cast<int32_t>(item - pair * a.Hq);
  it.hkv = it.hq / group;
  it.s = a.table.pair_seq[pair];
  it.qt = a.table.pair_qt[pair];
  it.L = a.table.len[it.s];
  it.pstart = a.table.pstart[it.s];
  it.tok0 = a.table.tok0[it.s];
  constexpr int BN = Cfg<D>::BN;
  const int kend = causal ? min(it.L, (it.qt + 1) * kQTile) : it.L;
  it.nkv = (kend + BN - 1) / BN;
  return it;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}


// OR of a flag over the 128 softmax threads (named barrier 1); also orders their
// shared-memory accesses like bar.sync.
__device__ __forceinline__ bool wg_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, 128, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

template <int D, bool kLogits>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap map_q,
                                                              const __grid_constant__ CUtensorMap map_k,
                                                              const __grid_constant__ CUtensorMap map_v,
                                                              const PrefillArgs a, DeviceStatus* st,
                                                              uint64_t limit_ns) {
  using C = Cfg<D>;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + C::kBarOff);
  float* sks = reinterpret_cast<float*>(smem + C::kScaleOff);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const bool causal = kLogits ? false : a.causal;
  const int group = a.Hq / a.Hkv;
  const int64_t n_items = static_cast<int64_t>(a.table.counts[0]) * a.Hq;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 1);
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 128);
      mbar_init(&bars.o_done[i], 1);
    }
    mbar_init(&bars.drain, 1);
    bars.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars.tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars.tmem_base;
  volatile int* abort_flag = &bars.abort;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      uint32_t g = 0, it = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
        const Item w = decode_item<D>(a, item, group, causal);
        const uint32_t qs = it % C::kQStages;
        if (it >= C::kQStages) ok = mbar_wait(&bars.q_empty[qs], ((it / C::kQStages) - 1) & 1, limit_ns, st, 10);
        if (!ok || *abort_flag) break;
        uint8_t* qdst = smem + C::kQOff + qs * C::kQBytes;
        mbar_arrive_expect_tx(&bars.q_full[qs], C::kQBytes);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(qdst + b * (kQTile * 128), &map_q, &bars.q_full[qs], b * 64, w.pstart + w.qt * kQTile, w.hq);
        for (int j = 0; j < w.nkv; ++j, ++g) {
          const uint32_t stg = g % C::kStages, n = g / C::kStages;
          if (g >= C::kStages) ok = mbar_wait(&bars.k_empty[stg], (n - 1) & 1, limit_ns, st, 11);
          if (!ok || *abort_flag) break;
          uint8_t* kdst = smem + C::kKOff + stg * C::kKBytes;
          mbar_arrive_expect_tx(&bars.k_full[stg], C::kKBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(kdst + b * (BN * 128), &map_k, &bars.k_full[stg], b * 64, w.pstart + j * BN, w.hkv);
          if (g >= C::kStages) ok = mbar_wait(&bars.v_empty[stg], (n - 1) & 1, limit_ns, st, 12);
          if (!ok || *abort_flag) break;
          uint8_t* vdst = smem + C::kVOff + stg * C::kVBytes;
          mbar_arrive_expect_tx(&bars.v_full[stg], C::kVBytes);
          for (int b = 0; b < C::kBoxes; ++b) {
            if (a.v16)
              tma_load_3d(vdst + b * (BN * 128), &map_v, &bars.v_full[stg], b * 64, w.pstart + j * BN, w.hkv);
            else if (a.varlen)
              tma_load_3d(vdst + b * (BN * 128), &map_v, &bars.v_full[stg], b * 64, w.hkv, w.tok0 + j * BN);
            else
              tma_load_3d(vdst + b * (BN * 128), &map_v, &bars.v_full[stg], b * 64, j * BN, w.s * a.Hkv + w.hkv);
          }
        }
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(kQTile, BN, true, false, false);
      constexpr uint32_t idesc_o = idesc_f16(kQTile, D, false, false, true);  // fp16 P x fp16 V
      // S stream state
      int64_t item_s = blockIdx.x;
      uint32_t it_s = 0;
      int j_s = 0;
      Item ws{};
      if (item_s < n_items) ws = decode_item<D>(a, item_s, group, causal);
      uint32_t gs = 0;
      // PV stream state
      int64_t item_p = blockIdx.x;
      int j_p = 0;
      Item wp{};
      if (item_p < n_items) wp = decode_item<D>(a, item_p, group, causal);
      uint32_t gp = 0;
      bool ok = true;
      bool issued_any = false;
      while (ok && item_p < n_items && !*abort_flag) {
        // issue S tiles up to gp + 1
        while (ok && item_s < n_items && gs <= gp + 1) {
          const uint32_t qs = it_s % C::kQStages;
          if (j_s == 0) ok = mbar_wait(&bars.q_full[qs], (it_s / C::kQStages) & 1, limit_ns, st, 20);
          const uint32_t stg = gs % C::kStages;
          if (ok) ok = mbar_wait(&bars.k_full[stg], (gs / C::kStages) & 1, limit_ns, st, 21);
          if (!ok) break;
          tc_fence_after();
          const uint32_t qaddr = smem_u32(smem + C::kQOff + qs * C::kQBytes);
          const uint32_t kaddr = smem_u32(smem + C::kKOff + stg * C::kKBytes);
          const uint32_t dcol = tbase + (gs & 1) * BN;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t da = desc_sw128(qaddr + (k / 4) * (kQTile * 128) + (k % 4) * 32, 16, 1024);
            const uint64_t db = desc_sw128(kaddr + (k / 4) * (BN * 128) + (k % 4) * 32, 16, 1024);
            mma_ss(dcol, da, db, idesc_s, k > 0 ? 1u : 0u);
          }
          issued_any = true;
          mma_commit(&bars.s_full[gs & 1]);
          mma_commit(&bars.k_empty[stg]);
          ++gs;
          if (++j_s == ws.nkv) {
            mma_commit(&bars.q_empty[qs]);
            j_s = 0;
            ++it_s;
            item_s += gridDim.x;
            if (item_s < n_items) ws = decode_item<D>(a, item_s, group, causal);
          }
        }
        if (!ok) break;
        // O += P V for tile gp
        ok = mbar_wait(&bars.p_full[gp & 1], (gp >> 1) & 1, limit_ns, st, 22);
        const uint32_t stg = gp % C::kStages;
        if (ok) ok = mbar_wait(&bars.v_full[stg], (gp / C::kStages) & 1, limit_ns, st, 23);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vaddr = smem_u32(smem + C::kVOff + stg * C::kVBytes);
        const uint32_t pcol = tbase + (gp & 1) * BN;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t db = desc_sw128(vaddr + k * 2048, BN * 128, 1024);
          mma_ts(tbase + C::kOCol, pcol + k * 8, db, idesc_o, (j_p > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&bars.o_done[gp & 1]);
        mma_commit(&bars.v_empty[stg]);
        ++gp;
        if (++j_p == wp.nkv) {
          j_p = 0;
          item_p += gridDim.x;
          if (item_p < n_items) wp = decode_item<D>(a, item_p, group, causal);
        }
      }
      if (!ok) *abort_flag = 1;
      if (issued_any) {
        // make sure every MMA this thread issued has finished before TMEM is released
        mma_commit(&bars.drain);
        mbar_wait(&bars.drain, 0, limit_ns, st, 24);
      }
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------------------------------ softmax / epilogue
    // Control flow here is uniform across the 128 threads: every wait result is made
    // warp-uniform with __all_sync and every exit decision group-uniform with a
    // reducing named barrier, so no thread is ever left waiting at a barrier.
    const int r = threadIdx.x - kSoftmaxWarp0 * 32;        // query row within the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp - kSoftmaxWarp0) * 32) << 16;
    const float qk_scale = 1.4426950408889634f / sqrtf(static_cast<float>(D));  // log2(e) / sqrt(d)
    const bool out_bf16 = a.out_dtype == SL8_BF16, out_f32 = a.out_dtype == SL8_F32;
    int64_t item = blockIdx.x;
    Item w{};
    if (item < n_items) w = decode_item<D>(a, item, group, causal);
    uint32_t g = 0;
    // prefetched per-row Q scale and per-tile K scale
    float qs_next = 0.0f, ks_next = 0.0f;
    int ve_next = 0;
    if (item < n_items) {
      qs_next = a.q_scales[static_cast<int64_t>(w.hq) * a.t_pad_max + w.pstart + w.qt * kQTile + r];
      if (a.v_exp) ve_next = a.v_exp[static_cast<int64_t>(w.s) * a.Hkv + w.hkv];
      if (r < BN) ks_next = a.k_scales[static_cast<int64_t>(w.hkv) * a.t_pad_max + w.pstart + r];
    }
    bool bad = false;
    while (item < n_items) {
      const int row_abs = w.qt * kQTile + r;
      const float alpha = qs_next * qk_scale;
      const float v_unscale = __int_as_float((127 + ve_next) << 23);  // 2^e undoes V's fp16 scaling
      float m = -INFINITY, l = 0.0f;
      for (int j = 0; j < w.nkv; ++j, ++g) {
        const uint32_t buf = g & 1;
        if (r < BN) sks[buf * BN + r] = ks_next;
        // prefetch the scales of the next tile (possibly of the next item)
        {
          int jn = j + 1;
          int64_t in = item;
          Item wn = w;
          if (jn == w.nkv) {
            jn = 0;
            in = item + gridDim.x;
            if (in < n_items) wn = decode_item<D>(a, in, group, causal);
          }
          if (in < n_items) {
            if (r < BN) ks_next = a.k_scales[static_cast<int64_t>(wn.hkv) * a.t_pad_max + wn.pstart + jn * BN + r];
            if (jn == 0) {
              qs_next = a.q_scales[static_cast<int64_t>(wn.hq) * a.t_pad_max + wn.pstart + wn.qt * kQTile + r];
              if (a.v_exp) ve_next = a.v_exp[static_cast<int64_t>(wn.s) * a.Hkv + wn.hkv];
            }
          }
        }
        if (wg_any(bad || *abort_flag)) { bad = true; break; }   // also publishes sks to the group
        if (!__all_sync(0xffffffffu, mbar_wait(&bars.s_full[buf], (g >> 1) & 1, limit_ns, st, 30))) {
          bad = true;
          continue;
        }
        tc_fence_after();
        float x[BN];
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_base + buf * BN + c0, v);
#pragma unroll
          for (int c = 0; c < 32; ++c) x[c0 + c] = __uint_as_float(v[c]);
        }
        tmem_wait_ld();
        if constexpr (kLogits) {
          // debug: write the exact int32 logits of this row for keys < L
          if (row_abs >= a.row_begin && row_abs < a.row_end && row_abs < w.L) {
            int32_t* dst = a.logits + ((static_cast<int64_t>(w.s) * a.Hq + w.hq) * (a.row_end - a.row_begin) +
                                       (row_abs - a.row_begin)) * a.N;
#pragma unroll
            for (int c = 0; c < BN; ++c) {
              const int key = j * BN + c;
              if (key < w.L) dst[key] = __float2int_rn(x[c]);
            }
          }
        } else {
          const float* ks = sks + buf * BN;
          const int key0 = j * BN;
          const bool need_mask = (causal && key0 + BN - 1 > w.qt * kQTile) || (key0 + BN > w.L);
          float tmax = -INFINITY;
          if (need_mask) {
#pragma unroll
            for (int c = 0; c < BN; ++c) {
              const int key = key0 + c;
              const bool valid = key < w.L && (!causal || key <= row_abs);
              x[c] = valid ? x[c] * ks[c] : -INFINITY;
              tmax = fmaxf(tmax, x[c]);
            }
          } else {
#pragma unroll
            for (int c = 0; c < BN; ++c) {
              x[c] = x[c] * ks[c];
              tmax = fmaxf(tmax, x[c]);
            }
          }
          const float m_tile = tmax == -INFINITY ? -INFINITY : tmax * alpha;
          float o_scale = 1.0f;
          bool rescale = false;
          if (j == 0) {
            m = m_tile;
          } else if (m_tile > m + kRescaleThreshold) {
            o_scale = exp2f(m - m_tile);
            l *= o_scale;
            m = m_tile;
            rescale = true;
          }
          const float neg_m = m == -INFINITY ? 0.0f : -m;
          float rowsum = 0.0f;
          uint32_t p[BN / 2];
#pragma unroll
          for (int c = 0; c < BN; c += 2) {
            const float p0 = x[c] == -INFINITY ? 0.0f : exp2f(fmaf(x[c], alpha, neg_m));
            const float p1 = x[c + 1] == -INFINITY ? 0.0f : exp2f(fmaf(x[c + 1], alpha, neg_m));
            rowsum += p0 + p1;
            p[c / 2] = pack2(p0, p1, false);
          }
          l += rowsum;
#pragma unroll
          for (int c0 = 0; c0 < BN / 2; c0 += 16) {
            uint32_t v[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = p[c0 + c];
            tmem_st16(tbase + lane_base + buf * BN + c0, v);
          }
          if (__any_sync(0xffffffffu, rescale)) {
            // O holds the sum up to tile g-1: wait for that PV, then scale it in place
            const uint32_t gprev = g - 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&bars.o_done[gprev & 1], (gprev >> 1) & 1, limit_ns, st, 31))) {
              bad = true;
              continue;
            }
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 16) {
              uint32_t v[16];
              tmem_ld16(tbase + lane_base + C::kOCol + c0, v);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 16; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * o_scale);
              tmem_st16(tbase + lane_base + C::kOCol + c0, v);
            }
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars.p_full[buf]);
      }
      if (wg_any(bad || *abort_flag)) { bad = true; break; }
      // ---- epilogue: O / l for this item
      const uint32_t glast = g - 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars.o_done[glast & 1], (glast >> 1) & 1, limit_ns, st, 32))) {
        bad = true;
      } else {
        tc_fence_after();
        if constexpr (!kLogits) {
          const bool row_ok = row_abs < w.L;
          const float inv_l = v_unscale / l;
          const int64_t orow = a.varlen ? (static_cast<int64_t>(w.tok0) + row_abs) * a.Hq + w.hq
                                        : (static_cast<int64_t>(w.s) * a.Hq + w.hq) * a.N + row_abs;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tbase + lane_base + C::kOCol + c0, v);
            tmem_wait_ld();
            if (row_ok) {
              if (out_f32) {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow * D + c0);
#pragma unroll
                for (int c = 0; c < 16; c += 4)
                  dst[c / 4] = make_float4(__uint_as_float(v[c]) * inv_l, __uint_as_float(v[c + 1]) * inv_l,
                                           __uint_as_float(v[c + 2]) * inv_l, __uint_as_float(v[c + 3]) * inv_l);
              } else {
                uint32_t pk[8];
#pragma unroll
                for (int c = 0; c < 16; c += 2)
                  pk[c / 2] = pack2(__uint_as_float(v[c]) * inv_l, __uint_as_float(v[c + 1]) * inv_l, out_bf16);
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + orow * D + c0);
                dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
              }
            }
          }
          if (row_ok && a.lse) a.lse[orow] = (m + log2f(l)) * 0.6931471805599453f;
        }
      }
      item += gridDim.x;
      if (item < n_items) w = decode_item<D>(a, item, group, causal);
    }
    if (bad) *abort_flag = 1;
  }
  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, C::kTmemCols);
}

}  // namespace

template <int D, bool kLogits>
static cudaError_t launch_prefill_d(const PrefillArgs& a, cudaStream_t s) {
  using C = Cfg<D>;
  bool ok = true;
  const CUtensorMap mq = make_tmap_3d(a.q_codes, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, a.t_pad_max, a.Hq, D * 2ull,
                                      a.t_pad_max * D * 2ull, 64, kQTile, 1, &ok);
  const CUtensorMap mk = make_tmap_3d(a.k_codes, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, a.t_pad_max, a.Hkv, D * 2ull,
                                      a.t_pad_max * D * 2ull, 64, C::BN, 1, &ok);
  // P.V runs in fp16: V is either the caller's fp16 tensor or the fp16 copy of a bf16 V
  // in the padded workspace layout (same coordinates as K)
  CUtensorMap mv;
  if (a.v16)
    mv = make_tmap_3d(a.v16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, D, a.t_pad_max, a.Hkv, D * 2ull, a.t_pad_max * D * 2ull,
                      64, C::BN, 1, &ok);
  else if (a.varlen)  // [T, Hkv, d]: dims (d, Hkv, T)
    mv = make_tmap_3d(a.v, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, D, a.Hkv, a.total_tokens, D * 2ull,
                      static_cast<uint64_t>(a.Hkv) * D * 2ull, 64, 1, C::BN, &ok);
  else  // [nseq, Hkv, N, d]: dims (d, N, nseq*Hkv)
    mv = make_tmap_3d(a.v, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, D, a.N, static_cast<uint64_t>(a.nseq) * a.Hkv, D * 2ull,
                      static_cast<uint64_t>(a.N) * D * 2ull, 64, C::BN, 1, &ok);
  if (!ok) return cudaErrorInvalidValue;
  auto kern = prefill_kernel<D, kLogits>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t max_items = a.max_pairs * a.Hq;
  const int grid = static_cast<int>(max_items < num_sms() ? max_items : num_sms());
  if (grid <= 0) return cudaSuccess;
  TraceScope tr(kLogits ? "prefill_logits" : "prefill_attn", s);
  kern<<<grid, kThreads, C::kSmemBytes, s>>>(mq, mk, mv, a, device_status_ptr(), spin_limit_ns());
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  const bool logits = a.logits != nullptr;
  switch (a.d) {
    case 64: return logits ? launch_prefill_d<64, true>(a, s) : launch_prefill_d<64, false>(a, s);
    case 128: return logits ? launch_prefill_d<128, true>(a, s) : launch_prefill_d<128, false>(a, s);
    case 256: return logits ? launch_prefill_d<256, true>(a, s) : launch_prefill_d<256, false>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sl8
