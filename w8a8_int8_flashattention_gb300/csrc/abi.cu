// C ABI of libsl8: argument validation, workspace planning, the per-device status
// word, tensor-map encoding and kernel tracing.  The kernels live in quant.cu,
// prefill.cu and decode.cu; every entry point here only validates and enqueues.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <map>
#include <string>
#include <vector>

#include "sl8_internal.h"

namespace sl8 {

// ---------------------------------------------------------------- device status
// One status word per device (a __device__ variable: loaded with the module, no
// allocation).  Its address is looked up once per device.
static __device__ DeviceStatus g_device_status;

static constexpr int kMaxDevices = 64;
static std::mutex g_mu;
static DeviceStatus* g_status_ptr[kMaxDevices] = {};
static int g_num_sms[kMaxDevices] = {};
static std::atomic<uint64_t> g_spin_limit_ns{2000000000ull};

static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

DeviceStatus* device_status_ptr() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<DeviceStatus*>(p);
  }
  return g_status_ptr[dev];
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_num_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

uint64_t spin_limit_ns() { return g_spin_limit_ns.load(std::memory_order_relaxed); }

cudaError_t ensure_smem(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;
  const int dev = current_device();
  std::lock_guard<std::mutex> lk(mu);
  int& have = done[{kernel, dev}];
  if (have >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

// ---------------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 3-D tiled map with zero fill out of bounds, 128-byte swizzle or none.
CUtensorMap make_tmap_3d(const void* base, CUtensorMapDataType dt, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                         bool* ok, bool swizzle128) {
  CUtensorMap m;
  memset(&m, 0, sizeof(m));
  auto fn = encode_fn();
  if (!fn) {
    *ok = false;
    return m;
  }
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(&m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) *ok = false;
  return m;
}

// ---------------------------------------------------------------- tracing
struct TraceRec {
  const char* name;
  cudaEvent_t start, stop;
};
static std::atomic<int> g_trace_on{0};
static std::mutex g_trace_mu;
static std::vector<TraceRec> g_trace;
static std::vector<cudaEvent_t> g_event_pool;

static cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

TraceScope::TraceScope(const char* name, cudaStream_t s) : slot(-1), stream(s) {
  if (!g_trace_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  TraceRec r{name, take_event(), take_event()};
  if (!r.start || !r.stop) return;
  cudaEventRecord(r.start, s);
  g_trace.push_back(r);
  slot = static_cast<int>(g_trace.size()) - 1;
}

TraceScope::~TraceScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (slot < static_cast<int>(g_trace.size())) cudaEventRecord(g_trace[slot].stop, stream);
}

// ---------------------------------------------------------------- workspace plans
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

PrefillWorkspace plan_prefill_workspace(int32_t nseq, int32_t Hq, int32_t Hkv, int32_t N, int32_t d,
                                        int64_t total_tokens, bool varlen) {
  if (d == 32) d = 64;  // head dim 32 runs as 64: code, V and partial rows of 64
  PrefillWorkspace w{};
  w.max_tiles = (N + kQTile - 1) / kQTile;
  w.max_chunks = (N + kMeanChunk - 1) / kMeanChunk;
  const int64_t dense_rows = static_cast<int64_t>(nseq) * w.max_tiles * kPadRows;
  if (varlen) {
    const int64_t bound = (total_tokens + static_cast<int64_t>(nseq) * (kPadRows - 1)) / kPadRows * kPadRows;
    w.t_pad_max = bound < dense_rows ? bound : dense_rows;
    const int64_t pb = (total_tokens + kQTile - 1) / kQTile + nseq;
    w.max_pairs = pb < static_cast<int64_t>(nseq) * w.max_tiles ? pb : static_cast<int64_t>(nseq) * w.max_tiles;
  } else {
    w.t_pad_max = dense_rows;
    w.max_pairs = static_cast<int64_t>(nseq) * w.max_tiles;
  }
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  w.q_codes = take(static_cast<size_t>(Hq) * w.t_pad_max * d * 2);
  w.q_scales = take(static_cast<size_t>(Hq) * w.t_pad_max * 4);
  w.k_codes = take(static_cast<size_t>(Hkv) * w.t_pad_max * d * 2);
  w.k_scales = take(static_cast<size_t>(Hkv) * w.t_pad_max * 4);
  w.v16 = take(static_cast<size_t>(Hkv) * w.t_pad_max * d * 2);
  w.k_mean = take(static_cast<size_t>(nseq) * Hkv * d * 4);
  w.k_partials = take(static_cast<size_t>(nseq) * Hkv * w.max_chunks * d * 4);
  w.v_partials = take(static_cast<size_t>(nseq) * Hkv * w.max_chunks * 4);
  w.v_exp = take(static_cast<size_t>(nseq) * Hkv * 4);
  w.kv_done = take(static_cast<size_t>(nseq) * Hkv * 4);
  w.pstart = take(static_cast<size_t>(nseq) * 4);
  w.len = take(static_cast<size_t>(nseq) * 4);
  w.tok0 = take(static_cast<size_t>(nseq) * 4);
  w.pair_seq = take(static_cast<size_t>(w.max_pairs) * 4);
  w.pair_qt = take(static_cast<size_t>(w.max_pairs) * 4);
  w.counts = take(16);
  w.hist = take(static_cast<size_t>(3) * (w.max_tiles + 2) * 4);
  w.sorted = take(static_cast<size_t>(nseq) * 4);
  w.total = off;
  return w;
}

static SeqTable table_at(void* ws, const PrefillWorkspace& p) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  SeqTable t;
  t.pstart = reinterpret_cast<int32_t*>(b + p.pstart);
  t.len = reinterpret_cast<int32_t*>(b + p.len);
  t.tok0 = reinterpret_cast<int32_t*>(b + p.tok0);
  t.pair_seq = reinterpret_cast<int32_t*>(b + p.pair_seq);
  t.pair_qt = reinterpret_cast<int32_t*>(b + p.pair_qt);
  t.counts = reinterpret_cast<int32_t*>(b + p.counts);
  t.hist = reinterpret_cast<int32_t*>(b + p.hist);
  t.sorted = reinterpret_cast<int32_t*>(b + p.sorted);
  return t;
}

}  // namespace sl8

using namespace sl8;

// ---------------------------------------------------------------- validation helpers
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool is_half(int dt) { return dt == SL8_F16 || dt == SL8_BF16; }
bool head_dim_ok(int32_t d) { return d == 64 || d == 128 || d == 256; }
// The decode kernels also take head dim 32 (int8 V only).
static bool decode_head_dim_ok(int32_t d) { return d == 32 || head_dim_ok(d); }
// Head dim the prefill kernels compute in: 32 runs as 64 (codes, V copy and O zero past 32).
int32_t compute_dim(int32_t d) { return d == 32 ? 64 : d; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SL8_OK : SL8_ERR_CUDA; }

#define SL8_CHECK(cond, code) \
  do {                        \
    if (!(cond)) return (code); \
  } while (0)

// The CUDA error behind the calling thread's last SL8_ERR_CUDA.
static thread_local cudaError_t g_last_cuda_error = cudaSuccess;
#define SL8_LAUNCH(expr)                     \
  do {                                       \
    cudaError_t e_ = (expr);                 \
    if (e_ != cudaSuccess) {                 \
      g_last_cuda_error = e_;                \
      return SL8_ERR_CUDA;                   \
    }                                        \
  } while (0)

int validate_prefill(const void* q, const void* k, int qk_dtype, int32_t B, int32_t Hq, int32_t Hkv, int32_t N,
                     int32_t d) {
  SL8_CHECK(q && k, SL8_ERR_INVALID_ARG);
  SL8_CHECK(aligned16(q) && aligned16(k), SL8_ERR_INVALID_ARG);
  SL8_CHECK(is_half(qk_dtype), SL8_ERR_INVALID_ARG);
  SL8_CHECK(B >= 0 && N >= 0 && Hq > 0 && Hkv > 0 && d > 0, SL8_ERR_INVALID_ARG);
  SL8_CHECK(Hq % Hkv == 0, SL8_ERR_INVALID_ARG);
  SL8_CHECK(d == 32 || head_dim_ok(d), SL8_ERR_UNSUPPORTED);  // head dim 32 runs as 64
  SL8_CHECK(N <= (1 << 24) && B <= (1 << 24), SL8_ERR_UNSUPPORTED);
  return SL8_OK;
}

}  // namespace

extern "C" {

const char* sl8_status_string(int status) {
  switch (status) {
    case SL8_OK: return "ok";
    case SL8_ERR_INVALID_ARG: return "invalid argument";
    case SL8_ERR_UNSUPPORTED: return "unsupported configuration";
    case SL8_ERR_WORKSPACE: return "workspace missing or too small";
    case SL8_ERR_CUDA: return "CUDA error";
    case SL8_ERR_TIMEOUT: return "device-side wait timed out";
    case SL8_ERR_DEVICE_ARG: return "device-side argument out of range";
    default: return "unknown status";
  }
}

int sl8_version(void) { return 100; }

const char* sl8_last_cuda_error_string(void) {
  return g_last_cuda_error == cudaSuccess ? "no CUDA error recorded" : cudaGetErrorString(g_last_cuda_error);
}

int sl8_quant_rowwise(const void* x, int x_dtype, int64_t rows, int32_t cols, int64_t row_stride_elems,
                      const float* sub_mean, int64_t rows_per_group, int8_t* q_out, float* scale_out, void* stream) {
  if (rows == 0 && cols >= 1) return SL8_OK;  // nothing to read or write; pointers may be null
  SL8_CHECK(x && q_out && scale_out, SL8_ERR_INVALID_ARG);
  SL8_CHECK(x_dtype == SL8_F16 || x_dtype == SL8_BF16 || x_dtype == SL8_F32, SL8_ERR_INVALID_ARG);
  SL8_CHECK(rows >= 0 && cols >= 1 && row_stride_elems >= cols, SL8_ERR_INVALID_ARG);
  SL8_CHECK(!sub_mean || rows_per_group >= 1, SL8_ERR_INVALID_ARG);
  SL8_CHECK(rows / 8 < (1ll << 31), SL8_ERR_UNSUPPORTED);
  if (rows == 0) return SL8_OK;
  return cuda_status(launch_quant_rowwise(x, static_cast<sl8_dtype>(x_dtype), rows, cols, row_stride_elems, sub_mean,
                                          sub_mean ? rows_per_group : 1, q_out, scale_out,
                                          static_cast<cudaStream_t>(stream)));
}

size_t sl8_k_channel_mean_workspace_size(int32_t B, int32_t Hkv, int32_t N, int32_t d) {
  if (B < 0 || Hkv <= 0 || N < 0 || d <= 0) return 0;
  // the table part of the prefill plan (Hq = Hkv) plus the chunk partials
  const PrefillWorkspace p = plan_prefill_workspace(B, Hkv, Hkv, N, d, 0, false);
  return p.total - p.k_mean;
}

int sl8_k_channel_mean(const void* k, int k_dtype, int32_t B, int32_t Hkv, int32_t N, int32_t d,
                       const int32_t* cu_seqlens, int64_t total_tokens, float* mean_out, void* workspace,
                       size_t workspace_bytes, void* stream) {
  SL8_CHECK(k && mean_out && aligned16(k), SL8_ERR_INVALID_ARG);
  SL8_CHECK(k_dtype == SL8_F16 || k_dtype == SL8_BF16 || k_dtype == SL8_F32, SL8_ERR_INVALID_ARG);
  SL8_CHECK(B >= 0 && Hkv > 0 && N >= 0 && d > 0 && d <= 1024, SL8_ERR_INVALID_ARG);
  SL8_CHECK(!cu_seqlens || total_tokens >= 0, SL8_ERR_INVALID_ARG);
  if (B == 0 || N == 0) return SL8_OK;
  const size_t need = sl8_k_channel_mean_workspace_size(B, Hkv, N, d);
  SL8_CHECK(workspace && workspace_bytes >= need && aligned16(workspace), SL8_ERR_WORKSPACE);
  // reuse the prefill plan's layout shifted so that k_mean starts at the workspace base
  const PrefillWorkspace p = plan_prefill_workspace(B, Hkv, Hkv, N, d, 0, false);
  uint8_t* base = static_cast<uint8_t*>(workspace) - p.k_mean;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const SeqTable t = table_at(base, p);
  int32_t* kv_done = reinterpret_cast<int32_t*>(base + p.kv_done);
  SL8_LAUNCH(launch_schedule(cu_seqlens, B, N, cu_seqlens ? total_tokens : static_cast<int64_t>(B) * N,
                             static_cast<int64_t>(B) * p.max_tiles * kPadRows, t, kQTile, kv_done, B * Hkv, s));
  SL8_LAUNCH(launch_kv_stats(k, static_cast<sl8_dtype>(k_dtype), nullptr, cu_seqlens != nullptr, B, Hkv, N, d, t.len,
                             t.tok0, reinterpret_cast<float*>(base + p.k_partials), nullptr, p.max_chunks, mean_out,
                             nullptr, kv_done, s));
  return SL8_OK;
}

size_t sl8_attn_int8_fwd_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t N, int32_t d,
                                        int64_t total_tokens) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || N < 0 || d <= 0 || total_tokens < 0) return 0;
  return plan_prefill_workspace(B, Hq, Hkv, N, d, total_tokens, total_tokens > 0).total;
}

// Scheduler, K/V statistics and quantisation ahead of the attention kernel.  With a
// bf16 V (v non-null) V is also re-expressed in fp16 (scaled by 2^-e) for the P.V MMA.
static int prefill_prepare(const void* q, const void* k, const void* v, int qk_dtype, int v_dtype, int32_t B,
                           int32_t Hq, int32_t Hkv, int32_t N, int32_t d, const int32_t* cu_seqlens,
                           int64_t total_tokens, int smooth_k, void* workspace, size_t workspace_bytes,
                           cudaStream_t s, bool want_table, PrefillWorkspace* plan, SeqTable* table,
                           int32_t q_off = 0, const QuantGroups& groups = QuantGroups()) {
  const bool varlen = cu_seqlens != nullptr;
  const PrefillWorkspace p = plan_prefill_workspace(B, Hq, Hkv, N, d, varlen ? total_tokens : 0, varlen);
  SL8_CHECK(workspace && aligned16(workspace) && workspace_bytes >= p.total, SL8_ERR_WORKSPACE);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const SeqTable t = table_at(ws, p);
  const int64_t tokens = varlen ? total_tokens : static_cast<int64_t>(B) * N;
  // head dim 32 runs as 64 (zero channels past 32): V always goes through the padded copy
  const int32_t dc = compute_dim(d);
  const bool convert_v = v && (v_dtype == SL8_BF16 || dc != d);
  const bool v_stats = v && v_dtype == SL8_BF16;
  // the scheduler's table is needed for varlen input (and by the code export); dense
  // input is laid out arithmetically
  if (varlen || want_table)
    SL8_LAUNCH(launch_schedule(cu_seqlens, B, N, tokens, p.t_pad_max, t, prefill_item_rows(dc, Hq / Hkv), nullptr, 0,
                               s));
  float* k_partials = smooth_k ? reinterpret_cast<float*>(ws + p.k_partials) : nullptr;
  float* v_partials = v_stats ? reinterpret_cast<float*>(ws + p.v_partials) : nullptr;
  if (smooth_k || v_stats) {
    SL8_LAUNCH(launch_kv_partials(k, static_cast<sl8_dtype>(qk_dtype), v_stats ? v : nullptr, varlen, B, Hkv, N, d,
                                  varlen ? t.len : nullptr, varlen ? t.tok0 : nullptr, k_partials, v_partials,
                                  p.max_chunks, tokens, s));
    SL8_LAUNCH(launch_kv_finalize(varlen, B, Hkv, N, d, varlen ? t.len : nullptr, k_partials, v_partials, p.max_chunks,
                                  reinterpret_cast<float*>(ws + p.k_mean), reinterpret_cast<int32_t*>(ws + p.v_exp),
                                  s));
  }
  SL8_LAUNCH(launch_quant_qk(q, k, static_cast<sl8_dtype>(qk_dtype), varlen, B, Hq, Hkv, N, dc, tokens, t,
                             p.t_pad_max, k_partials, v_partials, p.max_chunks,
                             reinterpret_cast<uint16_t*>(ws + p.q_codes), reinterpret_cast<float*>(ws + p.q_scales),
                             reinterpret_cast<uint16_t*>(ws + p.k_codes), reinterpret_cast<float*>(ws + p.k_scales),
                             convert_v ? v : nullptr, convert_v ? reinterpret_cast<int32_t*>(ws + p.v_exp) : nullptr,
                             convert_v ? reinterpret_cast<uint16_t*>(ws + p.v16) : nullptr, s, q_off, d,
                             v_dtype == SL8_F16, groups, smooth_k ? reinterpret_cast<float*>(ws + p.k_mean) : nullptr));
  *plan = p;
  *table = t;
  return SL8_OK;
}

// Key splits of a dense query chunk (the attention kernel for d <= 128 only).  When the
// chunk's (query tile, head) items number at most half the SMs, each item's keys are cut
// into SMs / items parts (at most kMaxKeySplit, each keeping at least two key tiles of
// the longest item), so that the parts run as one wave.  Larger chunks are not split: a
// part costs about one key tile's time to fill and drain the tile pipeline, and the merge
// reads every partial once more, which outweighs rebalancing a wave that is mostly full.
static int32_t chunk_kv_split(int32_t B, int32_t Hq, int32_t Hkv, int32_t Nk, int32_t Nq, int32_t d) {
  const int32_t dc = compute_dim(d);
  if (dc > 128 || Nq <= 0 || B <= 0) return 1;
  const int32_t item_rows = prefill_item_rows(dc, Hq / Hkv);
  const int64_t per_seq = (Nk + item_rows - 1) / item_rows - (Nk - Nq) / item_rows;
  const int64_t items = static_cast<int64_t>(B) * per_seq * (prefill_head_pairs(dc, Hq / Hkv) ? Hq / 2 : Hq);
  const int64_t sms = num_sms();
  if (2 * items > sms) return 1;
  int64_t split = sms / items;
  const int64_t max_tiles = (Nk + kQTile - 1) / kQTile;
  if (split > max_tiles / 2) split = max_tiles / 2;
  if (split > kMaxKeySplit) split = kMaxKeySplit;
  return split < 1 ? 1 : static_cast<int32_t>(split);
}

// Bytes of the key-split partials of a chunk split into `split` parts: O [split][B * Hq *
// Nq][d] fp32, then (256-byte aligned) the LSE [split][B * Hq * Nq].
static size_t chunk_partial_o_bytes(int32_t split, int64_t rows, int32_t d) {
  return align_up(static_cast<size_t>(split) * rows * d * sizeof(float), 256);
}

// Workspace of a query chunk: the prefill plan over Nk keys, then the key-split partials
// when the chunk is split on this device.
static size_t chunk_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t Nq, int32_t Nk, int32_t d) {
  const PrefillWorkspace p = plan_prefill_workspace(B, Hq, Hkv, Nk, d, 0, false);
  const int32_t split = chunk_kv_split(B, Hq, Hkv, Nk, Nq, d);
  if (split <= 1) return p.total;
  const int64_t rows = static_cast<int64_t>(B) * Hq * Nq;
  return p.total + chunk_partial_o_bytes(split, rows, d) + static_cast<size_t>(split) * rows * sizeof(float);
}

// The attention launch after the codes are in the workspace (plan p, table t): with use_v16
// V is read from the workspace's fp16 copy and its exponents, else from v (fp16).
static int prefill_attend(const PrefillWorkspace& p, const SeqTable& t, void* workspace, size_t workspace_bytes,
                          const void* v, int v_dtype, bool use_v16, int32_t B, int32_t Hq, int32_t Hkv, int32_t N,
                          int32_t d, const int32_t* cu_seqlens, int64_t total_tokens, int causal, void* out,
                          int out_dtype, float* lse_out, cudaStream_t s, int32_t q_off) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PrefillArgs a{};
  a.q_off = q_off;
  const int32_t dc = compute_dim(d);
  a.q_codes = reinterpret_cast<const uint16_t*>(ws + p.q_codes);
  a.q_scales = reinterpret_cast<const float*>(ws + p.q_scales);
  a.k_codes = reinterpret_cast<const uint16_t*>(ws + p.k_codes);
  a.k_scales = reinterpret_cast<const float*>(ws + p.k_scales);
  a.v = v;
  a.v_dtype = static_cast<sl8_dtype>(v_dtype);
  if (use_v16) {  // the padded / rescaled fp16 copy of V
    a.v16 = reinterpret_cast<const uint16_t*>(ws + p.v16);
    a.v_exp = reinterpret_cast<const int32_t*>(ws + p.v_exp);
  }
  a.varlen = cu_seqlens != nullptr;
  a.nseq = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.N = N;
  a.d = dc;
  a.d_io = d;
  a.total_tokens = a.varlen ? total_tokens : static_cast<int64_t>(B) * N;
  a.t_pad_max = p.t_pad_max;
  a.table = t;
  const int32_t item_rows = prefill_item_rows(dc, Hq / Hkv);
  a.dense_first = q_off / item_rows;
  a.dense_items = (N + item_rows - 1) / item_rows - a.dense_first;
  a.head_pairs = prefill_head_pairs(dc, Hq / Hkv);
  a.max_pairs = p.max_pairs;
  a.causal = causal != 0;
  a.out = out;
  a.out_dtype = static_cast<sl8_dtype>(out_dtype);
  a.lse = lse_out;
  a.logits = nullptr;
  a.kv_split = 1;
  // A query chunk on few items: split each item's keys so that the parts fill the GPU,
  // when the caller's workspace holds the partials (sl8_attn_int8_fwd_chunk_workspace_size).
  const int32_t split = q_off > 0 ? chunk_kv_split(B, Hq, Hkv, N, N - q_off, d) : 1;
  if (split > 1 && workspace_bytes >= chunk_workspace_bytes(B, Hq, Hkv, N - q_off, N, d)) {
    const int64_t rows = static_cast<int64_t>(B) * Hq * (N - q_off);
    a.kv_split = split;
    a.o_part = reinterpret_cast<float*>(ws + p.total);
    a.lse_part = reinterpret_cast<float*>(ws + p.total + chunk_partial_o_bytes(split, rows, d));
    a.out = nullptr;
    a.lse = nullptr;
    SL8_LAUNCH(launch_prefill(a, s));
    SL8_LAUNCH(launch_prefill_combine(a.o_part, a.lse_part, rows, d, split, out, static_cast<sl8_dtype>(out_dtype),
                                      lse_out, s));
    return SL8_OK;
  }
  SL8_LAUNCH(launch_prefill(a, s));
  return SL8_OK;
}

// Prefill over N keys per sequence; q_off > 0 (dense only): a query chunk of the last
// N - q_off positions, aligned bottom-right.
static int prefill_run(const void* q, const void* k, const void* v, int qk_dtype, int v_dtype, int32_t B, int32_t Hq,
                       int32_t Hkv, int32_t N, int32_t d, const int32_t* cu_seqlens, int64_t total_tokens, int causal,
                       int smooth_k, void* out, int out_dtype, float* lse_out, void* workspace, size_t workspace_bytes,
                       void* stream, int32_t q_off, const QuantGroups& groups = QuantGroups()) {
  int rc = validate_prefill(q, k, qk_dtype, B, Hq, Hkv, N, d);
  if (rc != SL8_OK) return rc;
  SL8_CHECK(v && out && aligned16(v) && aligned16(out), SL8_ERR_INVALID_ARG);
  SL8_CHECK(is_half(v_dtype), SL8_ERR_INVALID_ARG);
  SL8_CHECK(out_dtype == v_dtype || out_dtype == SL8_F32, SL8_ERR_INVALID_ARG);
  SL8_CHECK(!cu_seqlens || total_tokens >= 0, SL8_ERR_INVALID_ARG);
  SL8_CHECK(!cu_seqlens || total_tokens < (1ll << 31), SL8_ERR_UNSUPPORTED);
  SL8_CHECK(static_cast<int64_t>(B) * N < (1ll << 31), SL8_ERR_UNSUPPORTED);
  if (B == 0 || N == 0 || (cu_seqlens && total_tokens == 0)) return SL8_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PrefillWorkspace p;
  SeqTable t;
  rc = prefill_prepare(q, k, v, qk_dtype, v_dtype, B, Hq, Hkv, N, d, cu_seqlens, total_tokens, smooth_k, workspace,
                       workspace_bytes, s, false, &p, &t, q_off, groups);
  if (rc != SL8_OK) return rc;
  return prefill_attend(p, t, workspace, workspace_bytes, v, v_dtype, v_dtype == SL8_BF16 || compute_dim(d) != d, B,
                        Hq, Hkv, N, d, cu_seqlens, total_tokens, causal, out, out_dtype, lse_out, s, q_off);
}

int sl8_attn_int8_fwd(const void* q, const void* k, const void* v, int qk_dtype, int v_dtype, int32_t B, int32_t Hq,
                      int32_t Hkv, int32_t N, int32_t d, const int32_t* cu_seqlens, int64_t total_tokens,
                      int causal, int smooth_k, void* out, int out_dtype, float* lse_out, void* workspace,
                      size_t workspace_bytes, void* stream) {
  return prefill_run(q, k, v, qk_dtype, v_dtype, B, Hq, Hkv, N, d, cu_seqlens, total_tokens, causal, smooth_k, out,
                     out_dtype, lse_out, workspace, workspace_bytes, stream, 0);
}

size_t sl8_attn_int8_fwd_chunk_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t Nq, int32_t Nk, int32_t d) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < Nq || d <= 0) return 0;
  return chunk_workspace_bytes(B, Hq, Hkv, Nq, Nk, d);
}

int sl8_attn_int8_fwd_chunk(const void* q, const void* k, const void* v, int qk_dtype, int v_dtype, int32_t B,
                            int32_t Hq, int32_t Hkv, int32_t Nq, int32_t Nk, int32_t d, int causal, int smooth_k,
                            void* out, int out_dtype, float* lse_out, void* workspace, size_t workspace_bytes,
                            void* stream) {
  SL8_CHECK(Nq >= 0 && Nq <= Nk, SL8_ERR_INVALID_ARG);
  if (Nq == 0) return SL8_OK;
  return prefill_run(q, k, v, qk_dtype, v_dtype, B, Hq, Hkv, Nk, d, nullptr, 0, causal, smooth_k, out, out_dtype,
                     lse_out, workspace, workspace_bytes, stream, Nk - Nq);
}

int sl8_attn_int8_fwd_chunk_cache(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale,
                                  const int8_t* v_cache, const float* v_scale, int32_t B, int32_t Hq, int32_t Hkv,
                                  int32_t Nq, int32_t Nk, int32_t Lmax, int32_t d, int causal, void* out,
                                  int out_dtype, float* lse_out, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  SL8_CHECK(q && k_cache && k_scale && v_cache && v_scale && out, SL8_ERR_INVALID_ARG);
  SL8_CHECK(aligned16(q) && aligned16(k_cache) && aligned16(v_cache) && aligned16(out), SL8_ERR_INVALID_ARG);
  SL8_CHECK(is_half(q_dtype) && (is_half(out_dtype) || out_dtype == SL8_F32), SL8_ERR_INVALID_ARG);
  SL8_CHECK(B >= 0 && Hq > 0 && Hkv > 0 && d > 0 && Hq % Hkv == 0, SL8_ERR_INVALID_ARG);
  SL8_CHECK(Nq >= 0 && Nq <= Nk && Nk <= Lmax, SL8_ERR_INVALID_ARG);
  SL8_CHECK(d == 32 || head_dim_ok(d), SL8_ERR_UNSUPPORTED);  // head dim 32 runs as 64
  SL8_CHECK(Nk <= (1 << 24) && B <= (1 << 24) && static_cast<int64_t>(B) * Nk < (1ll << 31), SL8_ERR_UNSUPPORTED);
  if (B == 0 || Nq == 0) return SL8_OK;
  const PrefillWorkspace p = plan_prefill_workspace(B, Hq, Hkv, Nk, d, 0, false);
  SL8_CHECK(workspace && aligned16(workspace) && workspace_bytes >= p.total, SL8_ERR_WORKSPACE);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const SeqTable t = table_at(ws, p);
  const int32_t dc = compute_dim(d);
  // K and V codes from the cache (a plain launch: it follows every earlier reader of the
  // workspace in stream order), then the Q rows, then the attention
  SL8_LAUNCH(launch_cache_codes(k_cache, k_scale, v_cache, v_scale, B, Hkv, Nk, Lmax, dc, d, p.t_pad_max,
                                reinterpret_cast<uint16_t*>(ws + p.k_codes), reinterpret_cast<float*>(ws + p.k_scales),
                                reinterpret_cast<uint16_t*>(ws + p.v16), reinterpret_cast<int32_t*>(ws + p.v_exp), s));
  SL8_LAUNCH(launch_quant_qk(q, nullptr, static_cast<sl8_dtype>(q_dtype), false, B, Hq, Hkv, Nk, dc,
                             static_cast<int64_t>(B) * Nk, t, p.t_pad_max, nullptr, nullptr, p.max_chunks,
                             reinterpret_cast<uint16_t*>(ws + p.q_codes), reinterpret_cast<float*>(ws + p.q_scales),
                             reinterpret_cast<uint16_t*>(ws + p.k_codes), reinterpret_cast<float*>(ws + p.k_scales),
                             nullptr, nullptr, nullptr, s, Nk - Nq, d));
  return prefill_attend(p, t, workspace, workspace_bytes, nullptr, SL8_F16, true, B, Hq, Hkv, Nk, d, nullptr, 0,
                        causal, out, out_dtype, lse_out, s, Nk - Nq);
}

// Group sizes: powers of two from 1 to 64 (a group never leaves one 64-row CTA of the
// quantiser); the outlier ratio: finite and >= 0.
static int make_groups(int32_t q_group, int32_t k_group, float q_outlier_ratio, QuantGroups* g) {
  auto pow2 = [](int32_t x) { return x >= 1 && x <= 64 && (x & (x - 1)) == 0; };
  SL8_CHECK(pow2(q_group) && pow2(k_group), SL8_ERR_INVALID_ARG);
  SL8_CHECK(q_outlier_ratio >= 0.0f && q_outlier_ratio <= 3.0e38f, SL8_ERR_INVALID_ARG);  // also rejects NaN
  g->q_group = q_group;
  g->k_group = k_group;
  g->q_tau = q_outlier_ratio;
  return SL8_OK;
}

int sl8_attn_w8a8_fwd(const void* q, const void* k, const void* v, int qk_dtype, int v_dtype, int32_t B, int32_t Hq,
                      int32_t Hkv, int32_t N, int32_t d, const int32_t* cu_seqlens, int64_t total_tokens,
                      int causal, int smooth_k, int32_t q_group, int32_t k_group, float q_outlier_ratio, void* out,
                      int out_dtype, float* lse_out, void* workspace, size_t workspace_bytes, void* stream) {
  QuantGroups g;
  const int rc = make_groups(q_group, k_group, q_outlier_ratio, &g);
  if (rc != SL8_OK) return rc;
  return prefill_run(q, k, v, qk_dtype, v_dtype, B, Hq, Hkv, N, d, cu_seqlens, total_tokens, causal, smooth_k, out,
                     out_dtype, lse_out, workspace, workspace_bytes, stream, 0, g);
}

static int qk_logits_debug(const void* q, const void* k, int qk_dtype, int32_t B, int32_t Hq, int32_t Hkv, int32_t N,
                           int32_t d, const int32_t* cu_seqlens, int64_t total_tokens, int smooth_k,
                           int32_t row_begin, int32_t row_end, int32_t* logits_out, int8_t* q_codes, float* q_scales,
                           int8_t* k_codes, float* k_scales, void* workspace, size_t workspace_bytes, void* stream,
                           const QuantGroups& groups) {
  int rc = validate_prefill(q, k, qk_dtype, B, Hq, Hkv, N, d);
  if (rc != SL8_OK) return rc;
  const bool varlen = cu_seqlens != nullptr;
  SL8_CHECK(0 <= row_begin && row_begin <= row_end && row_end <= N, SL8_ERR_INVALID_ARG);
  SL8_CHECK(!varlen || total_tokens >= 0, SL8_ERR_INVALID_ARG);
  SL8_CHECK(!varlen || total_tokens < (1ll << 31), SL8_ERR_UNSUPPORTED);
  SL8_CHECK(static_cast<int64_t>(B) * N < (1ll << 31), SL8_ERR_UNSUPPORTED);
  SL8_CHECK(!q_codes == !q_scales && !k_codes == !k_scales, SL8_ERR_INVALID_ARG);
  if (B == 0 || N == 0 || (varlen && total_tokens == 0)) return SL8_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PrefillWorkspace p;
  SeqTable t;
  rc = prefill_prepare(q, k, nullptr, qk_dtype, qk_dtype, B, Hq, Hkv, N, d, cu_seqlens, total_tokens, smooth_k,
                       workspace, workspace_bytes, s, true, &p, &t, 0, groups);
  if (rc != SL8_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int32_t dc = compute_dim(d);
  if (q_codes)
    SL8_LAUNCH(launch_export_codes(reinterpret_cast<const uint16_t*>(ws + p.q_codes),
                                   reinterpret_cast<const float*>(ws + p.q_scales), varlen, B, Hq, N, dc, t,
                                   p.t_pad_max, q_codes, q_scales, s, d));
  if (k_codes)
    SL8_LAUNCH(launch_export_codes(reinterpret_cast<const uint16_t*>(ws + p.k_codes),
                                   reinterpret_cast<const float*>(ws + p.k_scales), varlen, B, Hkv, N, dc, t,
                                   p.t_pad_max, k_codes, k_scales, s, d));
  if (logits_out && row_end > row_begin) {
    PrefillArgs a{};
    a.q_codes = reinterpret_cast<const uint16_t*>(ws + p.q_codes);
    a.q_scales = reinterpret_cast<const float*>(ws + p.q_scales);
    a.k_codes = reinterpret_cast<const uint16_t*>(ws + p.k_codes);
    a.k_scales = reinterpret_cast<const float*>(ws + p.k_scales);
    // V is not used for logits; the V tiles are read from the Q code rows, a readable
    // [Hq >= Hkv][t_pad][d] fp16-sized region of the workspace
    a.v = nullptr;
    a.v_dtype = SL8_F16;
    a.v16 = reinterpret_cast<const uint16_t*>(ws + p.q_codes);
    a.varlen = varlen;
    a.nseq = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.N = N;
    a.d = dc;
    a.d_io = d;
    a.total_tokens = varlen ? total_tokens : static_cast<int64_t>(B) * N;
    a.t_pad_max = p.t_pad_max;
    a.table = t;
    a.dense_items = (N + prefill_item_rows(dc, Hq / Hkv) - 1) / prefill_item_rows(dc, Hq / Hkv);
    a.head_pairs = prefill_head_pairs(dc, Hq / Hkv);
    a.max_pairs = p.max_pairs;
    a.causal = false;
    a.out = nullptr;
    a.out_dtype = SL8_F32;
    a.lse = nullptr;
    a.logits = logits_out;
    a.row_begin = row_begin;
    a.row_end = row_end;
    SL8_LAUNCH(launch_prefill(a, s));
  }
  return SL8_OK;
}

int sl8_attn_int8_qk_logits_debug(const void* q, const void* k, int qk_dtype, int32_t B, int32_t Hq, int32_t Hkv,
                                  int32_t N, int32_t d, const int32_t* cu_seqlens, int64_t total_tokens, int smooth_k,
                                  int32_t row_begin, int32_t row_end, int32_t* logits_out, int8_t* q_codes,
                                  float* q_scales, int8_t* k_codes, float* k_scales, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return qk_logits_debug(q, k, qk_dtype, B, Hq, Hkv, N, d, cu_seqlens, total_tokens, smooth_k, row_begin, row_end,
                         logits_out, q_codes, q_scales, k_codes, k_scales, workspace, workspace_bytes, stream,
                         QuantGroups());
}

int sl8_attn_w8a8_qk_logits_debug(const void* q, const void* k, int qk_dtype, int32_t B, int32_t Hq, int32_t Hkv,
                                  int32_t N, int32_t d, const int32_t* cu_seqlens, int64_t total_tokens, int smooth_k,
                                  int32_t q_group, int32_t k_group, float q_outlier_ratio, int32_t row_begin,
                                  int32_t row_end, int32_t* logits_out, int8_t* q_codes, float* q_scales,
                                  int8_t* k_codes, float* k_scales, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  QuantGroups g;
  const int rc = make_groups(q_group, k_group, q_outlier_ratio, &g);
  if (rc != SL8_OK) return rc;
  return qk_logits_debug(q, k, qk_dtype, B, Hq, Hkv, N, d, cu_seqlens, total_tokens, smooth_k, row_begin, row_end,
                         logits_out, q_codes, q_scales, k_codes, k_scales, workspace, workspace_bytes, stream, g);
}

// The split plan.  split_size_for(Lmax, S, d) = ceil(Lmax / S) rounded up to a whole
// number of the decode kernel's stages (decode_chunk_tokens(d) tokens; to 16 tokens below
// one stage): every stage of the cache then starts on a 16-byte boundary of the scale
// rows, and only a sequence's last split ends in a partial stage.  A request n (0: about
// 10 work slots per SM over the B x Hkv pairs, at most one per stage) becomes
// S = ceil(Lmax / split_size_for(Lmax, n, d)) splits; the split kernel and the combine
// both use split_size_for(Lmax, S, d).
static int32_t split_size_for(int32_t Lmax, int32_t S, int32_t d) {
  const int32_t per = (Lmax + S - 1) / S;
  const int32_t chunk = decode_chunk_tokens(d);
  const int32_t step = per >= chunk ? chunk : 16;
  return (per + step - 1) / step * step;
}

int32_t sl8_attn_decode_num_splits(int32_t B, int32_t Hkv, int32_t Lmax, int32_t d, int32_t num_splits) {
  if (B <= 0 || Hkv <= 0 || Lmax <= 0 || !decode_head_dim_ok(d) || num_splits < 0) return 0;
  int64_t n = num_splits;
  if (n == 0) {
    const int64_t pairs = static_cast<int64_t>(B) * Hkv;
    n = (10ll * num_sms() + pairs - 1) / pairs;
    const int64_t chunks = (Lmax + decode_chunk_tokens(d) - 1) / decode_chunk_tokens(d);
    if (n > chunks) n = chunks;
  }
  const int64_t cap = (Lmax + 15) / 16;
  if (n > cap) n = cap;
  if (n < 1) n = 1;
  const int32_t ss = split_size_for(Lmax, static_cast<int32_t>(n), d);
  return (Lmax + ss - 1) / ss;
}

int32_t sl8_attn_decode_split_size(int32_t B, int32_t Hkv, int32_t Lmax, int32_t d, int32_t num_splits) {
  const int32_t S = sl8_attn_decode_num_splits(B, Hkv, Lmax, d, num_splits);
  return S > 0 ? split_size_for(Lmax, S, d) : 0;
}

size_t sl8_attn_decode_lse_offset(int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax, int32_t d, int32_t num_splits) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv) return 0;
  const int32_t S = sl8_attn_decode_num_splits(B, Hkv, Lmax, d, num_splits);
  if (S <= 0) return 0;
  return align_up(static_cast<size_t>(B) * Hq * S * d * sizeof(float), 256);
}

size_t sl8_attn_decode_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax, int32_t d,
                                      int32_t num_splits) {
  const size_t off = sl8_attn_decode_lse_offset(B, Hq, Hkv, Lmax, d, num_splits);
  if (!off) return 0;
  const int32_t S = sl8_attn_decode_num_splits(B, Hkv, Lmax, d, num_splits);
  return off + static_cast<size_t>(B) * Hq * S * sizeof(float);
}

// A paged cache (see DecodeArgs): the block table and the page geometry.
struct Paging {
  const int32_t* table;
  int32_t page_size, max_blocks, num_pages;
};

// Virtual kv heads per cache kv head: a work slot of the split kernel holds at most 8 query
// heads, so a kv head with G = Hq / Hkv > 8 query heads is split into the fewest equal
// groups of <= 8 (the smallest divisor ng of G with G / ng <= 8); each group streams the
// kv head's cache once.  1 for G <= 8.
static int32_t decode_kv_groups(int32_t Hq, int32_t Hkv) {
  const int32_t G = Hkv > 0 ? Hq / Hkv : 1;
  int32_t ng = (G + 7) / 8;
  while (ng < G && G % ng) ++ng;
  return ng < 1 ? 1 : ng;
}

static int decode_validate(const void* q, int q_dtype, const void* k_cache, const float* k_scale, const void* v_cache,
                           const float* v_scale, const int32_t* seqlens, int32_t B, int32_t Hq, int32_t Hkv,
                           int32_t Lmax, int32_t d, const Paging* pg, bool v16) {
  SL8_CHECK(q && k_cache && k_scale && v_cache && (v_scale || v16) && seqlens, SL8_ERR_INVALID_ARG);
  SL8_CHECK(!v16 || (d >= 64 && d <= 128 && !pg), SL8_ERR_UNSUPPORTED);
  SL8_CHECK(aligned16(q) && aligned16(k_cache) && aligned16(v_cache), SL8_ERR_INVALID_ARG);
  SL8_CHECK(q_dtype == SL8_F16 || q_dtype == SL8_BF16 || q_dtype == SL8_F32, SL8_ERR_INVALID_ARG);
  SL8_CHECK(B >= 0 && Hq > 0 && Hkv > 0 && Lmax >= 0 && d > 0, SL8_ERR_INVALID_ARG);
  SL8_CHECK(Hq % Hkv == 0, SL8_ERR_INVALID_ARG);
  SL8_CHECK(decode_head_dim_ok(d), SL8_ERR_UNSUPPORTED);
  SL8_CHECK(B <= 65535 && static_cast<int64_t>(Hkv) * decode_kv_groups(Hq, Hkv) <= 65535, SL8_ERR_UNSUPPORTED);
  if (pg) {
    // pages are loaded in 16-token units (TMA rows, 64-byte scale pieces)
    SL8_CHECK(pg->table && pg->page_size > 0 && pg->max_blocks > 0 && pg->num_pages > 0, SL8_ERR_INVALID_ARG);
    SL8_CHECK(pg->page_size % 16 == 0, SL8_ERR_UNSUPPORTED);
    SL8_CHECK(aligned16(k_scale) && aligned16(v_scale), SL8_ERR_INVALID_ARG);
    SL8_CHECK(static_cast<int64_t>(pg->num_pages) * Hkv * pg->page_size < (int64_t(1) << 31), SL8_ERR_UNSUPPORTED);
  } else {
    // the caches are addressed as [B * Hkv * Lmax] rows with 32-bit row coordinates
    SL8_CHECK(static_cast<int64_t>(B) * Hkv * Lmax < (int64_t(1) << 31), SL8_ERR_UNSUPPORTED);
  }
  return SL8_OK;
}

static int decode_launch(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale, const void* v_cache,
                         const float* v_scale, const int32_t* seqlens, int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax,
                         int32_t d, int32_t num_splits, float* o_partial, float* lse_partial, int32_t* logits,
                         int8_t* q_codes, float* q_scales, void* stream, const Paging* pg = nullptr,
                         bool v16 = false, int32_t verify_T = 0, const uint32_t* tree_mask = nullptr,
                         int32_t verify_dps = 1) {
  int rc = decode_validate(q, q_dtype, k_cache, k_scale, v_cache, v_scale, seqlens, B, Hq, Hkv, Lmax, d, pg, v16);
  if (rc != SL8_OK) return rc;
  SL8_CHECK(o_partial && lse_partial && num_splits >= 0, SL8_ERR_INVALID_ARG);
  if (B == 0 || Lmax == 0) return SL8_OK;
  DecodeArgs a{};
  a.q = q;
  a.q_dtype = static_cast<sl8_dtype>(q_dtype);
  a.k_cache = k_cache;
  a.k_scale = k_scale;
  a.v_cache = static_cast<const int8_t*>(v_cache);
  a.v_scale = v16 ? nullptr : v_scale;
  a.v16 = v16;
  a.verify_T = verify_T;
  a.tree_mask = tree_mask;
  a.verify_dps = verify_dps;
  a.verify_ng = verify_T ? (verify_T + verify_dps - 1) / verify_dps : 1;
  a.seqlens = seqlens;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Lmax = Lmax;
  a.d = d;
  a.split_size = sl8_attn_decode_split_size(B, Hkv, Lmax, d, num_splits);
  a.num_splits = sl8_attn_decode_num_splits(B, Hkv, Lmax, d, num_splits);
  SL8_CHECK(a.num_splits > 0 && a.num_splits <= 65535, SL8_ERR_UNSUPPORTED);
  // MQA beyond 8 query heads per kv head: virtual kv heads (the split plan above stays that
  // of the caller's Hkv, so the partials keep the size the queries report)
  a.kv_groups = decode_kv_groups(Hq, Hkv);
  a.Hkv = Hkv * a.kv_groups;
  a.o_partial = o_partial;
  a.lse_partial = lse_partial;
  a.logits = logits;
  a.q_codes = q_codes;
  a.q_scales = q_scales;
  if (pg) {
    a.block_table = pg->table;
    a.page_size = pg->page_size;
    a.max_blocks = pg->max_blocks;
    a.num_pages = pg->num_pages;
  }
  SL8_LAUNCH(launch_decode_split(a, static_cast<cudaStream_t>(stream)));
  return SL8_OK;
}

// Drafts per slot of the verify: as many as fit the 8 query columns beside their G heads.
static int32_t verify_dps(int32_t T, int32_t Hq, int32_t Hkv) {
  const int32_t G = Hkv > 0 ? Hq / Hkv : 1;
  const int32_t fit = G > 0 ? 8 / G : 1;
  return std::max<int32_t>(1, std::min<int32_t>(T, fit));
}

int32_t sl8_attn_decode_verify_num_splits(int32_t B, int32_t T, int32_t Hq, int32_t Hkv, int32_t Lmax, int32_t d,
                                          int32_t num_splits) {
  if (T < 1 || T > 32 || Hkv <= 0 || Hq % Hkv) return 0;
  const int32_t dps = verify_dps(T, Hq, Hkv);
  return sl8_attn_decode_num_splits(B * ((T + dps - 1) / dps), Hkv, Lmax, d, num_splits);
}

int sl8_attn_int8_decode_verify(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale,
                                 const int8_t* v_cache, const float* v_scale, const int32_t* seqlens,
                                 const uint32_t* tree_mask, int32_t T, int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax,
                                 int32_t d, int32_t num_splits, float* o_partial, float* lse_partial, void* out,
                                 int out_dtype, float* lse_out, void* stream) {
  SL8_CHECK(T >= 1 && T <= 32 && B >= 0, SL8_ERR_INVALID_ARG);
  SL8_CHECK(tree_mask && out, SL8_ERR_INVALID_ARG);
  SL8_CHECK(out_dtype == SL8_F16 || out_dtype == SL8_BF16 || out_dtype == SL8_F32, SL8_ERR_INVALID_ARG);
  SL8_CHECK(Hkv > 0 && Hq % Hkv == 0, SL8_ERR_INVALID_ARG);
  SL8_CHECK(Hq / Hkv <= 8, SL8_ERR_UNSUPPORTED);  // drafts share a slot's 8 query columns with their heads
  // the drafts of sequence b go dps at a time into one slot's query columns: virtual
  // sequences b * ng + group (q [B][T][Hq][d])
  const int32_t dps = verify_dps(T, Hq, Hkv), ng = (T + dps - 1) / dps;
  const int64_t bv = static_cast<int64_t>(B) * ng;
  SL8_CHECK(bv <= 65535 && static_cast<int64_t>(B) * T <= 65535, SL8_ERR_UNSUPPORTED);
  if (B == 0 || Lmax == 0) return SL8_OK;
  int rc = decode_launch(q, q_dtype, k_cache, k_scale, v_cache, v_scale, seqlens, static_cast<int32_t>(bv), Hq, Hkv,
                         Lmax, d, num_splits, o_partial, lse_partial, nullptr, nullptr, nullptr, stream, nullptr,
                         false, T, tree_mask, dps);
  if (rc != SL8_OK) return rc;
  const int32_t S = sl8_attn_decode_num_splits(static_cast<int32_t>(bv), Hkv, Lmax, d, num_splits);
  SL8_LAUNCH(launch_decode_combine(o_partial, lse_partial, seqlens, B * T, Hq, d, S, split_size_for(Lmax, S, d), out,
                                   static_cast<sl8_dtype>(out_dtype), lse_out, static_cast<cudaStream_t>(stream), T));
  return SL8_OK;
}

int sl8_attn_int8_decode_splitkv_f16v(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale,
                                      const void* v_cache, const int32_t* seqlens, int32_t B, int32_t Hq,
                                      int32_t Hkv, int32_t Lmax, int32_t d, int32_t num_splits, float* o_partial,
                                      float* lse_partial, void* stream) {
  return decode_launch(q, q_dtype, k_cache, k_scale, v_cache, nullptr, seqlens, B, Hq, Hkv, Lmax, d, num_splits,
                       o_partial, lse_partial, nullptr, nullptr, nullptr, stream, nullptr, true);
}

int sl8_attn_int8_paged_decode_splitkv(const void* q, int q_dtype, const int8_t* k_pages, const float* k_scale_pages,
                                       const int8_t* v_pages, const float* v_scale_pages, const int32_t* block_table,
                                       int32_t max_blocks, int32_t page_size, int32_t num_pages,
                                       const int32_t* seqlens, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                                       int32_t num_splits, float* o_partial, float* lse_partial, void* stream) {
  SL8_CHECK(max_blocks > 0 && page_size > 0, SL8_ERR_INVALID_ARG);
  const int64_t lmax = static_cast<int64_t>(max_blocks) * page_size;
  SL8_CHECK(lmax < (int64_t(1) << 31), SL8_ERR_UNSUPPORTED);
  const Paging pg{block_table, page_size, max_blocks, num_pages};
  return decode_launch(q, q_dtype, k_pages, k_scale_pages, v_pages, v_scale_pages, seqlens, B, Hq, Hkv,
                       static_cast<int32_t>(lmax), d, num_splits, o_partial, lse_partial, nullptr, nullptr, nullptr,
                       stream, &pg);
}

int sl8_attn_int8_decode_splitkv(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale,
                                 const int8_t* v_cache, const float* v_scale, const int32_t* seqlens, int32_t B,
                                 int32_t Hq, int32_t Hkv, int32_t Lmax, int32_t d, int32_t num_splits,
                                 float* o_partial, float* lse_partial, void* stream) {
  return decode_launch(q, q_dtype, k_cache, k_scale, v_cache, v_scale, seqlens, B, Hq, Hkv, Lmax, d, num_splits,
                       o_partial, lse_partial, nullptr, nullptr, nullptr, stream);
}

int sl8_attn_decode_combine(const float* o_partial, const float* lse_partial, const int32_t* seqlens, int32_t B,
                            int32_t Hq, int32_t Lmax, int32_t d, int32_t num_splits, void* out, int out_dtype,
                            float* lse_out, void* stream) {
  SL8_CHECK(o_partial && lse_partial && seqlens && out, SL8_ERR_INVALID_ARG);
  SL8_CHECK(out_dtype == SL8_F16 || out_dtype == SL8_BF16 || out_dtype == SL8_F32, SL8_ERR_INVALID_ARG);
  SL8_CHECK(B >= 0 && Hq > 0 && Lmax >= 0 && num_splits >= 1, SL8_ERR_INVALID_ARG);
  SL8_CHECK(decode_head_dim_ok(d), SL8_ERR_UNSUPPORTED);
  if (B == 0) return SL8_OK;
  SL8_CHECK(num_splits <= (Lmax > 0 ? Lmax : 1), SL8_ERR_INVALID_ARG);
  const int32_t split_size = Lmax > 0 ? split_size_for(Lmax, num_splits, d) : 16;
  SL8_LAUNCH(launch_decode_combine(o_partial, lse_partial, seqlens, B, Hq, d, num_splits, split_size, out,
                                   static_cast<sl8_dtype>(out_dtype), lse_out, static_cast<cudaStream_t>(stream)));
  return SL8_OK;
}

int sl8_attn_int8_decode_logits_debug(const void* q, int q_dtype, const int8_t* k_cache, const float* k_scale,
                                      const int8_t* v_cache, const float* v_scale, const int32_t* seqlens,
                                      int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax, int32_t d,
                                      int32_t* logits_out, int8_t* q_codes, float* q_scales, float* o_partial,
                                      float* lse_partial, void* stream) {
  SL8_CHECK(logits_out, SL8_ERR_INVALID_ARG);
  SL8_CHECK(!q_codes == !q_scales, SL8_ERR_INVALID_ARG);
  SL8_CHECK((reinterpret_cast<uintptr_t>(q_codes) & 3u) == 0, SL8_ERR_INVALID_ARG);  // written in 4-byte words
  return decode_launch(q, q_dtype, k_cache, k_scale, v_cache, v_scale, seqlens, B, Hq, Hkv, Lmax, d, 0, o_partial,
                       lse_partial, logits_out, q_codes, q_scales, stream);
}

int sl8_last_device_status(void* stream, int* site) {
  if (site) *site = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SL8_ERR_CUDA;
  DeviceStatus* p = device_status_ptr();
  if (!p) return SL8_ERR_CUDA;
  DeviceStatus h{};
  if (cudaMemcpy(&h, p, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return SL8_ERR_CUDA;
  if (h.code == kStatusOk) return SL8_OK;
  if (cudaMemset(p, 0, sizeof(DeviceStatus)) != cudaSuccess) return SL8_ERR_CUDA;
  if (site) *site = h.site;
  return h.code == kStatusTimeout ? SL8_ERR_TIMEOUT : SL8_ERR_DEVICE_ARG;
}

void sl8_set_spin_limit_ns(uint64_t limit_ns) {
  g_spin_limit_ns.store(limit_ns ? limit_ns : 1, std::memory_order_relaxed);
}
uint64_t sl8_get_spin_limit_ns(void) { return spin_limit_ns(); }

int sl8_selftest_timeout(uint64_t limit_ns, void* stream) {
  SL8_LAUNCH(launch_timeout_selftest(limit_ns, static_cast<cudaStream_t>(stream)));
  return SL8_OK;
}

void sl8_trace_enable(int on) { g_trace_on.store(on ? 1 : 0); }

int sl8_trace_collect(const char** names, int64_t* launches, double* total_ms, int max) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  int n = 0;
  for (const TraceRec& r : g_trace) {
    float ms = 0.0f;
    if (cudaEventSynchronize(r.stop) == cudaSuccess) cudaEventElapsedTime(&ms, r.start, r.stop);
    int i = 0;
    while (i < n && std::strcmp(names[i], r.name) != 0) ++i;
    if (i == n) {
      if (n == max) continue;
      names[n] = r.name;
      launches[n] = 0;
      total_ms[n] = 0.0;
      ++n;
    }
    launches[i] += 1;
    total_ms[i] += ms;
    g_event_pool.push_back(r.start);
    g_event_pool.push_back(r.stop);
  }
  g_trace.clear();
  return n;
}

}  // extern "C"
