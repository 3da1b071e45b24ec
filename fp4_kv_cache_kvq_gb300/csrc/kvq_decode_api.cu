// kvq_decode_api.cu -- the C entry points of decode attention: workspace
// sizing, kvq_decode_attn, kvq_append_decode_attn (the append fused into
// the decode launch), kvq_decode_attn_tc and kvq_decode_attn_noalloc.
// Argument checks run on the host before anything is enqueued; a call
// enqueues the decode kernel (kvq_decode_kernel.cuh, instantiated in
// kvq_decode.cu, or kvq_decode_tc.cu), preceded by an append launch when the
// fused append falls back to one (the decode then runs as that launch's
// programmatic dependent), and the merge (kvq_merge.cu).
#include "kvq_common.cuh"
#include "kvq_decode.cuh"
#include "kvq_host.cuh"

#include <atomic>

namespace kvq {
namespace {

constexpr int kFuseMinChunksPerRange = 16;  // fused append only when a CTA's range is at least this long

// kvq_test_set_wait_limit_ns: the mma.sync decode kernel's work-wait limit
// in ns; 0 (the default) launches the production instantiation with the
// fixed kWaitLimitNs, anything else the test instantiation.
std::atomic<uint64_t> g_wait_limit_ns{0};

struct WsLayout {
  size_t rec_off, ml_off, o_off, total;
};

WsLayout ws_layout(int64_t batch, int64_t hkv, int64_t g, int64_t d, int64_t ctas) {
  WsLayout L;
  const int64_t units = batch * hkv;
  const int64_t slots = units + ctas;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  L.rec_off = 0;
  L.ml_off = up((size_t)units * sizeof(int2));
  L.o_off = L.ml_off + up((size_t)slots * g * 2 * sizeof(float));
  L.total = L.o_off + up((size_t)slots * g * d * sizeof(float));
  return L;
}

int decode_ctas() { return 3 * device_sm_count(); }

constexpr int kSmallRangeChunks = 8;

// The mma.sync decode grid: three CTAs per SM, or two when the cache's
// capacity (max_pages_per_seq * page_size, which the host knows) would give
// each of three per SM fewer than kSmallRangeChunks chunks -- then fewer,
// longer ranges mean fewer per-CTA prologues and fewer partials to merge
// (gqa_outliers, about 4.6 chunks per range at three per SM: 22.5 -> 20.5 us
// per call with L2 flushed; one per SM was slower, 23.6 us; at 9 chunks per
// range the two grids tie, at 18 three per SM wins).  The tcgen05 kernel
// always covers the ranges of three per SM.
int grid_ctas(const kvq_cache* c, int64_t batch, int64_t hkv, bool tcgen05) {
  const int full = decode_ctas();
  if (tcgen05 || full <= 0) return full;
  const int64_t cap = (int64_t)c->max_pages_per_seq * c->page_size;
  const int64_t cap_chunks = batch * hkv * ((cap + kChunk - 1) / kChunk);
  return cap_chunks < (int64_t)kSmallRangeChunks * full ? full / 3 * 2 : full;
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" size_t kvq_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_dim) {
  if (batch < 1 || num_kv_heads < 1 || num_q_heads < num_kv_heads || num_q_heads % num_kv_heads != 0 ||
      head_dim < 16)
    return 0;
  const int ctas = decode_ctas();
  if (ctas <= 0) return 0;
  return ws_layout(batch, num_kv_heads, num_q_heads / num_kv_heads, head_dim, ctas).total;
}

namespace {

// kvq_decode_attn, kvq_decode_attn_tc and kvq_append_decode_attn: the same
// checks, workspace, partials and merge; `tcgen05` picks the tensor-memory
// decode kernel (head_dim 128); k_new / v_new (non-null) fuse the append of
// every sequence's newest token into the decode kernel.
kvq_status decode_attn(const kvq_cache* global, const kvq_cache* swa, int32_t batch, int32_t num_q_heads,
                       const int32_t* d_seq_lens, const void* k_new, const void* v_new, const void* q,
                       float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                       int32_t* d_err_flag, kvq_stream stream, bool tcgen05) {
  if (batch < 1) return KVQ_ERR_INVALID_ARGUMENT;
  kvq_status st = check_cache(global, batch);
  if (st != KVQ_OK) return st;
  if (!is_fp4_layout(global)) return KVQ_ERR_INVALID_ARGUMENT;
  const int hkv = global->num_kv_heads, D = global->head_dim;
  if (num_q_heads < hkv || num_q_heads % hkv != 0) return KVQ_ERR_INVALID_ARGUMENT;
  const int g = num_q_heads / hkv;
  if (!(softmax_scale > 0.0f) || !(softmax_scale < 3.0e38f)) return KVQ_ERR_INVALID_ARGUMENT;
  if (d_seq_lens == nullptr || q == nullptr || out == nullptr || workspace == nullptr)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned_to(q, 16) || !aligned_to(out, 16) || !aligned_to(workspace, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  const bool fused = k_new != nullptr || v_new != nullptr;
  if (fused && (k_new == nullptr || v_new == nullptr || !aligned_to(k_new, 16) || !aligned_to(v_new, 16)))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (fused && (swa != nullptr || tcgen05)) return KVQ_ERR_UNSUPPORTED;
  if (swa != nullptr) {
    st = check_cache(swa, batch);
    if (st != KVQ_OK) return st;
    if (swa->format != KVQ_FORMAT_FP8_E4M3_HEAD || swa->num_kv_heads != hkv || swa->head_dim != D)
      return KVQ_ERR_INVALID_ARGUMENT;
  }
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if (tcgen05 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if (g > kNG) return KVQ_ERR_UNSUPPORTED;
  if (swa != nullptr && swa->page_size > kMaxWindow) return KVQ_ERR_UNSUPPORTED;
  const int ctas = grid_ctas(global, batch, hkv, tcgen05);
  if (ctas <= 0) return KVQ_ERR_CUDA;
  const WsLayout L = ws_layout(batch, hkv, g, D, ctas);
  if (workspace_bytes < L.total) return KVQ_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  DecodeParams dp = {};
  dp.lens = d_seq_lens;
  dp.page_table = global->page_table;
  dp.pool = static_cast<const uint8_t*>(global->data);
  dp.q = static_cast<const uint16_t*>(q);
  dp.part_o = reinterpret_cast<float*>(ws + L.o_off);
  dp.part_ml = reinterpret_cast<float*>(ws + L.ml_off);
  dp.unit_rec = reinterpret_cast<int2*>(ws + L.rec_off);
  dp.flag = d_err_flag;
  const bool nv = global->format == KVQ_FORMAT_NVFP4;
  dp.k_gscale = nv ? static_cast<const float*>(global->k_scale) : nullptr;
  dp.v_gscale = nv ? static_cast<const float*>(global->v_scale) : nullptr;
  dp.num_pages = global->num_pages;
  dp.batch = batch;
  dp.hkv = hkv;
  dp.g = g;
  dp.hq = num_q_heads;
  dp.page = global->page_size;
  dp.max_pages = global->max_pages_per_seq;
  dp.window = swa ? swa->page_size : 0;
  dp.head_dim = D;
  dp.pool_bytes = global->num_pages * (int64_t)hkv * global->page_size * 9 * D / 8;
  dp.n_slots = (int64_t)batch * hkv + ctas;
  dp.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  dp.qk_log2 = softmax_scale * kLog2e;
  dp.k_new = fused ? static_cast<const uint16_t*>(k_new) : nullptr;
  dp.v_new = fused ? static_cast<const uint16_t*>(v_new) : nullptr;
  dp.cache = *global;
  dp.nvfp4 = nv ? 1 : 0;
  bool after_append = false;  // the decode follows its own append launch (small caches)
  if (fused) {
    // The producer warp's appends hide behind a CTA's first copies only when
    // its range is long; with short ranges (judged from the cache's capacity,
    // which the host knows) the append runs as its own launch first -- the
    // same quantiser, so the same bytes -- and the decode is launched as its
    // programmatic dependent: its CTAs start (barriers, range walk, query
    // rows) while the append runs, and its producer waits for the append
    // before the first copy.
    const int64_t cap = (int64_t)global->max_pages_per_seq * global->page_size;
    const int64_t cap_chunks = (int64_t)batch * hkv * ((cap + kChunk - 1) / kChunk);
    if (cap_chunks < (int64_t)kFuseMinChunksPerRange * ctas) {
      st = launch_fp4_append(global, batch, 1, d_seq_lens, -1, dp.k_new, dp.v_new, d_err_flag, s);
      if (st != KVQ_OK) return st;
      dp.k_new = dp.v_new = nullptr;
      after_append = true;
    }
  }
  if (tcgen05)
    st = launch_decode_tc(dp, s);
  else if (dp.wait_ns != 0)
    st = launch_decode_mma_test_wait(dp, s, ctas, after_append);
  else
    st = launch_decode_mma(dp, s, ctas, after_append);
  if (st != KVQ_OK) return st;

  MergeParams mp;
  mp.lens = d_seq_lens;
  mp.q = dp.q;
  mp.part_o = dp.part_o;
  mp.part_ml = dp.part_ml;
  mp.unit_rec = dp.unit_rec;
  mp.out = out;
  mp.flag = d_err_flag;
  mp.k8 = swa ? static_cast<const uint8_t*>(swa->data) : nullptr;
  mp.v8 = swa ? static_cast<const uint8_t*>(swa->v_data) : nullptr;
  mp.k8_scale = swa ? static_cast<const float*>(swa->k_scale) : nullptr;
  mp.v8_scale = swa ? static_cast<const float*>(swa->v_scale) : nullptr;
  mp.window = swa ? swa->page_size : 0;
  mp.hkv = hkv;
  mp.g = g;
  mp.hq = num_q_heads;
  mp.head_dim = D;
  mp.qk_log2 = dp.qk_log2;
  mp.n_slots = dp.n_slots;
  mp.batch = batch;
  return launch_merge(mp, (int64_t)batch * hkv, s);
}

}  // namespace

extern "C" kvq_status kvq_decode_attn(const kvq_cache* global, const kvq_cache* swa, int32_t batch,
                                      int32_t num_q_heads, const int32_t* d_seq_lens, const void* q,
                                      float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                                      int32_t* d_err_flag, kvq_stream stream) {
  return decode_attn(global, swa, batch, num_q_heads, d_seq_lens, nullptr, nullptr, q, softmax_scale, out,
                     workspace, workspace_bytes, d_err_flag, stream, false);
}

extern "C" kvq_status kvq_append_decode_attn(const kvq_cache* global, int32_t batch, int32_t num_q_heads,
                                             const int32_t* d_seq_lens, const void* k_new, const void* v_new,
                                             const void* q, float softmax_scale, float* out, void* workspace,
                                             size_t workspace_bytes, int32_t* d_err_flag, kvq_stream stream) {
  if (k_new == nullptr || v_new == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  return decode_attn(global, nullptr, batch, num_q_heads, d_seq_lens, k_new, v_new, q, softmax_scale, out,
                     workspace, workspace_bytes, d_err_flag, stream, false);
}

extern "C" kvq_status kvq_decode_attn_tc(const kvq_cache* global, const kvq_cache* swa, int32_t batch,
                                         int32_t num_q_heads, const int32_t* d_seq_lens, const void* q,
                                         float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                                         int32_t* d_err_flag, kvq_stream stream) {
  return decode_attn(global, swa, batch, num_q_heads, d_seq_lens, nullptr, nullptr, q, softmax_scale, out,
                     workspace, workspace_bytes, d_err_flag, stream, true);
}

// ------------------------------------------------------------------ decode without caller scratch
// For callers that may not allocate device memory on their call path (see the
// header).  The workspace lives in a fixed device array that every GPU loading
// this library holds until the process exits; calls share it.
#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (host code cannot use the array's name as a device address).
kvq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return KVQ_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attn_noalloc(const kvq_cache* global, const kvq_cache* swa, int32_t batch,
                                              int32_t num_q_heads, const int32_t* d_seq_lens, const void* q,
                                              float softmax_scale, float* out, int32_t* d_err_flag,
                                              kvq_stream stream) {
  if (global == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  const size_t need = kvq_decode_workspace_bytes(batch, num_q_heads, global->num_kv_heads, global->head_dim);
  if (need == 0) return KVQ_ERR_INVALID_ARGUMENT;
  if (need > kNoAllocScratchBytes) return KVQ_ERR_WORKSPACE;
  void* scratch = nullptr;
  const kvq_status st = scratch_address(&scratch);
  if (st != KVQ_OK) return st;
  return kvq_decode_attn(global, swa, batch, num_q_heads, d_seq_lens, q, softmax_scale, out, scratch,
                         kNoAllocScratchBytes, d_err_flag, stream);
}

extern "C" void kvq_test_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns, std::memory_order_relaxed); }
