// kvq_merge.cu -- the merge of the decode kernels' per-range partials into
// the attention output, and (with an FP8 sliding window) the window's own
// attention terms folded into the same softmax.
//
// Method: "Quantising the KV cache", section "Code" (the quantised K/V feed an
// unchanged attention) and "Week 6 -- FP4 KV Caches and Bounded Replay"
// (recent positions kept at FP8): the output of a (sequence, kv head) unit is
// softmax over the union of its FP4 positions (split over CTA ranges) and its
// window positions, combined by the log-sum-exp rule
//   M = max m_i,  o = sum_i e^(m_i - M) o_i / sum_i e^(m_i - M) l_i.
// Both merges launch as programmatic dependents of the decode kernel: their
// grids may be scheduled as decode CTAs retire, and they wait
// (griddepcontrol.wait) before reading the partials; the window merge does
// its window terms before that wait.
#include "kvq_common.cuh"
#include "kvq_decode.cuh"
#include "kvq_host.cuh"

namespace kvq {
namespace {


// Merge without a window: one CTA per unit, thread (row r, 4 channels) takes
// float4 partials.  The unit's record and length load together, then the
// partials in batches of kMergeBatch whose loads are all in flight at once:
// two L2 round trips for up to kMergeBatch splits.
constexpr int kMergeBatch = 8;
template <int D>
__global__ void __launch_bounds__(kNG * D / 4) merge_splits_kernel(const MergeParams p) {
  grid_dependency_wait();  // the decode grid has finished and its partials are visible
  const int u = blockIdx.x;
  const int b = u / p.hkv, h = u % p.hkv;
  const int r = threadIdx.x / (D / 4), c4 = threadIdx.x % (D / 4);
  if (r >= p.g) return;
  int2 rec = __ldg(p.unit_rec + u);  // loaded beside the length (unused when T == 0)
  int32_t T = __ldg(p.lens + b);
  if (T < 0) {
    if (threadIdx.x == 0 && h == 0) set_flag(p.flag, KVQ_FLAG_BAD_LENGTH);
    T = 0;
  }
  const int64_t qrow = (int64_t)b * p.hq + (int64_t)h * p.g + r;
  if (!KVQ_IN(b < p.batch, p.flag)) return;
  float4* dst = reinterpret_cast<float4*>(p.out + qrow * D) + c4;
  if (T > 0 && !KVQ_IN(rec.x >= 0 && rec.y >= 0 && (int64_t)rec.x + rec.y <= p.n_slots, p.flag)) rec.y = 0;
  if (T == 0) {
    *dst = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  // the unit's partials, kMergeBatch at a time with every load of a batch
  // in flight together: the batch's maximum first, then one rescale of the
  // sums so far (online log-sum-exp merge)
  float mx = -INFINITY;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.0f;
  for (int k0 = 0; k0 < rec.y; k0 += kMergeBatch) {
    float2 ml[kMergeBatch];
    float4 ov[kMergeBatch];
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      const int k = min(k0 + j, rec.y - 1);  // past the end: a repeat, masked below
      const int64_t sl = (int64_t)(rec.x + k) * p.g + r;
      ml[j] = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + sl);
      ov[j] = __ldcg(reinterpret_cast<const float4*>(p.part_o + sl * D) + c4);
      if (k0 + j >= rec.y) ml[j].x = -INFINITY;
    }
    float mb = ml[0].x;
#pragma unroll
    for (int j = 1; j < kMergeBatch; ++j) mb = fmaxf(mb, ml[j].x);
    const float mn = fmaxf(mx, mb);
    if (mn == -INFINITY) continue;  // no position of this unit so far
    const float a = mx == -INFINITY ? 0.0f : fast_exp2(mx - mn);
    o = make_float4(o.x * a, o.y * a, o.z * a, o.w * a);
    l *= a;
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      const float f = ml[j].x == -INFINITY ? 0.0f : fast_exp2(ml[j].x - mn);
      o.x = fmaf(f, ov[j].x, o.x);
      o.y = fmaf(f, ov[j].y, o.y);
      o.z = fmaf(f, ov[j].z, o.z);
      o.w = fmaf(f, ov[j].w, o.w);
      l = fmaf(f, ml[j].y, l);
    }
    mx = mn;
  }
  const float inv = l > 0.0f ? 1.0f / l : 0.0f;
  *dst = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
}

// Merge with the FP8 window: CTAs of 256 threads, one per (unit, slice of
// the group's query rows: 2 rows at head_dim 128, 4 at 64).
//   scores: thread (token t, row half) takes window token t for its rows (its
//           K row read once as uint4s; fp32 x^ = E4M3(c) * s_h, fp32 dot
//           products in channel order);
//   softmax per row, a warp each;
//   PV:     the window's V is staged 128 tokens at a time in shared memory
//           (coalesced uint4 loads, token order); thread (channel c, row
//           group) accumulates its rows over the tile;
// then the log-sum-exp merge of the window with the unit's FP4 partials.
constexpr int kWinThreads = 256;
// CTAs per unit, each a slice of the query rows (every thread keeps at least
// one row in the scores and in PV)
template <int D>
__host__ __device__ constexpr int win_row_split() { return D == 128 ? 4 : 2; }
constexpr int kWinTile = 128;  // window tokens staged per V tile

template <int D>
__global__ void __launch_bounds__(kWinThreads) merge_window_kernel(const MergeParams p) {
  constexpr int kRows = kNG / win_row_split<D>();             // query rows of this CTA
  constexpr int kRowsQK = kRows / (kWinThreads / kWinTile);  // query rows per thread in the scores
  constexpr int kGroupsPV = kWinThreads / D;                 // row groups in PV
  constexpr int kRowsPV = kRows / kGroupsPV;                 // query rows per thread in PV
  static_assert(kRowsQK >= 1 && kRowsPV >= 1, "row split");
  extern __shared__ float wsm[];
  const int W = p.window;
  float* qs = wsm;                                   // [kRows][D] fp32 query rows
  float* sc = qs + kRows * D;                        // [kRows][W] scores, then probabilities
  float* stat = sc + kRows * W;                      // [kRows] max, [kRows] sum
  uint8_t* vt = reinterpret_cast<uint8_t*>(stat + 2 * kRows);  // [kWinTile][D] V codes
  const int g = max(0, min(kRows, p.g - (int)blockIdx.y * kRows));  // rows of this CTA
  const int u = blockIdx.x;
  const int b = u / p.hkv, h = u % p.hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (!KVQ_IN(b < p.batch, p.flag)) return;  // the whole CTA: its rings and rows
  int32_t T = __ldg(p.lens + b);
  if (T < 0) {
    if (tid == 0 && h == 0) set_flag(p.flag, KVQ_FLAG_BAD_LENGTH);
    T = 0;
  }
  const int w = min(W, T);
  const int nch = (T - w + kChunk - 1) / kChunk;
  if (g == 0) return;
  const int rbase = blockIdx.y * kRows;  // first row of the group handled here
  const int64_t qrow0 = (int64_t)b * p.hq + (int64_t)h * p.g + rbase;
  for (int i = tid; i < kRows * D; i += kWinThreads)
    qs[i] = i < g * D ? __uint_as_float((uint32_t)p.q[qrow0 * D + i] << 16) : 0.0f;
  __syncthreads();
  const int64_t ring = ((int64_t)b * p.hkv + h) * W;
  const int first = ((T - w) % W + W) % W;  // ring slot of the window's first token
  if (w > 0) {
    const float sk = __ldg(p.k8_scale + h);
    const int r0 = (tid / kWinTile) * kRowsQK;
    for (int t = tid % kWinTile; t < w; t += kWinTile) {
      const int slot = first + t < W ? first + t : first + t - W;
      const uint4* krow = reinterpret_cast<const uint4*>(p.k8 + (ring + slot) * D);
      uint4 kc[D / 16];
#pragma unroll
      for (int c16 = 0; c16 < D / 16; ++c16) kc[c16] = __ldg(krow + c16);
      float acc[kRowsQK];
#pragma unroll
      for (int r = 0; r < kRowsQK; ++r) acc[r] = 0.0f;
#pragma unroll
      for (int c16 = 0; c16 < D / 16; ++c16) {
        const uint32_t ws4[4] = {kc[c16].x, kc[c16].y, kc[c16].z, kc[c16].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 f = f16x2_to_float2(f16x2_from_e4m3x2((ws4[j >> 1] >> (16 * (j & 1))) & 0xFFFFu));
          const float x0 = f.x * sk, x1 = f.y * sk;
          const int ch = 16 * c16 + 2 * j;
#pragma unroll
          for (int r = 0; r < kRowsQK; ++r)
            acc[r] = fmaf(qs[(r0 + r) * D + ch + 1], x1, fmaf(qs[(r0 + r) * D + ch], x0, acc[r]));
        }
      }
#pragma unroll
      for (int r = 0; r < kRowsQK; ++r)
        if (r0 + r < g) sc[(r0 + r) * W + t] = acc[r] * p.qk_log2;
    }
    __syncthreads();
    for (int r = warp; r < g; r += kWinThreads / 32) {
      float mx = -INFINITY;
      for (int t = lane; t < w; t += 32) mx = fmaxf(mx, sc[r * W + t]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      float sum = 0.0f;
      for (int t = lane; t < w; t += 32) {
        const float e = fast_exp2(sc[r * W + t] - mx);
        sc[r * W + t] = e;
        sum += e;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
      if (lane == 0) {
        stat[r] = mx;
        stat[kRows + r] = sum;
      }
    }
  }
  const int c = tid % D, rp = (tid / D) * kRowsPV;
  float ow[kRowsPV];
#pragma unroll
  for (int r = 0; r < kRowsPV; ++r) ow[r] = 0.0f;
  if (w > 0) {
    const float sv = __ldg(p.v8_scale + h);
    for (int t0 = 0; t0 < w; t0 += kWinTile) {
      const int n = min(kWinTile, w - t0);
      __syncthreads();  // scores and stats published; the previous tile consumed
      for (int i = tid; i < n * (D / 16); i += kWinThreads) {
        const int t = i / (D / 16), c16 = i % (D / 16);
        const int slot = first + t0 + t < W ? first + t0 + t : first + t0 + t - W;
        reinterpret_cast<uint4*>(vt + t * D)[c16] = __ldg(reinterpret_cast<const uint4*>(p.v8 + (ring + slot) * D) + c16);
      }
      __syncthreads();
#pragma unroll 8
      for (int t = 0; t < n; ++t) {
        const float x = e4m3_to_f32(vt[t * D + c]) * sv;
#pragma unroll
        for (int r = 0; r < kRowsPV; ++r) ow[r] = fmaf(sc[(rp + r) * W + t0 + t], x, ow[r]);
      }
    }
  }
  grid_dependency_wait();  // the window's terms are done; now the decode grid's partials
  int2 rec = nch > 0 ? __ldg(p.unit_rec + u) : make_int2(0, 0);
  if (!KVQ_IN(rec.x >= 0 && rec.y >= 0 && (int64_t)rec.x + rec.y <= p.n_slots, p.flag)) rec = make_int2(0, 0);
#pragma unroll
  for (int r = 0; r < kRowsPV; ++r) {
    const int row = rp + r;
    if (row >= g) break;
    const float mw = w > 0 ? stat[row] : -INFINITY;
    float mx = mw;
    for (int k = 0; k < rec.y; ++k) mx = fmaxf(mx, __ldcg(p.part_ml + ((int64_t)(rec.x + k) * p.g + rbase + row) * 2));
    float o = 0.0f, l = 0.0f;
    if (mx != -INFINITY) {
      if (mw != -INFINITY) {
        const float f = fast_exp2(mw - mx);
        o = f * ow[r];
        l = f * stat[kRows + row];
      }
      for (int k = 0; k < rec.y; ++k) {
        const int64_t sl = (int64_t)(rec.x + k) * p.g + rbase + row;
        const float m = __ldcg(p.part_ml + sl * 2);
        if (m == -INFINITY) continue;
        const float f = fast_exp2(m - mx);
        o = fmaf(f, __ldcg(p.part_o + sl * D + c), o);
        l = fmaf(f, __ldcg(p.part_ml + sl * 2 + 1), l);
      }
    }
    p.out[(qrow0 + row) * D + c] = l > 0.0f ? o / l : 0.0f;
  }
}

// ------------------------------------------------------------------ host side
// Launch a merge kernel as a programmatic dependent of the decode kernel just
// enqueued on the stream: its grid may be scheduled as the decode's CTAs
// retire (the decode releases dependents at its start), and it runs
// griddepcontrol.wait before it reads the decode's partials.
template <typename... Args>
cudaError_t launch_dependent(void (*kernel)(Args...), dim3 grid, dim3 block, int smem, cudaStream_t s,
                             const MergeParams& mp) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, mp);
}

int window_smem_bytes(int d, int window) {
  const int rows = kNG / (d == 128 ? win_row_split<128>() : win_row_split<64>());
  return (rows * d + rows * window + 2 * rows) * (int)sizeof(float) + kWinTile * d;
}

template <int D>
kvq_status launch_window_merge(const MergeParams& mp, cudaStream_t s, int smem, int64_t units) {
  static DeviceOnce attr_set;  // opt in to the largest window's shared memory, once per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (attr_set.pending(dev)) {
    if (cudaFuncSetAttribute(merge_window_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             window_smem_bytes(D, kMaxWindow)) != cudaSuccess)
      return KVQ_ERR_CUDA;
    attr_set.mark(dev);
  }
  const cudaError_t e =
      launch_dependent(merge_window_kernel<D>, dim3((unsigned)units, win_row_split<D>()), dim3(kWinThreads), smem, s, mp);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace

kvq_status launch_merge(const MergeParams& mp, int64_t units, cudaStream_t s) {
  if (mp.k8 == nullptr) {
    const cudaError_t e =
        mp.head_dim == 128
            ? launch_dependent(merge_splits_kernel<128>, dim3((unsigned)units), dim3(kNG * 128 / 4), 0, s, mp)
            : launch_dependent(merge_splits_kernel<64>, dim3((unsigned)units), dim3(kNG * 64 / 4), 0, s, mp);
    return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
  }
  const int wsmem = window_smem_bytes(mp.head_dim, mp.window);
  return mp.head_dim == 128 ? launch_window_merge<128>(mp, s, wsmem, units)
                            : launch_window_merge<64>(mp, s, wsmem, units);
}

}  // namespace kvq
