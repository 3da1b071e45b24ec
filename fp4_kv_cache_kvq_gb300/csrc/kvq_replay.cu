// kvq_replay.cu -- replay of a toy multilayer sliding-window (SWA) network
// over a range of positions, rebuilding every layer's window state.
//
// Method: "Week 6 -- FP4 KV Caches and Bounded Replay", Core Concepts
// "Bounded replay" and Lab: the SWA state of a layer is the K and V of the last
// n_win positions; an exact replay must reach back n_win - 1 positions per
// layer below the top one (about L n_win tokens), a bounded replay starts only
// n_win back and accepts a small error in the upper layers.  The pages give
// the toy network no shapes; it is L layers of width d with one head each:
//   u_i = x_i / sqrt(mean(x_i^2) + 1e-6);  q_i, k_i, v_i = Wq u_i, Wk u_i, Wv u_i
//   a_i = sum_{s = max(0, i - n_win + 1)}^{i} softmax_s(q_i . k_s / sqrt(d)) v_s
//   x_i += Wo a_i
// with each layer's q, k, v taken from that layer's input.
//
// Work is data-parallel over positions.  Per layer:
//   swa_proj_kernel  8 positions and one of q, k, v per CTA, thread = output
//                    channel: the transposed weight copied to shared memory
//                    (cp.async) during the RMS normalisation (fixed-order
//                    reductions), then the projection; the last n_win
//                    positions' k, v also go to the caller's state array
//   swa_attn_kernel  8 positions per CTA, one warp each for the scores and
//                    the softmax: the window rows of all 8 are staged 32 at a
//                    time in shared memory (the next tile loaded into
//                    registers meanwhile) and each lane takes a row's dot
//                    product; the probabilities are laid out by row so that
//                    each V value loaded serves 4 positions; then Wo (copied
//                    to shared memory from the start) and the residual
//                    update in place
// A position's arithmetic depends only on its window's contents, in an order
// fixed by the offset within the window (rows outside a position's window
// enter its V sum with probability zero, which leaves the sum unchanged), so
// a replay from the exact start reproduces the whole sequence's state bit for
// bit.
#include "kvq_common.cuh"
#include "kvq_host.cuh"

namespace kvq {
namespace {

constexpr int kProjPos = 8;     // positions per projection CTA
constexpr int kMaxWin = 4096;   // largest window
constexpr int kAttnPos = 8;     // positions per attention CTA (a warp each)
constexpr int kAttnThreads = 32 * kAttnPos;
constexpr int kKTile = 32;      // window rows staged per tile (a lane each in the scores)
constexpr int kRowPad = 4;      // floats of padding per staged row

// Shared-memory floats of one attention CTA: query rows [P][D], a staged
// tile [kKTile][D + kRowPad], probabilities by row [n_win + P][P], the
// attention outputs by channel [D][P], the softmax sums [P], then the
// layer's transposed Wo [D][D] (every region a multiple of 4 floats).
__host__ __device__ constexpr int attn_smem_floats(int d, int n_win) {
  return kAttnPos * d + kKTile * (d + kRowPad) + (n_win + kAttnPos) * kAttnPos + d * kAttnPos + kAttnPos + d * d;
}

// 16-byte asynchronous copy global -> shared; a thread's copies are complete
// after cp_async_wait_all, and visible to the CTA after a barrier.
__device__ __forceinline__ void cp_async16(float* smem, const float* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Copy a [D][D] float matrix into shared memory, 16 bytes per copy, spread
// over `nthreads` threads.
template <int D>
__device__ __forceinline__ void stage_matrix(float* dst, const float* __restrict__ src, int nthreads) {
  for (int e = threadIdx.x; e < D * D / 4; e += nthreads) cp_async16(dst + 4 * e, src + 4 * e);
}

// wt[m][c][r] = w[m][r][c] for each d x d matrix m.
__global__ void transpose_kernel(const float* __restrict__ w, float* __restrict__ wt, int d) {
  __shared__ float tile[32][33];
  const size_t m = blockIdx.z;
  const float* src = w + m * d * d;
  float* dst = wt + m * d * d;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  for (int k = threadIdx.y; k < 32; k += 8) tile[k][threadIdx.x] = src[(size_t)(r0 + k) * d + c0 + threadIdx.x];
  __syncthreads();
  for (int k = threadIdx.y; k < 32; k += 8) dst[(size_t)(c0 + k) * d + r0 + threadIdx.x] = tile[threadIdx.x][k];
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Sum / max over the CTA (D threads), warps combined in index order; every
// thread gets the result.  `red` holds D / 32 floats.
template <int D>
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = red[0];
#pragma unroll
  for (int w = 1; w < D / 32; ++w) s += red[w];
  __syncthreads();
  return s;
}
template <int D>
__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = red[0];
#pragma unroll
  for (int w = 1; w < D / 32; ++w) s = fmaxf(s, red[w]);
  __syncthreads();
  return s;
}

// One of q, k, v (blockIdx.y = 0, 1, 2) for kProjPos positions from the
// layer input x; wt = this layer's transposed Wq, Wk, Wv ([3][D][D],
// wt[m][c][o] = W_m[o][c]).
template <int D>
__global__ void __launch_bounds__(D) swa_proj_kernel(const float* __restrict__ x, const float* __restrict__ wt,
                                                      float* __restrict__ qb, float* __restrict__ kb,
                                                      float* __restrict__ vb, float* __restrict__ st_k,
                                                      float* __restrict__ st_v, int64_t n, int n_win) {
  __shared__ float u[kProjPos][D];
  __shared__ float part[kProjPos][D / 32];
  extern __shared__ float4 proj_smem4[];
  float* wsm = reinterpret_cast<float*>(proj_smem4);  // [D][D]: wsm[c * D + o] = W_m[o][c]
  const int o = threadIdx.x, lane = o & 31, wp = o >> 5;
  const int m = blockIdx.y;
  stage_matrix<D>(wsm, wt + (size_t)m * D * D, D);  // in flight during the normalisation
  // the layer's kernels run as a chain of programmatic dependents: this one
  // reads x (and overwrites q, k, v) only once the previous kernel has
  // finished; the weights, transposed before the chain started, are staged
  // before that
  grid_dependency_wait();
  const int64_t i0 = (int64_t)blockIdx.x * kProjPos;
  float xv[kProjPos];
#pragma unroll
  for (int p = 0; p < kProjPos; ++p) {
    const int64_t i = i0 + p;
    xv[p] = i < n ? x[i * D + o] : 0.0f;
    const float s = warp_sum(xv[p] * xv[p]);
    if (lane == 0) part[p][wp] = s;
  }
  __syncthreads();
#pragma unroll
  for (int p = 0; p < kProjPos; ++p) {
    float ms = part[p][0];
#pragma unroll
    for (int w = 1; w < D / 32; ++w) ms += part[p][w];
    u[p][o] = xv[p] * (1.0f / sqrtf(ms / (float)D + 1e-6f));
  }
  cp_async_wait_all();  // this thread's part of W_m
  __syncthreads();
  float acc[kProjPos];
#pragma unroll
  for (int p = 0; p < kProjPos; ++p) acc[p] = 0.0f;
#pragma unroll 8
  for (int c = 0; c < D; ++c) {
    const float wc = wsm[c * D + o];
#pragma unroll
    for (int p = 0; p < kProjPos; ++p) acc[p] = fmaf(wc, u[p][c], acc[p]);
  }
  float* out = m == 0 ? qb : (m == 1 ? kb : vb);
  float* st = m == 1 ? st_k : (m == 2 ? st_v : nullptr);
#pragma unroll
  for (int p = 0; p < kProjPos; ++p) {
    const int64_t i = i0 + p;
    if (i >= n) break;
    out[i * D + o] = acc[p];
    const int64_t j = i - (n - n_win);  // row of the window state
    if (st != nullptr && j >= 0) st[j * D + o] = acc[p];
  }
}

// A tile of kKTile rows (from row R, rows past hi read as zeros) of a [n][D]
// array: NQ float4s per thread, thread t taking float4s t, t + 256, ...
template <int D>
__device__ __forceinline__ void load_tile_regs(const float* __restrict__ src, int64_t R, int64_t hi,
                                               float4 (&reg)[kKTile * D / 4 / kAttnThreads]) {
  constexpr int NQ = kKTile * D / 4 / kAttnThreads;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int e = threadIdx.x + q * kAttnThreads;
    const int rr = e / (D / 4), c4 = e % (D / 4);
    reg[q] = R + rr <= hi ? __ldg(reinterpret_cast<const float4*>(src + (R + rr) * D) + c4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}
template <int D>
__device__ __forceinline__ void store_tile_regs(float* tile, const float4 (&reg)[kKTile * D / 4 / kAttnThreads]) {
  constexpr int NQ = kKTile * D / 4 / kAttnThreads;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int e = threadIdx.x + q * kAttnThreads;
    const int rr = e / (D / 4), c4 = e % (D / 4);
    *reinterpret_cast<float4*>(tile + rr * (D + kRowPad) + 4 * c4) = reg[q];
  }
}

// Positions i0 .. i0 + kAttnPos - 1 (i0 = blockIdx.x * kAttnPos): softmax
// attention over each one's window, then x_i += Wo a_i (wot[c][o] =
// Wo[o][c]).  The CTA walks the union of the windows, rows lo .. hi.
template <int D>
__global__ void __launch_bounds__(kAttnThreads) swa_attn_kernel(float* __restrict__ x, const float* __restrict__ qb,
                                                                 const float* __restrict__ kb,
                                                                 const float* __restrict__ vb,
                                                                 const float* __restrict__ wot, int64_t n, int n_win,
                                                                 float scale) {
  constexpr int P = kAttnPos;
  constexpr int RS = D + kRowPad;  // staged row stride: float4 rows without bank conflicts
  constexpr int PG = P * D / kAttnThreads;  // positions per thread in PV and Wo (4 at D 128, 2 at 64)
  constexpr int NQ = kKTile * D / 4 / kAttnThreads;  // float4s of a staged tile per thread
  static_assert(NQ * kAttnThreads * 4 == kKTile * D, "tile split");
  extern __shared__ float4 smem4[];
  float* qs = reinterpret_cast<float*>(smem4);  // [P][D]
  float* tile = qs + P * D;                     // [kKTile][RS]
  float* pr = tile + kKTile * RS;               // [n_win + P][P]: probability of row lo + r for position p
  float* as = pr + (n_win + P) * P;             // [D][P]
  float* sums = as + D * P;                     // [P]
  float* wos = sums + P;                        // [D][D]: wos[c * D + o] = Wo[o][c]
  stage_matrix<D>(wos, wot, kAttnThreads);      // in flight until the Wo phase
  grid_dependency_wait();                       // see swa_proj_kernel
  const int tid = threadIdx.x, lane = tid & 31, p = tid >> 5;
  const int64_t i0 = (int64_t)blockIdx.x * P;
  const int64_t i = i0 + p;  // this warp's position
  const bool live = i < n;
  const int64_t s0 = live ? (i - n_win + 1 > 0 ? i - n_win + 1 : 0) : 0;  // its window: rows s0 .. i
  const int64_t lo = i0 - n_win + 1 > 0 ? i0 - n_win + 1 : 0;
  const int64_t hi = (i0 + P < n ? i0 + P : n) - 1;
  const int rows = (int)(hi - lo + 1);
  for (int e = tid; e < P * D; e += kAttnThreads) {
    const int64_t ii = i0 + e / D;
    qs[e] = ii < n ? qb[ii * D + e % D] : 0.0f;
  }
  for (int e = tid; e < rows * P; e += kAttnThreads) pr[e] = 0.0f;
  // ---- scores: lane = row of the staged tile, four channel chains.  The
  // next tile's rows are loaded into registers while this one is used.
  float4 reg[NQ];
  load_tile_regs<D>(kb, lo, hi, reg);
  for (int64_t R = lo; R <= hi; R += kKTile) {
    __syncthreads();  // the previous tile is consumed (first pass: qs and pr are set)
    store_tile_regs<D>(tile, reg);
    __syncthreads();
    if (R + kKTile <= hi) load_tile_regs<D>(kb, R + kKTile, hi, reg);
    const int64_t s = R + lane;
    if (live && s >= s0 && s <= i) {
      const float4* qr = reinterpret_cast<const float4*>(qs + p * D);
      const float4* kr = reinterpret_cast<const float4*>(tile + lane * RS);
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
      for (int c4 = 0; c4 < D / 4; ++c4) {
        const float4 a = qr[c4], b = kr[c4];
        a0 = fmaf(a.x, b.x, a0);
        a1 = fmaf(a.y, b.y, a1);
        a2 = fmaf(a.z, b.z, a2);
        a3 = fmaf(a.w, b.w, a3);
      }
      pr[(s - lo) * P + p] = ((a0 + a1) + (a2 + a3)) * scale;
    }
  }
  load_tile_regs<D>(vb, lo, hi, reg);  // the first V tile, in flight during the softmax
  __syncwarp();
  // ---- softmax of this warp's position: lane l takes window offsets l, l + 32, ...
  if (live) {
    const int len = (int)(i - s0 + 1);
    float* col = pr + (s0 - lo) * P + p;  // offset r at col[r * P]
    float mx = -INFINITY;
    for (int r = lane; r < len; r += 32) mx = fmaxf(mx, col[r * P]);
    mx = warp_max(mx);
    float sum = 0.0f;
    for (int r = lane; r < len; r += 32) {
      const float e = expf(col[r * P] - mx);
      col[r * P] = e;
      sum += e;
    }
    sum = warp_sum(sum);
    if (lane == 0) sums[p] = sum;
  } else if (lane == 0) {
    sums[p] = 1.0f;
  }
  __syncthreads();
  // ---- weighted sum of V: thread = (channel, group of PG positions), rows
  // in order, V staged a tile at a time like K
  const int c = tid % D, g = tid / D;
  float acc[PG];
#pragma unroll
  for (int k = 0; k < PG; ++k) acc[k] = 0.0f;
  for (int64_t R = lo; R <= hi; R += kKTile) {
    __syncthreads();  // the previous tile is consumed (first pass: the softmax is done)
    store_tile_regs<D>(tile, reg);
    __syncthreads();
    if (R + kKTile <= hi) load_tile_regs<D>(vb, R + kKTile, hi, reg);
    const int nr = hi - R + 1 < kKTile ? (int)(hi - R + 1) : kKTile;
    const float* pcol = pr + (R - lo) * P + g * PG;
#pragma unroll 8
    for (int r = 0; r < nr; ++r) {
      const float vv = tile[r * RS + c];
#pragma unroll
      for (int j = 0; j < PG; ++j) acc[j] = fmaf(pcol[r * P + j], vv, acc[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < PG; ++j) as[c * P + g * PG + j] = acc[j] / sums[g * PG + j];
  cp_async_wait_all();  // this thread's part of Wo
  __syncthreads();
  // ---- x_i += Wo a_i: thread = (output channel, the same positions)
  float y[PG];
#pragma unroll
  for (int j = 0; j < PG; ++j) y[j] = 0.0f;
#pragma unroll 8
  for (int cc = 0; cc < D; ++cc) {
    const float wv = wos[cc * D + c];
#pragma unroll
    for (int j = 0; j < PG; ++j) y[j] = fmaf(wv, as[cc * P + g * PG + j], y[j]);
  }
#pragma unroll
  for (int j = 0; j < PG; ++j) {
    const int64_t ii = i0 + g * PG + j;
    if (ii < n) x[ii * D + c] += y[j];
  }
}

template <int D>
kvq_status run_replay(const float* w, int layers, const float* emb, int64_t n, int n_win, float* states,
                      float* hidden, float* ws, cudaStream_t st) {
  float* xb = ws;
  float* qb = xb + n * D;
  float* kb = qb + n * D;
  float* vb = kb + n * D;
  float* wt = vb + n * D;
  transpose_kernel<<<dim3(D / 32, D / 32, 4 * layers), dim3(32, 8), 0, st>>>(w, wt, D);
  if (cudaMemcpyAsync(xb, emb, (size_t)n * D * sizeof(float), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return KVQ_ERR_CUDA;
  static DeviceOnce attr_set;  // the kernels' shared-memory opt-ins, once per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (attr_set.pending(dev)) {
    if (cudaFuncSetAttribute(swa_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             attn_smem_floats(D, kMaxWin) * (int)sizeof(float)) != cudaSuccess ||
        cudaFuncSetAttribute(swa_proj_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             D * D * (int)sizeof(float)) != cudaSuccess)
      return KVQ_ERR_CUDA;
    attr_set.mark(dev);
  }
  const float scale = 1.0f / sqrtf((float)D);
  const dim3 proj_grid((unsigned)((n + kProjPos - 1) / kProjPos), 3);
  const unsigned attn_grid = (unsigned)((n + kAttnPos - 1) / kAttnPos);
  const int attn_smem = attn_smem_floats(D, n_win) * (int)sizeof(float);
  // every kernel after the first is a programmatic dependent of the one
  // before it (the first follows the copy of the embeddings)
  auto launch = [&](auto kernel, dim3 grid, dim3 block, size_t smem, bool dependent, auto... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
  };
  for (int l = 0; l < layers; ++l) {
    const float* wl = wt + (size_t)4 * l * D * D;
    float* st_k = states + (size_t)(2 * l) * n_win * D;
    float* st_v = states + (size_t)(2 * l + 1) * n_win * D;
    if (launch(swa_proj_kernel<D>, proj_grid, dim3(D), D * D * sizeof(float), l > 0, (const float*)xb, wl, qb, kb,
               vb, st_k, st_v, n, n_win) != cudaSuccess ||
        launch(swa_attn_kernel<D>, dim3(attn_grid), dim3(kAttnThreads), (size_t)attn_smem, true, xb,
               (const float*)qb, (const float*)kb, (const float*)vb, wl + (size_t)3 * D * D, n, n_win, scale) !=
            cudaSuccess)
      return KVQ_ERR_CUDA;
  }
  if (hidden != nullptr &&
      cudaMemcpyAsync(hidden, xb, (size_t)n * D * sizeof(float), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return launch_status();
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" size_t kvq_swa_replay_workspace_bytes(int32_t layers, int64_t n, int32_t d) {
  if (layers < 1 || layers > 16383 || n < 1 || n > 0x7FFFFFFF || (d != 64 && d != 128)) return 0;
  return ((size_t)4 * (size_t)n * d + (size_t)4 * layers * d * d) * sizeof(float);
}

extern "C" kvq_status kvq_swa_replay(const float* w, int32_t layers, int32_t d, const float* emb, int64_t n,
                                     int32_t n_win, float* states, float* hidden, void* workspace,
                                     size_t workspace_bytes, kvq_stream stream) {
  if (w == nullptr || emb == nullptr || states == nullptr || workspace == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (d != 64 && d != 128) return KVQ_ERR_INVALID_ARGUMENT;
  if (layers < 1 || layers > 16383 || n < 1 || n > 0x7FFFFFFF) return KVQ_ERR_INVALID_ARGUMENT;
  if (n_win < 1 || n_win > kMaxWin || (int64_t)n_win > n) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned_to(w, 4) || !aligned_to(emb, 4) || !aligned_to(states, 4) || !aligned_to(workspace, 16) ||
      (hidden != nullptr && !aligned_to(hidden, 4)))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < kvq_swa_replay_workspace_bytes(layers, n, d)) return KVQ_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  float* ws = static_cast<float*>(workspace);
  return d == 128 ? run_replay<128>(w, layers, emb, n, n_win, states, hidden, ws, st)
                  : run_replay<64>(w, layers, emb, n, n_win, states, hidden, ws, st);
}
