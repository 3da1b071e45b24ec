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
//   swa_proj_kernel  8 positions per CTA, thread = output channel: RMS
//                    normalisation (fixed-order reductions), q, k, v with the
//                    transposed weights read coalesced; the last n_win
//                    positions' k, v also go to the caller's state array
//   swa_attn_kernel  one CTA per position: window scores by warp dot
//                    products, softmax with fixed-order block reductions, the
//                    weighted sum of V, Wo, the residual update in place
// A position's arithmetic depends only on its window's contents, in an order
// fixed by the offset within the window, so a replay from the exact start
// reproduces the whole sequence's state bit for bit.
#include "kvq_common.cuh"
#include "kvq_host.cuh"

namespace kvq {
namespace {

constexpr int kProjPos = 8;     // positions per projection CTA
constexpr int kMaxWin = 4096;   // window positions held in shared memory

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

// q, k, v of kProjPos positions from the layer input x; wt = this layer's
// transposed Wq, Wk, Wv ([3][D][D], wt[m][c][o] = W_m[o][c]).
template <int D>
__global__ void __launch_bounds__(D) swa_proj_kernel(const float* __restrict__ x, const float* __restrict__ wt,
                                                      float* __restrict__ qb, float* __restrict__ kb,
                                                      float* __restrict__ vb, float* __restrict__ st_k,
                                                      float* __restrict__ st_v, int64_t n, int n_win) {
  __shared__ float u[kProjPos][D];
  __shared__ float part[kProjPos][D / 32];
  const int o = threadIdx.x, lane = o & 31, wp = o >> 5;
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
  __syncthreads();
  float q[kProjPos], k[kProjPos], v[kProjPos];
#pragma unroll
  for (int p = 0; p < kProjPos; ++p) q[p] = k[p] = v[p] = 0.0f;
#pragma unroll 4
  for (int c = 0; c < D; ++c) {
    const float wq = __ldg(wt + (size_t)(0 * D + c) * D + o);
    const float wk = __ldg(wt + (size_t)(1 * D + c) * D + o);
    const float wv = __ldg(wt + (size_t)(2 * D + c) * D + o);
#pragma unroll
    for (int p = 0; p < kProjPos; ++p) {
      const float uc = u[p][c];
      q[p] = fmaf(wq, uc, q[p]);
      k[p] = fmaf(wk, uc, k[p]);
      v[p] = fmaf(wv, uc, v[p]);
    }
  }
#pragma unroll
  for (int p = 0; p < kProjPos; ++p) {
    const int64_t i = i0 + p;
    if (i >= n) break;
    qb[i * D + o] = q[p];
    kb[i * D + o] = k[p];
    vb[i * D + o] = v[p];
    const int64_t j = i - (n - n_win);  // row of the window state
    if (j >= 0) {
      st_k[j * D + o] = k[p];
      st_v[j * D + o] = v[p];
    }
  }
}

// Position i = blockIdx.x: softmax attention over its window, then
// x_i += Wo a_i (wot[c][o] = Wo[o][c]).
template <int D>
__global__ void __launch_bounds__(D) swa_attn_kernel(float* __restrict__ x, const float* __restrict__ qb,
                                                      const float* __restrict__ kb, const float* __restrict__ vb,
                                                      const float* __restrict__ wot, int n_win, float scale) {
  constexpr int NW = D / 32;
  __shared__ float qs[D];
  __shared__ float as[D];
  __shared__ float sc[kMaxWin];
  __shared__ float red[NW];
  const int64_t i = blockIdx.x;
  const int o = threadIdx.x, lane = o & 31, wp = o >> 5;
  const int64_t s0 = i - n_win + 1 > 0 ? i - n_win + 1 : 0;
  const int len = (int)(i - s0 + 1);
  qs[o] = qb[i * D + o];
  __syncthreads();
  // scores: window offset r goes to warp r % NW, lanes split the channels
#pragma unroll 4
  for (int r = wp; r < len; r += NW) {
    const float* kr = kb + (s0 + r) * D;
    float acc = 0.0f;
#pragma unroll
    for (int m = 0; m < D / 32; ++m) acc = fmaf(qs[lane + 32 * m], __ldg(kr + lane + 32 * m), acc);
    acc = warp_sum(acc);
    if (lane == 0) sc[r] = acc * scale;
  }
  __syncthreads();
  float mx = -INFINITY;
  for (int r = o; r < len; r += D) mx = fmaxf(mx, sc[r]);
  mx = block_max<D>(mx, red);
  float sum = 0.0f;
  for (int r = o; r < len; r += D) {
    const float p = expf(sc[r] - mx);
    sc[r] = p;
    sum += p;
  }
  sum = block_sum<D>(sum, red);  // its barriers also publish the p values
  // weighted sum of V: four independent chains (window offset mod 4), joined
  // in a fixed order
  // (16 rows' loads issued before their multiply-adds)
  float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const float* vcol = vb + s0 * D + o;
  int r = 0;
  for (; r + 16 <= len; r += 16) {
    float vv[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) vv[k] = __ldg(vcol + (int64_t)(r + k) * D);
#pragma unroll
    for (int k = 0; k < 16; ++k) a4[k & 3] = fmaf(sc[r + k], vv[k], a4[k & 3]);
  }
  for (; r < len; ++r) a4[r & 3] = fmaf(sc[r], __ldg(vcol + (int64_t)r * D), a4[r & 3]);
  as[o] = ((a4[0] + a4[1]) + (a4[2] + a4[3])) / sum;
  __syncthreads();
  float y = 0.0f;
#pragma unroll 4
  for (int c = 0; c < D; ++c) y = fmaf(__ldg(wot + (size_t)c * D + o), as[c], y);
  x[i * D + o] += y;
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
  const float scale = 1.0f / sqrtf((float)D);
  const unsigned proj_grid = (unsigned)((n + kProjPos - 1) / kProjPos);
  for (int l = 0; l < layers; ++l) {
    const float* wl = wt + (size_t)4 * l * D * D;
    float* st_k = states + (size_t)(2 * l) * n_win * D;
    float* st_v = states + (size_t)(2 * l + 1) * n_win * D;
    swa_proj_kernel<D><<<proj_grid, D, 0, st>>>(xb, wl, qb, kb, vb, st_k, st_v, n, n_win);
    swa_attn_kernel<D><<<(unsigned)n, D, 0, st>>>(xb, qb, kb, vb, wl + (size_t)3 * D * D, n_win, scale);
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
