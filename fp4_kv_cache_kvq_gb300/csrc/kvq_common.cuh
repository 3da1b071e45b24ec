// kvq_common.cuh -- device helpers shared by the libkvq kernels (sm_103a).
//
// Conversions use the Blackwell E2M1/E4M3 conversion instructions:
//   cvt.rn.satfinite.e2m1x2.f32   two fp32 -> packed E2M1 pair (RNE, saturating)
//   cvt.rn.f16x2.e2m1x2           packed E2M1 pair -> f16x2 (exact)
//   cvt.rn.satfinite.e4m3x2.f32   two fp32 -> packed E4M3 pair (RNE, saturating)
//   cvt.rn.f16x2.e4m3x2           packed E4M3 pair -> f16x2 (exact)
// In every packed form the first (low) element sits in the low nibble/byte and
// the low f16 half.  Waits on mbarriers are bounded by the global timer.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded waits give up after ~2 s

__device__ __forceinline__ void set_flag(int32_t* flag, int32_t bits) {
  if (flag != nullptr) atomicOr(flag, bits);
}

// Bounds-checked build (-DKVQ_DEBUG_BOUNDS): KVQ_IN(cond, flag) checks that an
// index or address range lies inside its buffer before the access; when it
// does not, it raises KVQ_FLAG_BOUNDS and yields false, and the caller skips
// the access (no trap).  In a normal build it is the constant true and cond is
// not evaluated.
#ifdef KVQ_DEBUG_BOUNDS
__device__ __forceinline__ bool bounds_ok(bool ok, int32_t* flag) {
  if (!ok) set_flag(flag, KVQ_FLAG_BOUNDS);
  return ok;
}
#define KVQ_IN(cond, flag) (::kvq::bounds_ok((cond), (flag)))
#else
#define KVQ_IN(cond, flag) (true)
#endif

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- conversions
// Two fp32 magnitudes (a -> low nibble, b -> high nibble) to a packed E2M1 pair.
__device__ __forceinline__ uint32_t e2m1x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u16.u8 %0, t;\n}\n"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// Two fp32 values to a packed E4M3 pair (lo -> low byte).
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One byte holding two E2M1 codes -> f16x2 (low nibble -> low half).
__device__ __forceinline__ uint32_t f16x2_from_e2m1x2(uint32_t byte) {
  uint32_t r;
  uint16_t in = (uint16_t)(byte & 0xFFu);
  asm("{\n .reg .b8 b0, b1;\n mov.b16 {b0, b1}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b0;\n}\n"
      : "=r"(r)
      : "h"(in));
  return r;
}

// The four bytes of a word (8 E2M1 codes) -> four f16x2, byte k -> r[k].  The
// word is split into byte registers for the conversions, which lets the
// conversion read each byte in place instead of shifting it down first.
__device__ __forceinline__ void f16x2x4_from_e2m1x8(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

// Transpose of an 8x8 b16 tile held in mma fragment layout (thread (g, t)
// holds row g, columns 2t and 2t+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Two E4M3 bytes (low byte -> low half) -> f16x2.
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t two_bytes) {
  uint32_t r;
  uint16_t in = (uint16_t)(two_bytes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(in));
  return r;
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h2) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = h2;
  return __half22float2(h);
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  uint32_t h2 = f16x2_from_e4m3x2(byte & 0xFFu);
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------- mbarrier / bulk copies
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory loads on 32-bit shared-window addresses.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];\n" : "=h"(v) : "r"(a));
  return v & 0xFFu;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

// Non-blocking test of a phase (no suspension at all).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// try_wait that lets the hardware suspend the thread for up to `hint_ns` while
// the phase is incomplete (instead of returning at once).
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Wait for the phase with the given parity to complete; false after ~2 s.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_hint(bar, parity, 1000000u)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait_hint(bar, parity, 1000000u)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// The same wait with an explicit limit in ns (used by the decode kernel's
// test instantiation, whose limit a test shortens).  A limit under 1 ms polls
// with the non-blocking test, so a phase that is not complete at the first
// test gives up after the limit (a suspending try_wait may itself wait for a
// hardware-chosen time and hide a short limit); longer limits poll like
// mbar_wait.
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const bool short_limit = limit_ns < 1000000ull;
  if (short_limit ? mbar_test_wait(bar, parity) : mbar_try_wait_hint(bar, parity, 1000000u)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (global_ns() - t0 > limit_ns) return false;
    if (short_limit ? mbar_test_wait(bar, parity) : mbar_try_wait_hint(bar, parity, 1000000u)) return true;
  }
}

// 1-D bulk copy global -> shared, completing bytes on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 3-D tiled tensor copy global -> shared, completing bytes on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            int32_t z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch: wait until the previous kernel in the stream
// has finished and its writes are visible / let the next kernel start launching.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- tensor-core MMA
// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- FP4 page-pool layout
// One group = min(page_size, 128) tokens of one kv head, stored as a
// contiguous block: K codes [G][D/2], K scales [G][D/16], V codes [G/2][D]
// (token pairs interleaved by nibble, 16-byte or 8-byte chunks permuted per
// row), V scales [G/2][D/16][2] (the two tokens of a pair side by side).
// 9*D/8 bytes per token.
struct Fp4Layout {
  int D, P, G, nb;
  int64_t group_bytes;
  __host__ __device__ Fp4Layout(int head_dim, int page_size)
      : D(head_dim), P(page_size), G(page_size < 128 ? page_size : 128), nb(head_dim / 16),
        group_bytes((int64_t)(page_size < 128 ? page_size : 128) * 9 * head_dim / 8) {}
  __host__ __device__ int64_t k_scales() const { return (int64_t)G * D / 2; }
  __host__ __device__ int64_t v_codes() const { return (int64_t)G * (D / 2 + nb); }
  __host__ __device__ int64_t v_scales() const { return (int64_t)G * (D + nb); }
  // byte offset of the group holding (physical page, kv head, slot)
  __host__ __device__ int64_t group(int64_t phys, int hkv, int h, int slot) const {
    return ((phys * hkv + h) * (P / G) + slot / G) * group_bytes;
  }
  // byte offset, inside a group, of the V scale of local token t, block j
  __host__ __device__ int64_t v_scale(int t, int j) const { return v_scales() + (int64_t)(t >> 1) * 2 * nb + 2 * j + (t & 1); }
  // byte offset, inside a group, of the 16 V-code bytes of channels [16j, 16j+16)
  // of token pair row i (the permutation keeps these 16 bytes contiguous)
  __host__ __device__ int64_t v_block(int i, int j) const {
    if (D == 64) return v_codes() + (int64_t)i * D + 8 * ((2 * j) ^ (((i >> 1) & 1) << 2));
    return v_codes() + (int64_t)i * D + 16 * (j ^ ((i & 3) << 1));
  }
};

// ---------------------------------------------------------------- host helpers
struct HostCheck {
  static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
};

}  // namespace kvq
