// Device helpers shared by the kernels of the routed NVFP4 MoE decode step
// (sm_103a).  Inline PTX for the pieces CUDA C++ does not expose directly:
// mbarriers, bulk async copies, programmatic dependent launch, and the
// hardware conversions to and from e2m1 / e4m3.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_decode_internal.h"

namespace moe {

// ------------------------------------------------------------------ errors

// Latch a device-side error code (first one wins); the host reads it with
// moe_decode_last_error.
__device__ __forceinline__ void latch_error(unsigned* err, unsigned code) {
  if (err) atomicCAS(err, 0u, code);
}

// Bounds-check builds (-DMOE_BOUNDS_CHECK) test every index that comes from
// data -- a pair id, a pooled position, a routed row -- before it addresses
// memory: a bad one latches kDevBadIndex and the access is skipped, where
// the normal build (in which the routing makes the indexes valid) compiles
// the test away.  A substitute for a memory sanitizer, which this device's
// pool does not offer.
#ifdef MOE_BOUNDS_CHECK
#define MOE_IN_BOUNDS(cond, err_word) ((cond) ? true : (latch_error((err_word), kDevBadIndex), false))
constexpr bool kBoundsCheck = true;
#else
#define MOE_IN_BOUNDS(cond, err_word) true
constexpr bool kBoundsCheck = false;
#endif

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// --------------------------------------------------- programmatic launches

// Wait until the grid this launch depends on has completed and its memory
// is visible.  A no-op when the launch carries no programmatic dependency.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the dependent grid start launching (its pre-wait prologue may run).
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity: gives up after limit_ns
// of wall time (the handle's wait limit, Workspace::wait_ns) and returns
// false (the caller latches an error and winds down without touching the
// stage).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u && global_ns() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------- bulk async copies

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// fp32 store that asks L2 to keep the line (results read back soon while
// streamed weights pass through L2 marked evict-first).
__device__ __forceinline__ void st_keep(float* p, float v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(policy) : "memory");
}

// Contiguous global -> shared copy completed on `bar` (complete_tx).  Both
// addresses 16-byte aligned, `bytes` a multiple of 16.  The weights are
// streamed once per step, so they are marked evict-first in L2.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Named barrier over the first `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Arrive on a named barrier without waiting for it.
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ----------------------------------------------------------- conversions

// Two fp32 values -> one byte of two e2m1 codes (`lo` in the low nibble),
// round to nearest even, saturating to +-6.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  unsigned short r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "mov.b16 %0, {t, 0};\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// fp32 -> e4m3 byte, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t cvt_e4m3(float v) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// Two e4m3 bytes (low byte first) -> two fp32 values (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_bytes) {
  uint32_t h2;
  const unsigned short in = static_cast<unsigned short>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  __half2 hv = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hv);
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) { return e4m3x2_to_f32x2(byte).x; }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Eight e2m1 codes (nibbles of w, element i in nibble i) -> eight signed
// bytes holding 2 * value (exact integers in [-12, 12]), elements 0..3 in
// `lo`, 4..7 in `hi`.  Magnitudes come from a byte-permute table lookup, the
// signs from the nibbles' top bits replicated by prmt's sign mode.
__device__ __forceinline__ void e2m1x8_to_s8x8(uint32_t w, uint32_t& lo, uint32_t& hi) {
  constexpr uint32_t kPosLo = 0x03020100u, kPosHi = 0x0C080604u;  // 0 1 2 3 | 4 6 8 12
  constexpr uint32_t kNegLo = 0xFDFEFF00u, kNegHi = 0xF4F8FAFCu;  // negated
  const uint32_t m = w & 0x77777777u;
  const uint32_t mh = m >> 16;
  const uint32_t pl = prmt(kPosLo, kPosHi, m), nl = prmt(kNegLo, kNegHi, m);
  const uint32_t ph = prmt(kPosLo, kPosHi, mh), nh = prmt(kNegLo, kNegHi, mh);
  const uint32_t w4 = w << 4;
  const uint32_t sl = prmt(w4, w, 0xD9C8u);  // 0xFF where nibbles 0..3 are negative
  const uint32_t sh = prmt(w4, w, 0xFBEAu);  // nibbles 4..7
  lo = (nl & sl) | (pl & ~sl);
  hi = (nh & sh) | (ph & ~sh);
}

// ------------------------------------------------------------- quantizer

// One block of 16 values of an NVFP4 tensor with global scale sg:
//   sb = e4m3(fp32(fp32(ab / 6) / sg)), d = fp32(dec(sb) * sg),
//   code_i = e2m1(fp32(v_i / d)); all codes 0 when sg == 0 or d == 0.
// Every division is IEEE round-to-nearest (never a reciprocal multiply).
__device__ __forceinline__ void quant_block16(const float (&v)[16], float sg, uint32_t& c_lo,
                                              uint32_t& c_hi, uint32_t& sb) {
  float ab = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(v[i]));
  sb = 0;
  float d = 0.0f;
  if (sg > 0.0f) {
    const float q = __fdiv_rn(ab, 6.0f);
    const float t = __fdiv_rn(q, sg);
    sb = cvt_e4m3(t);
    d = __fmul_rn(e4m3_to_f32(sb), sg);
  }
  uint32_t c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    c[i] = (d > 0.0f) ? cvt_e2m1x2(__fdiv_rn(v[2 * i], d), __fdiv_rn(v[2 * i + 1], d)) : 0u;
  c_lo = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
  c_hi = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
}

// Non-negative float bits order like the floats: atomicMax on them is an
// exact max.
__device__ __forceinline__ void atomic_max_nonneg(unsigned* addr, float v) {
  atomicMax(addr, __float_as_uint(v));
}

// fp32 dot product of eight bf16 pairs, accumulated in element order.
__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b, float acc) {
  const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa = __bfloat1622float2(pa[i]), fb = __bfloat1622float2(pb[i]);
    acc = fmaf(fa.x, fb.x, acc);
    acc = fmaf(fa.y, fb.y, acc);
  }
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace moe
