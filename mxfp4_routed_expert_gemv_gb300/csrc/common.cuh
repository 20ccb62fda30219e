// common.cuh -- device helpers shared by the k3moe kernels (sm_103a).
//
// MXFP4 (README "kimi-k3-in-c", Part II section 4): a weight is E2M1[nibble] * 2^(s-127)
// with one E8M0 byte s per 32 consecutive weights of a row; the low nibble of a byte is the
// even column; s = 255 (NaN in the MX spec) makes the whole group zero.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "k3moe.h"

namespace k3 {

constexpr int kGroup = 32;          // weights per E8M0 scale
constexpr int kRowsPerHalf = 16;    // rows one half-warp reduces per step
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopk = 32;

// Status block slots (device int32[4]).
constexpr int kStatDropped = 0;
constexpr int kStatTimeout = 1;

// Bounded waits: an mbarrier wait gives up after this many polls (each poll is a
// try_wait that itself suspends for a hardware-chosen time), records a timeout in the
// status block and lets the kernel wind down instead of hanging.
constexpr uint32_t kWaitPolls = 1u << 22;

// ---- E8M0 and E2M1 decode --------------------------------------------------------

// 2^(s-127) as fp32 for every byte: s >= 1 is a normal (the exponent field itself),
// s == 0 is the subnormal 2^-127, s == 255 is zero (the group is silenced).
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  const uint32_t bits = (s == 0u) ? 0x00400000u : (s << 23);
  return (s == 255u) ? 0.0f : __uint_as_float(bits);
}

// Eight E2M1 weights (one 32-bit word: byte b holds columns 2b and 2b+1) times eight f16
// activations (x01..x67 as f16x2: low half = even column), accumulated into two fp32
// partial sums.  The hardware converts each nibble pair to an exact f16x2 (low nibble ->
// low half); every product of an E2M1 value and an f16 value is exact in fp32, so each
// fused multiply-add rounds only the sum.
__device__ __forceinline__ void dot8_e2m1_f16(uint32_t w, uint32_t x01, uint32_t x23,
                                              uint32_t x45, uint32_t x67, float& p0,
                                              float& p1) {
  asm("{\n\t"
      ".reg .b8 b0, b1, b2, b3;\n\t"
      ".reg .b32 h0, h1, h2, h3;\n\t"
      ".reg .f16 wl0, wh0, wl1, wh1, wl2, wh2, wl3, wh3;\n\t"
      ".reg .f16 xl0, xh0, xl1, xh1, xl2, xh2, xl3, xh3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %2;\n\t"
      "cvt.rn.f16x2.e2m1x2 h0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 h1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 h2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 h3, b3;\n\t"
      "mov.b32 {wl0, wh0}, h0;\n\t"
      "mov.b32 {wl1, wh1}, h1;\n\t"
      "mov.b32 {wl2, wh2}, h2;\n\t"
      "mov.b32 {wl3, wh3}, h3;\n\t"
      "mov.b32 {xl0, xh0}, %3;\n\t"
      "mov.b32 {xl1, xh1}, %4;\n\t"
      "mov.b32 {xl2, xh2}, %5;\n\t"
      "mov.b32 {xl3, xh3}, %6;\n\t"
      "fma.rn.f32.f16 %0, wl0, xl0, %0;\n\t"
      "fma.rn.f32.f16 %1, wh0, xh0, %1;\n\t"
      "fma.rn.f32.f16 %0, wl1, xl1, %0;\n\t"
      "fma.rn.f32.f16 %1, wh1, xh1, %1;\n\t"
      "fma.rn.f32.f16 %0, wl2, xl2, %0;\n\t"
      "fma.rn.f32.f16 %1, wh2, xh2, %1;\n\t"
      "fma.rn.f32.f16 %0, wl3, xl3, %0;\n\t"
      "fma.rn.f32.f16 %1, wh3, xh3, %1;\n\t"
      "}"
      : "+f"(p0), "+f"(p1)
      : "r"(w), "r"(x01), "r"(x23), "r"(x45), "r"(x67));
}

// Four nibble pairs (one 32-bit word) -> four exact f16x2 (low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t"
      ".reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t"
      "}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// acc += a * b with f16 operands and fp32 accumulation (exact product, one rounding).
__device__ __forceinline__ float fma_f16_f32(unsigned short a, unsigned short b, float acc) {
  asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(b));
  return acc;
}

// The 32 activations of one MX group as separate f16 halves, unpacked once and shared by
// every row that meets the group.
struct XHalves {
  unsigned short v[32];
  __device__ __forceinline__ explicit XHalves(const uint32_t (&x)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[2 * i] = (unsigned short)(x[i] & 0xffffu);
      v[2 * i + 1] = (unsigned short)(x[i] >> 16);
    }
  }
};

// One MX group of one row (16 bytes = 32 E2M1 weights) against pre-unpacked activations,
// unscaled; two accumulation chains.
__device__ __forceinline__ float dot32_halves(const uint4 w, const XHalves& x) {
  float p0 = 0.f, p1 = 0.f;
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h[4];
    e2m1x8_to_f16x2(words[q], h);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      p0 = fma_f16_f32((unsigned short)(h[b] & 0xffffu), x.v[8 * q + 2 * b], p0);
      p1 = fma_f16_f32((unsigned short)(h[b] >> 16), x.v[8 * q + 2 * b + 1], p1);
    }
  }
  return p0 + p1;
}

// One MX group: 32 E2M1 weights (16 bytes) dotted with 32 f16 activations (16 x f16x2),
// unscaled.
__device__ __forceinline__ float dot32_e2m1_f16(const uint4 w, const uint32_t (&x)[16]) {
  float p0 = 0.f, p1 = 0.f;
  dot8_e2m1_f16(w.x, x[0], x[1], x[2], x[3], p0, p1);
  dot8_e2m1_f16(w.y, x[4], x[5], x[6], x[7], p0, p1);
  dot8_e2m1_f16(w.z, x[8], x[9], x[10], x[11], p0, p1);
  dot8_e2m1_f16(w.w, x[12], x[13], x[14], x[15], p0, p1);
  return p0 + p1;
}

// ---- bf16 / f16 helpers ------------------------------------------------------------

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Mixed-precision dot step: acc += a (bf16) * b (bf16), exact product, one rounding.
__device__ __forceinline__ void fma_bf16x2(uint32_t a, uint32_t b, float& acc0, float& acc1) {
  asm("{\n\t"
      ".reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\t"
      "mov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.bf16 %1, ah, bh, %1;\n\t"
      "}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(a), "r"(b));
}

// Power-of-two exponent that brings a vector's largest magnitude m into [2^14, 2^15):
// x * 2^-e is then exact in f16 for every element within 2^28 of the maximum.
__device__ __forceinline__ int f16_exponent_for(float m) {
  if (!(m > 0.f) || !isfinite(m)) return 0;
  int e;
  frexpf(m, &e);  // m = f * 2^e, f in [0.5, 1)
  return e - 15;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);  // lo -> low half
  return *reinterpret_cast<const uint32_t*>(&h);
}

// v * 2^-e in two exact power-of-two steps (each factor is a normal float for any e the
// exponent helper returns).
struct Pow2Scale {
  float a, b;
  __device__ explicit Pow2Scale(int e) {
    const int e1 = -e / 2, e2 = -e - e1;
    a = __uint_as_float((uint32_t)(127 + e1) << 23);
    b = __uint_as_float((uint32_t)(127 + e2) << 23);
  }
  __device__ float operator()(float v) const { return (v * a) * b; }
};

// ---- memory helpers ------------------------------------------------------------------

// 16 bytes of data read once per call (weights): no L1 allocation, L2 evict-first.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile(
      "{\n\t.reg .b64 pol;\n\tcreatepolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], pol;\n\t}"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier + bulk copy (TMA, non-tensor) ----------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false (and counts a timeout) if the phase
// did not complete within kWaitPolls polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t phase, int32_t* status) {
  for (uint32_t i = 0; i < kWaitPolls; ++i)
    if (mbar_try_wait(bar, phase)) return true;
  if (status) atomicAdd(status + kStatTimeout, 1);
  return false;
}

// The same wait, which also gives up (without counting a timeout) once the CTA's abort flag
// is set, so that one role's failure winds the others down at once.  Only for waits on work
// whose completion the CTA does not need to see before it leaves: the waits that drain
// copies or MMAs still in flight use mbar_wait.
__device__ __forceinline__ bool mbar_wait_ab(uint64_t* bar, uint32_t phase, int32_t* status,
                                             volatile int* abort_v) {
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (mbar_try_wait(bar, phase)) return true;
    if (*abort_v) return false;
  }
  if (status) atomicAdd(status + kStatTimeout, 1);
  return false;
}

// Add `bytes` to the transaction count of the barrier's current phase without arriving (the
// phase completes once its arrivals are in and the count is back to zero).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;"
               ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// Bulk global -> shared copy of `bytes` (multiple of 16, both addresses 16-byte aligned),
// completing as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Named barrier among `nthreads` threads (multiple of 32), id != 0.
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch: wait for the preceding kernel's results / let the next
// kernel start its prologue.  Both are no-ops when the launch is not programmatic.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

// Bulk prefetch of `bytes` (a multiple of 16, from a 16-byte aligned address) into L2.  Only
// a hint: it returns at once and never changes what a later load reads.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)),
               "r"(bytes)
               : "memory");
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

// Reduce-scatter over the 16 lanes of a half-warp: on entry each lane holds v[0..15]
// (its partial of rows 0..15); on exit v[0] holds the full sum for row (lane & 15).
__device__ __forceinline__ void halfwarp_reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float give = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, give, off);
    }
  }
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

// 1/x from the hardware's approximate reciprocal (1 ulp; 1/inf = 0).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// SwiGLU with the hardware exponential and reciprocal (a few ulp of fp32, far below the
// activation terms' rounding); SiTU-GLU as in activation().
__device__ __forceinline__ float activation_fast(float g, float u, int act, float b1, float b2);

__device__ __forceinline__ float activation(float g, float u, int act, float b1, float b2) {
  if (act == K3MOE_ACT_SITU) {
    const float a = b1 * tanhf(g / b1) / (1.0f + expf(-g));  // sigmoid of the uncapped g
    return a * (b2 * tanhf(u / b2));
  }
  return silu_f32(g) * u;
}

__device__ __forceinline__ float activation_fast(float g, float u, int act, float b1, float b2) {
  if (act == K3MOE_ACT_SITU) return activation(g, u, act, b1, b2);
  return g * rcp_approx(1.0f + __expf(-g)) * u;
}

}  // namespace k3
