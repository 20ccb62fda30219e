// gemv.cu -- the expert input preparation for large batches and the standalone MXFP4
// mat-vec (README "kimi-k3-in-c", Part II section 4: y = W x straight from the packed
// nibbles and E8M0 scales, never expanded in memory).
#include "launch.h"

namespace k3 {
namespace {

// x (bf16) -> x16 (f16, scaled by 2^-xexp so the largest magnitude is in [2^14, 2^15)).
__global__ void __launch_bounds__(256) k_prep_x(const uint16_t* __restrict__ x, int L,
                                                __half* __restrict__ x16,
                                                int32_t* __restrict__ xexp) {
  pdl_wait();
  pdl_launch();
  __shared__ float wmax[8];
  const int t = blockIdx.x;
  const uint16_t* xr = x + (size_t)t * L;
  float m = 0.f;
  for (int c = threadIdx.x; c < L; c += blockDim.x) m = fmaxf(m, fabsf(__uint_as_float((uint32_t)xr[c] << 16)));
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  float mm = 0.f;
  for (int w = 0; w < 8; ++w) mm = fmaxf(mm, wmax[w]);
  const int xe = f16_exponent_for(mm);
  for (int c = threadIdx.x; c < L; c += blockDim.x)
    x16[(size_t)t * L + c] = __float2half_rn(ldexpf(__uint_as_float((uint32_t)xr[c] << 16), -xe));
  if (threadIdx.x == 0) xexp[t] = xe;
}

// Standalone MXFP4 mat-vec (one warp per row), the README's k3_matmul_mxfp4 statement on
// the GPU: y[r] = sum_g 2^(s_rg - 127) * sum_c E2M1[nib] * x[c].
__global__ void __launch_bounds__(256) k_matvec(float* __restrict__ y,
                                                const uint16_t* __restrict__ x,
                                                const uint8_t* __restrict__ packed,
                                                const uint8_t* __restrict__ scales, int in,
                                                int rows) {
  __shared__ float wmax[8];
  float m = 0.f;
  for (int c = threadIdx.x; c < in; c += blockDim.x) m = fmaxf(m, fabsf(__uint_as_float((uint32_t)x[c] << 16)));
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  float mm = 0.f;
  for (int w = 0; w < 8; ++w) mm = fmaxf(mm, wmax[w]);
  const int xe = f16_exponent_for(mm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + warp;
  if (r >= rows) return;
  const int G = in >> 5;
  float acc = 0.f;
  for (int g = lane; g < G; g += 32) {
    uint32_t xr[16];
    const uint32_t* xp = reinterpret_cast<const uint32_t*>(x + 32 * g);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const uint32_t v = xp[q];
      xr[q] = pack_half2(ldexpf(bf16lo(v), -xe), ldexpf(bf16hi(v), -xe));
    }
    const uint4 w = *reinterpret_cast<const uint4*>(packed + (size_t)r * (in >> 1) + 16 * g);
    acc += dot32_e2m1_f16(w, xr) * e8m0_to_f32(scales[(size_t)r * G + g]);
  }
  acc = warp_sum(acc);
  if (lane == 0) y[r] = ldexpf(acc, xe);
}

}  // namespace

cudaError_t launch_prep_x(const uint16_t* x, int T, int L, __half* x16, int32_t* xexp,
                          cudaStream_t s, bool pdl) {
  return launch_kernel(k_prep_x, dim3(T), dim3(256), 0, s, pdl, x, L, x16, xexp);
}

cudaError_t launch_matvec(float* y, const uint16_t* x, const uint8_t* packed,
                          const uint8_t* scales, int in, int rows, cudaStream_t s) {
  return launch_kernel(k_matvec, dim3((rows + 7) / 8), dim3(256), 0, s, false, y, x, packed,
                       scales, in, rows);
}

}  // namespace k3
