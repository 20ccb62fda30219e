// stack.cu -- link between stacked MoE layers: next-layer x (and h = [x, x]) from y.
//
// With norm on, each token is RMS-normalised with unit weight and eps inside the square
// root, the sum of squares in fp64 (README "kimi-k3-in-c", Part II section 5, RMSNorm);
// the result is rounded to fp32 and then to bf16 (nearest even).
#include <cuda_bf16.h>

#include "launch.h"

namespace k3 {
namespace {

__global__ void __launch_bounds__(256) k_stack_link(const float* __restrict__ y, int L, int norm,
                                                    float eps, uint16_t* __restrict__ x_out,
                                                    uint16_t* __restrict__ h_out) {
  __shared__ double wsum[8];
  const int t = blockIdx.x;
  const float* yr = y + (size_t)t * L;
  double inv = 1.0;
  if (norm) {
    double ss = 0.0;
    for (int c = threadIdx.x; c < L; c += blockDim.x) ss += (double)yr[c] * (double)yr[c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
    __syncthreads();
    double tot = 0.0;
    for (int w = 0; w < 8; ++w) tot += wsum[w];
    inv = 1.0 / sqrt(tot / (double)L + (double)eps);
  }
  for (int c = threadIdx.x; c < L; c += blockDim.x) {
    const float v = norm ? (float)((double)yr[c] * inv) : yr[c];
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    const uint16_t bits = *reinterpret_cast<const uint16_t*>(&b);
    x_out[(size_t)t * L + c] = bits;
    if (h_out) {
      h_out[(size_t)t * 2 * L + c] = bits;
      h_out[(size_t)t * 2 * L + L + c] = bits;
    }
  }
}

}  // namespace

cudaError_t launch_stack_link(const float* y, int T, int L, int norm, float eps, uint16_t* x_out,
                              uint16_t* h_out, cudaStream_t s) {
  return launch_kernel(k_stack_link, dim3(T), dim3(256), 0, s, false, y, L, norm, eps, x_out,
                       h_out);
}

}  // namespace k3
