// dense.cu -- the LatentMoE wrapper's dense layers around the routed experts (README
// "kimi-k3-in-c", Part II section 9, k3_moe): the down-projection of h into the experts'
// latent, the shared experts' gate and up rows on h, the RMSNorm of the routed aggregate
// (Part II section 5: eps inside the square root), and the
// up-projection together with the shared experts' down rows.  Every weight is bf16 and read
// once per call for a few tokens, so each launch streams its weights from HBM: a row is
// split into four quarters, one warp each, and every lane issues all its 16-byte loads of
// a batch before using them; the weights are constants of the layer, so each warp asks L2
// for its quarter before waiting on the preceding kernel.
#include <cuda_bf16.h>

#include "launch.h"

namespace k3 {
namespace {

constexpr int kDQ = 4;    // warps per weight row (quarters of the reduction)
constexpr int kDVec = 8;  // 16-byte weight pieces a lane keeps in flight per batch

struct Quarter {
  int qb, qe;  // [qb, qe) 8-element pieces of the row
};
__device__ __forceinline__ Quarter quarter_of(int n, int q) {
  const int nvec = n >> 3, qn = (nvec + kDQ - 1) / kDQ;
  const int qb = min(nvec, q * qn);
  return {qb, min(nvec, qb + qn)};
}

__device__ __forceinline__ void prefetch_quarter(const uint16_t* w, int n, int q) {
  const Quarter Q = quarter_of(n, q);
  if (Q.qe > Q.qb) prefetch_l2_bulk(w + (size_t)Q.qb * 8, (uint32_t)(Q.qe - Q.qb) * 16u);
}

// Quarter q of the bf16 row w (n elements, n % 8 == 0) against nt <= TT token vectors x
// (row stride xs elements; fp32 when XF, else bf16): acc[tt] = the warp's partial sum.
// Two fp32 partial sums per lane (even and odd elements), then the warp's sum.
template <int TT, bool XF>
__device__ __forceinline__ void quarter_dot(const uint16_t* __restrict__ w,
                                            const void* __restrict__ x, size_t xs, int nt,
                                            int n, int q, int lane, float (&acc)[TT]) {
  const Quarter Q = quarter_of(n, q);
  float a0[TT], a1[TT];
#pragma unroll
  for (int tt = 0; tt < TT; ++tt) a0[tt] = a1[tt] = 0.f;
  const uint4* w4 = reinterpret_cast<const uint4*>(w);
  for (int base = Q.qb; base < Q.qe; base += 32 * kDVec) {
    uint4 wv[kDVec];
#pragma unroll
    for (int i = 0; i < kDVec; ++i) {
      const int c = base + lane + 32 * i;
      wv[i] = c < Q.qe ? ldg_stream(w4 + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      if (tt >= nt) break;
#pragma unroll
      for (int i = 0; i < kDVec; ++i) {
        const int c = base + lane + 32 * i;
        if (c >= Q.qe) continue;
        if constexpr (XF) {
          const float4* xr =
              reinterpret_cast<const float4*>(static_cast<const float*>(x) + (size_t)tt * xs);
          const float4 p = __ldg(xr + 2 * c), r = __ldg(xr + 2 * c + 1);
          a0[tt] = fmaf(bf16lo(wv[i].x), p.x, a0[tt]);
          a1[tt] = fmaf(bf16hi(wv[i].x), p.y, a1[tt]);
          a0[tt] = fmaf(bf16lo(wv[i].y), p.z, a0[tt]);
          a1[tt] = fmaf(bf16hi(wv[i].y), p.w, a1[tt]);
          a0[tt] = fmaf(bf16lo(wv[i].z), r.x, a0[tt]);
          a1[tt] = fmaf(bf16hi(wv[i].z), r.y, a1[tt]);
          a0[tt] = fmaf(bf16lo(wv[i].w), r.z, a0[tt]);
          a1[tt] = fmaf(bf16hi(wv[i].w), r.w, a1[tt]);
        } else {
          const uint4* xr =
              reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + (size_t)tt * xs);
          const uint4 v = __ldg(xr + c);
          fma_bf16x2(wv[i].x, v.x, a0[tt], a1[tt]);
          fma_bf16x2(wv[i].y, v.y, a0[tt], a1[tt]);
          fma_bf16x2(wv[i].z, v.z, a0[tt], a1[tt]);
          fma_bf16x2(wv[i].w, v.w, a0[tt], a1[tt]);
        }
      }
    }
  }
#pragma unroll
  for (int tt = 0; tt < TT; ++tt) acc[tt] = warp_sum(a0[tt] + a1[tt]);
}

// quarter_dot for two rows of the same length against fp32 token vectors, every weight
// load of both rows issued before the first multiply; V 16-byte pieces per lane and row in
// a batch (six cover the quarter of a 6144-wide row in one batch, with registers left for
// three CTAs per SM).
template <int TT, int V = 6>
__device__ __forceinline__ void quarter_dot2(const uint16_t* __restrict__ w0,
                                             const uint16_t* __restrict__ w1,
                                             const float* __restrict__ x, size_t xs, int nt, int n,
                                             int q, int lane, float (&acc0)[TT],
                                             float (&acc1)[TT]) {
  const Quarter Q = quarter_of(n, q);
  float a0[TT], a1[TT], b0[TT], b1[TT];
#pragma unroll
  for (int tt = 0; tt < TT; ++tt) a0[tt] = a1[tt] = b0[tt] = b1[tt] = 0.f;
  const uint4 *u4 = reinterpret_cast<const uint4*>(w0), *v4 = reinterpret_cast<const uint4*>(w1);
  for (int base = Q.qb; base < Q.qe; base += 32 * V) {
    uint4 wu[V], wv[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int c = base + lane + 32 * i;
      wu[i] = c < Q.qe ? ldg_stream(u4 + c) : make_uint4(0u, 0u, 0u, 0u);
      wv[i] = c < Q.qe ? ldg_stream(v4 + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      if (tt >= nt) break;
      const float4* xr = reinterpret_cast<const float4*>(x + (size_t)tt * xs);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int c = base + lane + 32 * i;
        if (c >= Q.qe) continue;
        const float4 p = __ldg(xr + 2 * c), r = __ldg(xr + 2 * c + 1);
        a0[tt] = fmaf(bf16lo(wu[i].x), p.x, a0[tt]);
        a1[tt] = fmaf(bf16hi(wu[i].x), p.y, a1[tt]);
        a0[tt] = fmaf(bf16lo(wu[i].y), p.z, a0[tt]);
        a1[tt] = fmaf(bf16hi(wu[i].y), p.w, a1[tt]);
        a0[tt] = fmaf(bf16lo(wu[i].z), r.x, a0[tt]);
        a1[tt] = fmaf(bf16hi(wu[i].z), r.y, a1[tt]);
        a0[tt] = fmaf(bf16lo(wu[i].w), r.z, a0[tt]);
        a1[tt] = fmaf(bf16hi(wu[i].w), r.w, a1[tt]);
        b0[tt] = fmaf(bf16lo(wv[i].x), p.x, b0[tt]);
        b1[tt] = fmaf(bf16hi(wv[i].x), p.y, b1[tt]);
        b0[tt] = fmaf(bf16lo(wv[i].y), p.z, b0[tt]);
        b1[tt] = fmaf(bf16hi(wv[i].y), p.w, b1[tt]);
        b0[tt] = fmaf(bf16lo(wv[i].z), r.x, b0[tt]);
        b1[tt] = fmaf(bf16hi(wv[i].z), r.y, b1[tt]);
        b0[tt] = fmaf(bf16lo(wv[i].w), r.z, b0[tt]);
        b1[tt] = fmaf(bf16hi(wv[i].w), r.w, b1[tt]);
      }
    }
  }
#pragma unroll
  for (int tt = 0; tt < TT; ++tt) {
    acc0[tt] = warp_sum(a0[tt] + a1[tt]);
    acc1[tt] = warp_sum(b0[tt] + b1[tt]);
  }
}

// Everything that reads h: CTAs [0, ceil(L/2)) take two rows of `down` each (warps 0-3 and
// 4-7) and write z = bf16(down . h) (nearest even), the experts' latent input; CTAs
// [ceil(L/2), ceil(L/2) + SI) take row r of sh1 (warps 0-3) and of sh3 (warps 4-7) and write
// act[r] = activation(sh1[r] . h, sh3[r] . h) in fp32.  Grid y: groups of TT tokens.
template <int TT>
__global__ void __launch_bounds__(256) k_dense_in(const uint16_t* __restrict__ h, int T, int H,
                                                  const uint16_t* __restrict__ down, int L,
                                                  uint16_t* __restrict__ z,
                                                  const uint16_t* __restrict__ sh1,
                                                  const uint16_t* __restrict__ sh3, int SI,
                                                  float* __restrict__ act, int act_kind, float b1,
                                                  float b2) {
  __shared__ float part[8][TT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3, half = warp >> 2;
  const int ndown = (L + 1) >> 1;
  const bool is_down = (int)blockIdx.x < ndown;
  const int r = is_down ? 2 * (int)blockIdx.x + half : (int)blockIdx.x - ndown;
  const uint16_t* w = is_down ? (r < L ? down + (size_t)r * H : nullptr)
                              : (half == 0 ? sh1 : sh3) + (size_t)r * H;
  if (w && blockIdx.y == 0 && lane == 0) prefetch_quarter(w, H, q);
  pdl_wait();
  pdl_launch();
  const int t0 = blockIdx.y * TT, nt = min(TT, T - t0);
  float acc[TT];
#pragma unroll
  for (int tt = 0; tt < TT; ++tt) acc[tt] = 0.f;
  if (w) quarter_dot<TT, false>(w, h + (size_t)t0 * H, (size_t)H, nt, H, q, lane, acc);
  if (lane == 0)
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) part[warp][tt] = acc[tt];
  __syncthreads();
  const int i = threadIdx.x;
  if (is_down) {
    if (i < 2 * TT) {
      const int hf = i / TT, tt = i - hf * TT, rr = 2 * (int)blockIdx.x + hf;
      if (rr < L && tt < nt) {
        const float s = (part[4 * hf][tt] + part[4 * hf + 1][tt]) +
                        (part[4 * hf + 2][tt] + part[4 * hf + 3][tt]);
        const __nv_bfloat16 b = __float2bfloat16_rn(s);
        z[(size_t)(t0 + tt) * L + rr] = *reinterpret_cast<const uint16_t*>(&b);
      }
    }
  } else if (i < nt) {
    const float g = (part[0][i] + part[1][i]) + (part[2][i] + part[3][i]);
    const float u = (part[4][i] + part[5][i]) + (part[6][i] + part[7][i]);
    act[(size_t)(t0 + i) * SI + r] = activation(g, u, act_kind, b1, b2);
  }
}

// The RMSNorm of the routed aggregate y [T][L] (one CTA per token): yn = y * inv * w in fp32
// (w NULL: unit weight), inv = 1 / sqrt(mean(y^2) + eps), eps inside the square root as the
// README's k3_rmsnorm.  The README sums the squares in fp64; here they are summed in fp32
// by a fixed tree (each thread's elements pairwise, then the warp, then the warps), whose
// relative error, a few fp32 ulps times log2(L), stays far below the layer's tolerance: this
// kernel sits between two HBM-bound launches on the critical path, and an fp64 version
// measured 19 us on this GPU against a few us for this one.  norm 0: yn = y.
__global__ void __launch_bounds__(256) k_latent_norm(const float* __restrict__ y, int L, int norm,
                                                     const float* __restrict__ w, float eps,
                                                     float* __restrict__ yn) {
  __shared__ float wsum[8];
  pdl_wait();
  pdl_launch();
  const int t = blockIdx.x;
  const float* yr = y + (size_t)t * L;
  float inv = 1.f;
  if (norm) {
    // this thread's elements c = threadIdx.x + 256 i, added pairwise in a fixed order
    float sq[16];
    const int nmine = (L - (int)threadIdx.x + 255) / 256;
    float ss = 0.f;
    for (int i0 = 0; i0 < nmine; i0 += 16) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c = threadIdx.x + 256 * (i0 + i);
        const float v = i0 + i < nmine ? __ldg(yr + c) : 0.f;
        sq[i] = v * v;
      }
#pragma unroll
      for (int h = 8; h > 0; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) sq[i] += sq[i + h];
      ss += sq[0];
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
    __syncthreads();
    const float tot = ((wsum[0] + wsum[1]) + (wsum[2] + wsum[3])) +
                      ((wsum[4] + wsum[5]) + (wsum[6] + wsum[7]));
    inv = 1.0f / sqrtf(tot / (float)L + eps);
  }
  for (int c = threadIdx.x; c < L; c += blockDim.x)
    yn[(size_t)t * L + c] = norm ? yr[c] * inv * (w ? w[c] : 1.0f) : yr[c];
}

// out[t][r] = up[r] . yn[t] + sh2[r] . act[t]: two output rows per CTA, the up rows on warps
// 0-3 and the shared experts' down rows on warps 4-7 (idle without shared experts), each warp
// a quarter of both rows with all their loads in flight together (the up rows are short:
// one row's quarter alone left too few bytes in flight); the two sums are added last, each
// in a fixed order.  Grid y: groups of TT tokens.
template <int TT>
__global__ void __launch_bounds__(256, TT == 1 ? 3 : 1) k_dense_out(const float* __restrict__ yn, int T, int L,
                                                   const uint16_t* __restrict__ up, int H,
                                                   const float* __restrict__ act,
                                                   const uint16_t* __restrict__ sh2, int SI,
                                                   float* __restrict__ out) {
  __shared__ float part[2][8][TT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3, half = warp >> 2;
  const int r0 = 2 * blockIdx.x, r1 = min(r0 + 1, H - 1);  // an odd H repeats the last row
  const int n = half == 0 ? L : SI;
  const uint16_t* base = half == 0 ? up : (SI > 0 ? sh2 : nullptr);
  const uint16_t* w0 = base ? base + (size_t)r0 * n : nullptr;
  const uint16_t* w1 = base ? base + (size_t)r1 * n : nullptr;
  if (base && blockIdx.y == 0 && lane == 0) {
    prefetch_quarter(w0, n, q);
    prefetch_quarter(w1, n, q);
  }
  pdl_wait();
  pdl_launch();
  const int t0 = blockIdx.y * TT, nt = min(TT, T - t0);
  float acc0[TT], acc1[TT];
#pragma unroll
  for (int tt = 0; tt < TT; ++tt) acc0[tt] = acc1[tt] = 0.f;
  if (base)
    quarter_dot2<TT>(w0, w1, half == 0 ? yn + (size_t)t0 * L : act + (size_t)t0 * SI, (size_t)n,
                     nt, n, q, lane, acc0, acc1);
  if (lane == 0)
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      part[0][warp][tt] = acc0[tt];
      part[1][warp][tt] = acc1[tt];
    }
  __syncthreads();
  const int i = threadIdx.x;
  if (i < 2 * TT) {
    const int k = i / TT, tt = i - k * TT, r = r0 + k;
    if (r < H && tt < nt) {
      const float a = (part[k][0][tt] + part[k][1][tt]) + (part[k][2][tt] + part[k][3][tt]);
      const float b = (part[k][4][tt] + part[k][5][tt]) + (part[k][6][tt] + part[k][7][tt]);
      out[(size_t)(t0 + tt) * H + r] = a + b;
    }
  }
}

}  // namespace

cudaError_t launch_dense_in(const uint16_t* h, int T, int H, const uint16_t* down, int L,
                            uint16_t* z, const uint16_t* sh1, const uint16_t* sh3, int SI,
                            float* act, int act_kind, float b1, float b2, cudaStream_t s,
                            bool pdl) {
  const unsigned gx = (unsigned)((L + 1) / 2 + SI);
  if (T <= 2)
    return launch_kernel(k_dense_in<1>, dim3(gx, T), dim3(256), 0, s, pdl, h, T, H, down, L, z,
                         sh1, sh3, SI, act, act_kind, b1, b2);
  return launch_kernel(k_dense_in<4>, dim3(gx, (T + 3) / 4), dim3(256), 0, s, pdl, h, T, H, down,
                       L, z, sh1, sh3, SI, act, act_kind, b1, b2);
}

cudaError_t launch_latent_norm(const float* y, int T, int L, int norm, const float* w, float eps,
                               float* yn, cudaStream_t s, bool pdl) {
  return launch_kernel(k_latent_norm, dim3(T), dim3(256), 0, s, pdl, y, L, norm, w, eps, yn);
}

cudaError_t launch_dense_out(const float* yn, int T, int L, const uint16_t* up, int H,
                             const float* act, const uint16_t* sh2, int SI, float* out,
                             cudaStream_t s, bool pdl) {
  const unsigned gx = (unsigned)((H + 1) / 2);
  if (T <= 2)
    return launch_kernel(k_dense_out<1>, dim3(gx, T), dim3(256), 0, s, pdl, yn, T, L, up, H, act,
                         sh2, SI, out);
  return launch_kernel(k_dense_out<4>, dim3(gx, (T + 3) / 4), dim3(256), 0, s, pdl, yn, T, L, up,
                       H, act, sh2, SI, out);
}

}  // namespace k3
