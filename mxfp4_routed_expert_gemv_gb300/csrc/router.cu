// router.cu -- router GEMV and the per-token top-k with gates.
//
// README "kimi-k3-in-c", Part II section 9 "Picking 16 experts of 896": the unbiased score
// is sigmoid(h . Wr[e]); the selection score adds the correction bias; the top-k is taken
// by repeated arg-max where a tie goes to the lower expert index; the combine weights come
// from the unbiased scores, renormalised over the chosen k and multiplied by routed_scale.
#include "launch.h"
#include "mxq.cuh"
#include "tc.cuh"
#include "tmap.h"
#include "topk.cuh"

namespace k3 {
namespace {

constexpr int kQuarters = 4;      // warps per row, each a quarter of the hidden width
constexpr int kRpcFew = 2;        // router rows per CTA for one or two tokens
constexpr int kTopkBlockMaxTokens = 1 << 20;  // block-per-token top-k up to this batch
constexpr int kVecPerLane = 8;    // 16-byte pieces a lane keeps in flight per batch

// logits[t][e] = sum_i h[t][i] * wr[e][i].  A CTA holds 2 rows; each row is split into 4
// quarters, one warp each, and every lane issues all its 16-byte loads of a batch before
// using them, so a row's bytes are in flight at once.  Products of bf16 values are exact;
// each fused add rounds once (fp32).  The 4 quarter sums are added in a fixed order.
// With xq set (one token), warps 0 .. L/32-1 of the grid also write the token's x as kTerms
// MXFP4 terms (rows 0 .. kTerms-1 of xq / xsf), and CTA 0 zeroes `zero` [nzero]: work that
// does not depend on the routing, done here so that no separate launch is spent on it.
template <int TT, int RPC>
__global__ void __launch_bounds__(RPC * kQuarters * 32) k_router_logits(const uint16_t* __restrict__ h,
                                                       const uint16_t* __restrict__ wr, int T,
                                                       int E, int H,
                                                       float* __restrict__ logits,
                                                       const uint16_t* __restrict__ x, int L,
                                                       uint8_t* __restrict__ xq,
                                                       uint8_t* __restrict__ xsf,
                                                       int32_t* __restrict__ zero, int nzero) {
  __shared__ float part[RPC * kQuarters][TT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * RPC + (warp >> 2);
  const int q = warp & 3;
  const int t0 = blockIdx.y * TT;
  const int nvec = H >> 3;
  const int qn = (nvec + kQuarters - 1) / kQuarters;
  const int qb = q * qn, qe = min(nvec, qb + qn);
  // The router weights are constants of the layer, not results of the preceding kernel: while
  // that kernel drains, bring this warp's quarter row into L2 (a hint; the loads below come
  // after the wait and read whatever memory holds then).
  if (blockIdx.y == 0 && lane == 0 && e < E && qe > qb)
    prefetch_l2_bulk(wr + (size_t)e * H + (size_t)qb * 8, (uint32_t)(qe - qb) * 16u);
  pdl_wait();
  pdl_launch();
  if (zero && blockIdx.x == 0 && blockIdx.y == 0)  // counters the next launches start from
    for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
  float a0[TT], a1[TT];
#pragma unroll
  for (int tt = 0; tt < TT; ++tt) a0[tt] = a1[tt] = 0.f;
  if (e < E) {
    const uint4* wrow = reinterpret_cast<const uint4*>(wr + (size_t)e * H);
    for (int base = qb; base < qe; base += 32 * kVecPerLane) {
      uint4 wv[kVecPerLane];
#pragma unroll
      for (int i = 0; i < kVecPerLane; ++i) {
        const int c = base + lane + 32 * i;
        wv[i] = (c < qe) ? ldg_stream(wrow + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int tt = 0; tt < TT; ++tt) {
        if (t0 + tt >= T) break;
        const uint4* hrow = reinterpret_cast<const uint4*>(h + (size_t)(t0 + tt) * H);
#pragma unroll
        for (int i = 0; i < kVecPerLane; ++i) {
          const int c = base + lane + 32 * i;
          if (c < qe) {
            const uint4 v = __ldg(hrow + c);
            fma_bf16x2(wv[i].x, v.x, a0[tt], a1[tt]);
            fma_bf16x2(wv[i].y, v.y, a0[tt], a1[tt]);
            fma_bf16x2(wv[i].z, v.z, a0[tt], a1[tt]);
            fma_bf16x2(wv[i].w, v.w, a0[tt], a1[tt]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int tt = 0; tt < TT; ++tt) {
    const float s = warp_sum(a0[tt] + a1[tt]);
    if (lane == 0) part[warp][tt] = s;
  }
  __syncthreads();
  if (q == 0 && e < E && lane < TT && t0 + lane < T) {
    const int w0 = warp;  // warps w0..w0+3 hold this row's quarters
    const float s = (part[w0][lane] + part[w0 + 1][lane]) + (part[w0 + 2][lane] + part[w0 + 3][lane]);
    logits[(size_t)(t0 + lane) * E + e] = s;
  }
  if (xq) {
    // four lanes per group of 32 (eight elements each, the hardware E2M1 rounding), eight
    // groups per warp: the split is on the critical path of the layer (the expert GEMM waits
    // for this whole launch), so it is kept to one short chain per warp
    const int grp = (blockIdx.x * (RPC * kQuarters) + warp) * 8 + (lane >> 2);
    const int t4 = lane & 3;
    if (blockIdx.x * (RPC * kQuarters) * 8 < (L >> 5)) {  // whole warps take part
      float r[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (grp < (L >> 5)) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(x + 32 * grp + 8 * t4));
        r[0] = bf16lo(raw.x); r[1] = bf16hi(raw.x); r[2] = bf16lo(raw.y); r[3] = bf16hi(raw.y);
        r[4] = bf16lo(raw.z); r[5] = bf16hi(raw.z); r[6] = bf16lo(raw.w); r[7] = bf16hi(raw.w);
      }
      uint32_t w[kTerms], sf[kTerms];
      mx_split_quad8(r, w, sf);
      if (grp < (L >> 5)) {
#pragma unroll
        for (int t = 0; t < kTerms; ++t) {
          *reinterpret_cast<uint32_t*>(xq + (size_t)t * (L >> 1) + grp * 16 + 4 * t4) = w[t];
          if (t4 == 0) xsf[(size_t)t * (L >> 5) + grp] = (uint8_t)sf[t];
        }
      }
    }
  }
}

// Batches (T >= 3): the router as a tensor-core GEMM, logits[t][e] = sum_i h[t][i] Wr[e][i].
// One CTA per 128 experts x 128 tokens x one of `ks` ranges of the reduction: TMA brings
// 64-wide K slices of Wr and h (bf16, 128-byte swizzle) into a 4-stage ring, one thread issues
// tcgen05.mma kind::f16 (bf16 x bf16 -> fp32 in TMEM, K = 16 each), and all four warps read the
// accumulator back (lane = expert row, column = token).  With ks > 1 (few tokens: one range
// per CTA would leave most SMs idle) each CTA writes its range's partial sums to part
// [ks][T][E], and the kernel that takes the top-k adds them in range order (deterministic);
// with ks == 1 it writes the logits.  Products of bf16 values are exact; the sums are fp32.
// A K tail past H reads zeros.  Every wait is bounded: one that runs out counts a timeout and
// the CTA skips its output.
constexpr int kRtStages = 4;
constexpr uint32_t kRtTile = 128 * 128;  // one 128-row x 128-byte operand slice

__global__ void __launch_bounds__(128, 1) k_router_tc(const __grid_constant__ CUtensorMap mw,
                                                      const __grid_constant__ CUtensorMap mh,
                                                      int T, int E, int H, int ks,
                                                      float* __restrict__ logits,
                                                      int32_t* __restrict__ status) {
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[kRtStages], empty[kRtStages], done;
  __shared__ uint32_t tbase;
  __shared__ int bad;
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) &
                                           ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * 128, t0 = blockIdx.y * 128;
  const int nk_all = (H + 63) / 64;
  const int k_lo = (int)(((long long)nk_all * blockIdx.z) / ks);
  const int nk = (int)(((long long)nk_all * (blockIdx.z + 1)) / ks) - k_lo;
  float* const out = logits + (size_t)blockIdx.z * T * E;  // this range's partials (or logits)
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    fence_mbar_init();
    bad = 0;
  }
  if (warp == 1) {
    tc::tmem_alloc(&tbase, 128);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // Only h comes from the preceding launch (the router weights are constants of the layer, and
  // nothing before reads what this kernel writes): the first stages' weight slices are
  // requested before the wait, and only the thread that loads h waits.
  pdl_launch();
  const uint32_t tacc = tbase;
  if (warp == 0 && lane == 0) {
    const int pre = nk < kRtStages ? nk : kRtStages;
    for (int i = 0; i < pre; ++i) {
      mbar_arrive_expect_tx(&full[i], 2 * kRtTile);
      tc::tma_load_2d(sm + (size_t)i * 2 * kRtTile, &mw, (k_lo + i) * 128, e0, &full[i]);
    }
    pdl_wait();
    for (int i = 0; i < pre; ++i)
      tc::tma_load_2d(sm + (size_t)i * 2 * kRtTile + kRtTile, &mh, (k_lo + i) * 128, t0, &full[i]);
    int i = pre;
    for (; i < nk; ++i) {
      const int s = i % kRtStages;
      if (!mbar_wait(&empty[s], ((i / kRtStages) - 1) & 1, status)) {
        bad = 1;
        break;
      }
      uint8_t* st = sm + (size_t)s * 2 * kRtTile;
      mbar_arrive_expect_tx(&full[s], 2 * kRtTile);
      tc::tma_load_2d(st, &mw, (k_lo + i) * 128, e0, &full[s]);
      tc::tma_load_2d(st + kRtTile, &mh, (k_lo + i) * 128, t0, &full[s]);
    }
    if (bad)  // copies in flight land before the CTA leaves
      for (int d = 1; d <= kRtStages && d <= i; ++d)
        mbar_wait(&full[(i - d) % kRtStages], ((i - d) / kRtStages) & 1, nullptr);
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = tc::idesc_bf16(128, 128);
    int i = 0;
    for (; i < nk; ++i) {
      const int s = i % kRtStages;
      if (!mbar_wait(&full[s], (i / kRtStages) & 1, status)) {
        bad = 1;
        break;
      }
      tc::fence_after_sync();
      const uint32_t st = tc::smem_addr(sm + (size_t)s * 2 * kRtTile);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t ad = tc::smem_desc(st + 32 * j, 16, 1024, tc::kLayout128B);
        const uint64_t bd = tc::smem_desc(st + kRtTile + 32 * j, 16, 1024, tc::kLayout128B);
        tc::mma_bf16(tacc, ad, bd, idesc, (i == 0 && j == 0) ? 0u : 1u);
      }
      tc::mma_commit(&empty[s]);
    }
    tc::mma_commit(&done);
  }
  __syncwarp();
  const bool ok = mbar_wait(&done, 0, threadIdx.x == 0 ? status : nullptr);
  tc::fence_after_sync();
  if (__syncthreads_or(!ok || bad) == 0) {
    const int e = e0 + 32 * warp + lane;
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const int ncol = T - t0 < 128 ? T - t0 : 128;  // the tile's tokens
#pragma unroll 1
    for (int c0 = 0; c0 < ncol; c0 += 16) {
      uint32_t r[16];
      tc::tmem_ld_x16(tacc + lane_off + c0, r);
      tc::tmem_ld_wait();
      if (e < E) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int t = t0 + c0 + c;
          if (t < T) out[(size_t)t * E + e] = __uint_as_float(r[c]);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tacc, 128);
  }
}

__global__ void __launch_bounds__(256) k_topk(float* __restrict__ logits,
                                              const float* __restrict__ part, int ks,
                                              const float* __restrict__ bias, int T, int E,
                                              int k, int renorm, float routed_scale,
                                              int32_t* __restrict__ idx,
                                              float* __restrict__ gate,
                                              float* __restrict__ gap) {
  pdl_wait();
  pdl_launch();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  if (ks > 1) {
    sum_router_parts(part, ks, T, E, t, logits, threadIdx.x & 31, 32);
    __syncwarp();
  }
  topk_warp(logits + (size_t)t * E, bias, E, k, renorm, routed_scale, idx + (size_t)t * k,
            gate + (size_t)t * k, gap ? gap + t : nullptr, threadIdx.x & 31);
}

// Batches up to kTopkBlockMaxTokens: one CTA of 11 warps per token, the block top-k of the
// single-token path (topk_one_token: the keys at or above the (k+1)-th best list maximum,
// sorted by one warp; the full sort when ties leave too many).  Same choice, order, tie
// rule and gates as k_topk; E <= 1056, k <= 31 (or k == E).
__global__ void __launch_bounds__(352) k_topk_block(float* __restrict__ logits,
                                                    const float* __restrict__ part, int ks, int T,
                                                    const float* __restrict__ bias, int E, int k,
                                                    int renorm, float routed_scale,
                                                    int32_t* __restrict__ idx,
                                                    float* __restrict__ gate,
                                                    float* __restrict__ gap) {
  __shared__ unsigned long long lists[11 * 32];
  __shared__ float sig[1056];
  pdl_wait();
  pdl_launch();
  const int t = blockIdx.x;
  if (ks > 1) {
    sum_router_parts_block<3>(part, ks, T, E, t, logits);
    __syncthreads();
  }
  const OneTokenChoice c = topk_one_token<3>(logits + (size_t)t * E, bias, E, k, renorm,
                                             routed_scale, gap ? gap + t : nullptr, lists, sig);
  if (threadIdx.x < k) {
    idx[(size_t)t * k + threadIdx.x] = c.e;
    gate[(size_t)t * k + threadIdx.x] = c.g;
  }
}

}  // namespace

int router_splits(int T, int E, int H) {
  if (T < kRouterTcMinTokens || !router_tc_supported(H) || T > kRouterSplitMaxTokens) return 1;
  const int ctas = ((E + 127) / 128) * ((T + 127) / 128);
  const int nk = (H + 63) / 64;
  int ks = sm_count() / ctas;  // at most one CTA per SM (one wave: a CTA fills an SM's smem)
  ks = ks < nk / 2 ? ks : nk / 2;           // at least two K slices per range
  return ks > 1 ? ks : 1;
}

cudaError_t launch_router_logits(const uint16_t* h, const uint16_t* wr, int T, int E, int H,
                                 float* logits, cudaStream_t s, bool pdl, const uint16_t* x,
                                 int L, uint8_t* xq, uint8_t* xsf, int32_t* zero, int nzero,
                                 int32_t* status, float* part) {
  if (T >= kRouterTcMinTokens && !xq && !zero && router_tc_supported(H)) {
    const int ks = router_splits(T, E, H);
    if (ks > 1 && !part) return cudaErrorInvalidValue;
    CUtensorMap mw, mh;
    if (!make_map_2d(&mw, wr, (uint64_t)H * 2, E, 128, 128, true) ||
        !make_map_2d(&mh, h, (uint64_t)H * 2, T, 128, 128, true))
      return cudaErrorInvalidValue;
    static int configured[64] = {0};
    constexpr size_t smem = (size_t)kRtStages * 2 * kRtTile + 1024;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[dev]) {
      const cudaError_t e = cudaFuncSetAttribute(
          k_router_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) configured[dev] = 1;
    }
    return launch_kernel(k_router_tc, dim3((E + 127) / 128, (T + 127) / 128, ks), dim3(128), smem,
                         s, pdl, mw, mh, T, E, H, ks, ks > 1 ? part : logits, status);
  }
  if (T <= 2) {
    const unsigned gx = (E + kRpcFew - 1) / kRpcFew;
    if (xq && (T != 1 || (int)gx * kRpcFew * kQuarters * 8 < (L >> 5) || (L & 7) != 0))
      return cudaErrorInvalidValue;
    return launch_kernel(k_router_logits<1, kRpcFew>, dim3(gx, T), dim3(kRpcFew * kQuarters * 32),
                         0, s, pdl, h, wr, T, E, H, logits, x, L, xq, xsf, zero, nzero);
  }
  if (xq) return cudaErrorInvalidValue;
  const unsigned gx = (E + 1) / 2;
  return launch_kernel(k_router_logits<4, 2>, dim3(gx, (T + 3) / 4), dim3(2 * kQuarters * 32), 0,
                       s, pdl, h, wr, T, E, H, logits, x, L, xq, xsf, zero, nzero);
}

cudaError_t launch_topk(float* logits, const float* part, int ks, const float* bias, int T, int E,
                        int k, int renorm, float routed_scale, int32_t* idx, float* gate,
                        float* gap, cudaStream_t s, bool pdl) {
  if (T <= kTopkBlockMaxTokens && E <= 1056 && (k <= 31 || k == E))
    return launch_kernel(k_topk_block, dim3(T), dim3(352), 0, s, pdl, logits, part, ks, T, bias, E,
                         k, renorm, routed_scale, idx, gate, gap);
  return launch_kernel(k_topk, dim3((T + 7) / 8), dim3(256), 0, s, pdl, logits, part, ks, bias, T,
                       E, k, renorm, routed_scale, idx, gate, gap);
}

}  // namespace k3
