// topk.cuh -- the top-k with gates for one token (README "kimi-k3-in-c", Part II section 9
// "Picking 16 experts of 896"): one warp's version for the router's top-k kernel, and a
// block's version for the batch-1 preparation and the expert GEMMs that route in-kernel.
#pragma once

#include "common.cuh"

namespace k3 {

__device__ __forceinline__ float sigmoid_f32(float z) { return 1.0f / (1.0f + expf(-z)); }

// Lane l holds the selection scores (sigmoid(logit) + bias) of experts l, l+32, ... in
// registers (E <= 1024).  Each round finds the lane-local best among untaken experts,
// visited in increasing index order with a strict '>' (the lowest index of equal scores),
// then a warp arg-max where a larger score wins and equal scores go to the lower index.
// One extra round gives the best unchosen score for the gap.  NaN scores count as -inf.
// Gates: the unbiased scores of the chosen experts, renormalised by their sum when renorm
// is set and the sum is positive, times routed_scale.
__device__ __forceinline__ void topk_warp(const float* lt, const float* bias, int E, int k,
                                          int renorm, float routed_scale, int32_t* idx,
                                          float* gate, float* gap, int lane) {
  float ch[32];
  uint32_t taken = 0;
#pragma unroll
  for (int m = 0; m < 32; ++m) {
    const int e = lane + 32 * m;
    float v = -INFINITY;
    if (e < E) {
      v = sigmoid_f32(lt[e]) + (bias ? bias[e] : 0.0f);
      if (isnan(v)) v = -INFINITY;
    } else {
      taken |= 1u << m;  // not an expert
    }
    ch[m] = v;
  }
  int my_e = -1;
  float last_v = 0.f, next_v = -INFINITY;
  const int rounds = (k < E) ? k + 1 : k;
  for (int j = 0; j < rounds; ++j) {
    float bv = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      if (!((taken >> m) & 1u) && (be == INT_MAX || ch[m] > bv)) {
        bv = ch[m];
        be = lane + 32 * m;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
        bv = ov;
        be = oe;
      }
    }
    if (j < k) {
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == j) my_e = be;
      last_v = bv;
    } else {
      next_v = bv;
    }
  }
  const float s = (lane < k) ? sigmoid_f32(lt[my_e]) : 0.f;  // unbiased score of choice j
  const float sum = warp_sum(s);
  float g = s;
  if (renorm && sum > 0.f) g = s / sum;
  g *= routed_scale;
  if (lane < k) {
    idx[lane] = my_e;
    gate[lane] = g;
  }
  if (gap && lane == 0) *gap = (k < E) ? (last_v - next_v) : INFINITY;
}

// Order-preserving map of a float onto uint32 (NaN and -0 normalised first).
__device__ __forceinline__ uint32_t ordered_bits(float v) {
  if (isnan(v)) v = -INFINITY;
  v += 0.0f;  // -0 -> +0
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float from_ordered_bits(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// The same top-k for one token with a whole block of exactly 1024 threads (E <= 1024):
// keys (descending selection score, then ascending expert index) are sorted by a bitonic
// network in shared memory; the first k keys are the choice, key k gives the gap.  The
// order and the tie rule are those of topk_warp.
__device__ __forceinline__ void topk_block_sort(const float* lt, const float* bias, int E, int k,
                                                int renorm, float routed_scale, int32_t* idx,
                                                float* gate, float* gap, uint64_t* keys) {
  const int tid = threadIdx.x;
  uint64_t key = ~0ull;
  if (tid < E) {
    const float v = sigmoid_f32(lt[tid]) + (bias ? bias[tid] : 0.0f);
    key = ((uint64_t)(~ordered_bits(v)) << 32) | (uint32_t)tid;
  }
  keys[tid] = key;
  __syncthreads();
  for (int size = 2; size <= 1024; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int j = tid ^ stride;
      if (j > tid) {
        const uint64_t a = keys[tid], b = keys[j];
        const bool asc = (tid & size) == 0;
        if ((a > b) == asc) {
          keys[tid] = b;
          keys[j] = a;
        }
      }
      __syncthreads();
    }
  }
  if (tid < 32) {
    const int lane = tid;
    int e = -1;
    float s = 0.f;
    if (lane < k) {
      e = (int)(uint32_t)(keys[lane] & 0xffffffffu);
      s = sigmoid_f32(lt[e]);  // the unbiased score of choice j
    }
    const float sum = warp_sum(s);
    float g = s;
    if (renorm && sum > 0.f) g = s / sum;
    g *= routed_scale;
    if (lane < k) {
      idx[lane] = e;
      gate[lane] = g;
    }
    if (gap && lane == 0)
      *gap = (k < E) ? from_ordered_bits(~(uint32_t)(keys[k - 1] >> 32)) -
                           from_ordered_bits(~(uint32_t)(keys[k] >> 32))
                     : INFINITY;
  }
  __syncthreads();
}

// One token's top-k with a whole block, for decode: the same choice, order and tie rule as
// topk_warp, by sorting instead of repeated arg-max.  Key = (order bits of the selection
// score, then ~expert), so a larger key is a better choice and equal scores go to the lower
// index; key 0 stands for "no expert" and sorts last.
//  1. warp w holds the keys of experts 32(LPW w + j) + lane, j < LPW, and sorts each 32-key
//     list descending (bitonic, shuffles; the LPW lists are independent, so they overlap);
//  2. two sorted lists merge into the top 32 of their union by one max against the other
//     list reversed (a bitonic sequence) and five clean-up steps; the warp merges its own
//     lists, then the warps' lists merge pairwise in a tree through shared memory;
//  3. warp 0 ends with the top 32 keys, best first: choice j < k on lane j, key k for the gap.
// Needs k <= 31 (or k == E), E <= 32 * LPW * (warps); every thread calls it.  lists: shared
// [max(warps * 32, 129)]; sig: shared [E] (each expert's unbiased score, for the gates).  On warp 0,
// lane j < k returns choice j's expert e, gate g, and rank (its place among the chosen
// experts in ascending index order); lane 0 writes the gap when gap is set.
struct OneTokenChoice {
  int e;
  float g;
  int rank;
};

__device__ __forceinline__ unsigned long long top32_clean(unsigned long long v, int lane) {
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, stride);
    const bool lo = (lane & stride) == 0;
    v = lo ? (v > o ? v : o) : (v > o ? o : v);
  }
  return v;
}

template <int LPW>
__device__ __forceinline__ OneTokenChoice topk_one_token(const float* lt, const float* bias,
                                                         int E, int k, int renorm,
                                                         float routed_scale, float* gap,
                                                         unsigned long long* lists, float* sig) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  unsigned long long key[LPW];
  float lg[LPW], bs[LPW];
#pragma unroll
  for (int j = 0; j < LPW; ++j) {  // lt read at L2 (written by an earlier launch)
    const int e = (warp * LPW + j) * 32 + lane;
    lg[j] = e < E ? __ldcg(lt + e) : 0.f;
    bs[j] = (e < E && bias) ? bias[e] : 0.f;
  }
#pragma unroll
  for (int j = 0; j < LPW; ++j) {
    const int e = (warp * LPW + j) * 32 + lane;
    key[j] = 0ull;
    if (e < E) {
      const float sg = sigmoid_f32(lg[j]);
      sig[e] = sg;
      key[j] = ((unsigned long long)ordered_bits(sg + bs[j]) << 32) | (uint32_t)(~(uint32_t)e);
    }
  }
  // Fast path: the (k+1)-th best of the lists' maxima is a lower bound of the (k+1)-th best
  // key (k+1 lists each hold a key at least that good), so the keys at or above it contain
  // the top k+1.  They are few (gathered in shared memory), and each finds its place by
  // counting the candidates that beat it: a few dependent steps, where a sort in one warp
  // would chain twenty.  More than 64 (many equal scores), or fewer lists than k+1: the
  // full sort below.
  const int nl = (E + 31) >> 5;
  unsigned long long acc = 0ull;
  bool fast = false;
  if (k + 1 <= nl && nl <= 32) {
    unsigned long long* lmax = lists;       // [32] best key of each list
    unsigned long long* cand = lists + 32;  // [64] candidates
    unsigned long long* top = lists + 96;   // [32] the best candidates, best first
    unsigned int* ncand = reinterpret_cast<unsigned int*>(lists + 128);
    // each list's best key: the highest score (one max over the warp), then among the lanes
    // holding it the lowest expert (the highest ~e)
    unsigned long long m[LPW];
#pragma unroll
    for (int j = 0; j < LPW; ++j) {
      const uint32_t hi = (uint32_t)(key[j] >> 32);
      const uint32_t mh = __reduce_max_sync(0xffffffffu, hi);
      const uint32_t ml = __reduce_max_sync(0xffffffffu, hi == mh ? (uint32_t)key[j] : 0u);
      m[j] = ((unsigned long long)mh << 32) | ml;
    }
    if (lane == 0)
#pragma unroll
      for (int j = 0; j < LPW; ++j)
        if (warp * LPW + j < 32) lmax[warp * LPW + j] = m[j];
    if (threadIdx.x == 0) *ncand = 0u;
    __syncthreads();
    // every warp finds the threshold itself: the list maximum with exactly k better ones
    // (keys are distinct, so exactly one lane has that rank)
    const unsigned long long mine = lane < nl ? lmax[lane] : 0ull;
    int rank = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) rank += (i < nl && lmax[i] > mine) ? 1 : 0;
    const unsigned int who = __ballot_sync(0xffffffffu, lane < nl && rank == k);
    const unsigned long long th = __shfl_sync(0xffffffffu, mine, __ffs(who) - 1);
    // gather the keys at or above it: one shared-memory atomic per warp
    unsigned int bal[LPW], cnt = 0u;
#pragma unroll
    for (int j = 0; j < LPW; ++j) {
      bal[j] = __ballot_sync(0xffffffffu, key[j] >= th);
      cnt += __popc(bal[j]);
    }
    unsigned int base = 0u;
    if (lane == 0 && cnt) base = atomicAdd(ncand, cnt);
    base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
    for (int j = 0; j < LPW; ++j) {
      const unsigned int pos = base + __popc(bal[j] & ((1u << lane) - 1u));
      if (((bal[j] >> lane) & 1u) && pos < 64u) cand[pos] = key[j];
      base += __popc(bal[j]);
    }
    __syncthreads();
    const unsigned int nc = *ncand;
    if (nc <= 64u) {
      fast = true;
      // candidate i's place = how many candidates beat it (distinct keys: a permutation);
      // threads 0..nc-1 count side by side, reading the list by broadcast
      if (threadIdx.x < nc) {
        const unsigned long long ci = cand[threadIdx.x];
        int r = 0;
#pragma unroll 1
        for (unsigned int j0 = 0; j0 < nc; j0 += 8) {
#pragma unroll
          for (unsigned int jj = 0; jj < 8; ++jj)
            r += (j0 + jj < nc && cand[j0 + jj] > ci) ? 1 : 0;
        }
        if (r < 32) top[r] = ci;
      }
      __syncthreads();
      if (warp == 0) acc = lane < (int)nc ? top[lane] : 0ull;
    }
    __syncthreads();  // the full path below reuses the scratch
  }
  if (!fast) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const bool desc = (lane & size) == 0, lo = (lane & stride) == 0;
#pragma unroll
        for (int j = 0; j < LPW; ++j) {
          const unsigned long long o = __shfl_xor_sync(0xffffffffu, key[j], stride);
          const unsigned long long mx = key[j] > o ? key[j] : o, mn = key[j] > o ? o : key[j];
          key[j] = (lo == desc) ? mx : mn;
        }
      }
    }
    acc = key[0];
#pragma unroll
    for (int j = 1; j < LPW; ++j) {
      const unsigned long long o = __shfl_sync(0xffffffffu, key[j], 31 - lane);
      acc = top32_clean(acc > o ? acc : o, lane);
    }
    lists[warp * 32 + lane] = acc;
    __syncthreads();
    for (int n = nwarps; n > 1;) {
      const int h = (n + 1) >> 1;
      if (warp < n - h) {
        const unsigned long long o = lists[(warp + h) * 32 + 31 - lane];
        acc = top32_clean(acc > o ? acc : o, lane);
        lists[warp * 32 + lane] = acc;
      }
      n = h;
      __syncthreads();
    }
  }
  OneTokenChoice c = {-1, 0.f, 0};
  if (warp == 0) {
    const unsigned long long kth = __shfl_sync(0xffffffffu, acc, k > 0 ? k - 1 : 0);
    const unsigned long long next = __shfl_sync(0xffffffffu, acc, k < 32 ? k : 31);
    float s = 0.f;
    if (lane < k) {
      c.e = (int)(~(uint32_t)(acc & 0xffffffffull));
      s = sig[c.e];  // the unbiased score of choice j
    }
    const float sum = warp_sum(s);
    c.g = s;
    if (renorm && sum > 0.f) c.g = s / sum;
    c.g *= routed_scale;
    if (gap && lane == 0)
      *gap = (k < E) ? from_ordered_bits((uint32_t)(kth >> 32)) -
                           from_ordered_bits((uint32_t)(next >> 32))
                     : INFINITY;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int ei = __shfl_sync(0xffffffffu, c.e, i);
      if (i < k && ei < c.e) ++c.rank;
    }
  }
  return c;
}

}  // namespace k3
