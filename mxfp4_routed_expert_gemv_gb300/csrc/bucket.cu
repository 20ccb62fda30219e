// bucket.cu -- token -> expert bucketing (a counting sort of the T*k assignments) and the
// per-call preparation of the expert GEMVs.
//
// An assignment whose index is kRemoteExpert belongs to an expert held elsewhere (the
// expert-range entry point marks them so): it is skipped like an out-of-range index, but not
// counted as a drop.
//
// Output: counts[E], offsets[E+1] (exclusive prefix of counts), perm[] = the valid
// assignment ids a = t*k + j sorted by expert and, within an expert, by token (stable),
// the list of active experts (count > 0) in ascending order with each one's perm offset
// and token count, nvalid[t] (valid assignments of token t), and x in the GEMVs' f16 form.  An
// expert index outside [0, E) is skipped and counted in status[0] (the README's "counted,
// never silent" expert-drop rule, Part II section 9).
//
// Batches of up to 4096 assignments take one CTA for everything (up to 32 tokens optionally
// including the router's top-k), so the whole preparation is one launch.
#include "launch.h"
#include "mxq.cuh"
#include "topk.cuh"

namespace k3 {
namespace {

constexpr int kChunkTokens = 16;  // tokens per block in the multi-block path
constexpr int kSmallTokens = 32;     // the one-CTA preparation also takes the top-k up to here
constexpr int kSortAssign = 4096;    // assignments (T k) the one-CTA preparation takes
static_assert(kMaxExperts <= (1 << 20) && kSortAssign <= (1 << 12), "sort key fields");

// Exclusive scans of N ints per thread at once over a block of exactly 1024 threads (one
// round of barriers for all N); tot[i] gets the block sum of component i.
template <int N>
__device__ void block_exclusive_scan_1024_n(const int (&v)[N], int (&excl)[N], int (&tot)[N]) {
  __shared__ int warp_tot[32][N];
  __shared__ int btot[N];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl[N];
#pragma unroll
  for (int i = 0; i < N; ++i) incl[i] = v[i];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int n = __shfl_up_sync(0xffffffffu, incl[i], o);
      if (lane >= o) incl[i] += n;
    }
  }
  if (lane == 31)
#pragma unroll
    for (int i = 0; i < N; ++i) warp_tot[warp][i] = incl[i];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int w = warp_tot[lane][i];
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += n;
      }
      warp_tot[lane][i] = wi - w;  // exclusive prefix of the warp totals
      if (lane == 31) btot[i] = wi;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    excl[i] = warp_tot[warp][i] + incl[i] - v[i];
    tot[i] = btot[i];
  }
  __syncthreads();  // warp_tot and btot are reused by the next call
}

// Shared-memory copies of the active experts' segments, for the descriptors below.
struct SegSmem {
  int gbase[kMaxExperts + 1];  // groups of the descriptors' table before each active expert
  int act[kMaxExperts];        // expert id
  int soff[kMaxExperts];       // perm offset
  int scnt[kMaxExperts];       // tokens
};

// Writes offsets/counts/active lists and the group tables from per-expert counts c (thread e
// holds c; every thread also brings `dropped`, the invalid assignments it saw, whose sum is
// counted in the status block), and the large-batch tile descriptors when o.wdesc is set.
// Returns expert e's perm offset on thread e.
__device__ int publish_counts(int c, int dropped, int E, const BucketOut& o, int32_t* status,
                              SegSmem& sg) {
  const int e = threadIdx.x;
  const int flag = (e < E && c > 0) ? 1 : 0;
  // one scan for everything: tokens, active experts, groups of 16 / kTcWideTok / kTcRowTok
  // tokens, invalid assignments
  const int v[6] = {c, flag, flag ? (c + kTcTokTile - 1) / kTcTokTile : 0,
                    flag ? (c + kTcWideTok - 1) / kTcWideTok : 0,
                    flag ? (c + kTcRowTok - 1) / kTcRowTok : 0, dropped};
  int ex[6], tot[6];
  block_exclusive_scan_1024_n<6>(v, ex, tot);
  const int excl = ex[0], total = tot[0], pos = ex[1], nact = tot[1];
  if (e < E) {
    o.offsets[e] = excl;
    o.counts[e] = c;
  }
  if (e == 0) {
    o.offsets[E] = total;
    o.meta[0] = nact;
    o.meta[1] = total;
    o.meta[2] = tot[2];
    o.meta[3] = tot[3];
    o.meta[4] = tot[4];
    o.ntile_base[nact] = tot[2];
    o.nbase_w[nact] = tot[3];
    o.nbase_r[nact] = tot[4];
    if (tot[5] > 0 && status) atomicAdd(status + kStatDropped, tot[5]);
  }
  const bool rows = o.wmode == 2;
  if (flag) {
    o.active[pos] = e;
    o.seg_off[pos] = excl;
    o.seg_cnt[pos] = c;
    // tensor-core tiles and the large-batch group tables: per active expert its groups'
    // expert, first position and tokens
    o.ntile_base[pos] = ex[2];
    for (int n = 0; n * kTcTokTile < c; ++n)
      o.tiles[ex[2] + n] = make_int4(e, excl + n * kTcTokTile, min(kTcTokTile, c - n * kTcTokTile), 0);
    o.nbase_w[pos] = ex[3];
    for (int n = 0; n * kTcWideTok < c; ++n)
      o.tiles_w[ex[3] + n] = make_int4(e, excl + n * kTcWideTok, min(kTcWideTok, c - n * kTcWideTok), 0);
    o.nbase_r[pos] = ex[4];
    for (int n = 0; n * kTcRowTok < c; ++n)
      o.tiles_r[ex[4] + n] = make_int4(e, excl + n * kTcRowTok, min(kTcRowTok, c - n * kTcRowTok), 0);
    sg.gbase[pos] = rows ? ex[4] : ex[3];
    sg.act[pos] = e;
    sg.soff[pos] = excl;
    sg.scnt[pos] = c;
  }
  if (e == 0) sg.gbase[nact] = rows ? tot[4] : tot[3];
  for (int i = e; i < kTcFlagWords; i += blockDim.x) o.flags[i] = 0;
  if (o.wdesc) {
    // The large-batch GEMMs' tile descriptors: for each GEMM, tile t is the active expert
    // whose block of (groups x row blocks) holds t (bisection over the group prefix), its row
    // block and its group (groups fastest): expert, first position, tokens, row block | the
    // expert's groups << 8.
    __syncthreads();  // sg
    const int tok = rows ? kTcRowTok : kTcWideTok;
    for (int ph = 0; ph < 2; ++ph) {
      const int RB = ph == 0 ? o.wrb0 : o.wrb1;
      int4* desc = o.wdesc + (ph == 0 ? 0 : o.wdesc1);
      const int n = sg.gbase[nact] * RB;
      for (int t = threadIdx.x; t < n; t += blockDim.x) {
        int lo = 0, hi = nact - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (sg.gbase[mid] * RB <= t) lo = mid; else hi = mid - 1;
        }
        const int gb = sg.gbase[lo], ng = sg.gbase[lo + 1] - gb;
        const int local = t - gb * RB;
        const int rb = local / ng;
        const int g = local - rb * ng;
        const int n0 = g * tok;
        desc[t] = make_int4(sg.act[lo], sg.soff[lo] + n0, min(tok, sg.scnt[lo] - n0), rb | (ng << 8));
      }
    }
  }
  __syncthreads();  // sg is reused by the next call
  return excl;
}

// One warp: x row (bf16) -> f16 scaled by 2^-e with the largest magnitude in [2^14, 2^15).
// L % 32 == 0; 16-byte vector accesses when L % 256 == 0.
__device__ void prep_x_warp(const uint16_t* xr, int L, __half* out, int32_t* xexp, int lane) {
  float m = 0.f;
  const bool vec = (L & 255) == 0;
  if (vec) {
    for (int c = lane * 8; c < L; c += 256) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + c));
      m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16lo(v.x)), fabsf(bf16hi(v.x))), fmaxf(fabsf(bf16lo(v.y)), fabsf(bf16hi(v.y)))));
      m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16lo(v.z)), fabsf(bf16hi(v.z))), fmaxf(fabsf(bf16lo(v.w)), fabsf(bf16hi(v.w)))));
    }
  } else {
    for (int c = lane; c < L; c += 32) m = fmaxf(m, fabsf(__uint_as_float((uint32_t)xr[c] << 16)));
  }
  m = warp_max(m);
  const int e = f16_exponent_for(m);
  const Pow2Scale sc(e);
  if (vec) {
    for (int c = lane * 8; c < L; c += 256) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + c));
      uint4 o;
      o.x = pack_half2(sc(bf16lo(v.x)), sc(bf16hi(v.x)));
      o.y = pack_half2(sc(bf16lo(v.y)), sc(bf16hi(v.y)));
      o.z = pack_half2(sc(bf16lo(v.z)), sc(bf16hi(v.z)));
      o.w = pack_half2(sc(bf16lo(v.w)), sc(bf16hi(v.w)));
      *reinterpret_cast<uint4*>(out + c) = o;
    }
  } else {
    for (int c = lane; c < L; c += 32) out[c] = __float2half_rn(sc(__uint_as_float((uint32_t)xr[c] << 16)));
  }
  if (lane == 0) *xexp = e;
}

// Per token: count valid assignments (y of a token without one is zeroed here; the
// combine writes every token's y as well).
__device__ void token_valid_warp(const int32_t* idx_t, int k, int E, int L, int32_t* nvalid_t,
                                 float* y_t, int lane) {
  int v = 0;
  if (lane < k) {
    const int e = idx_t[lane];
    v = (e >= 0 && e < E) ? 1 : 0;
  }
  const int n = __popc(__ballot_sync(0xffffffffu, v));
  if (lane == 0) *nvalid_t = n;
  if (n == 0)
    for (int c = lane; c < L; c += 32) y_t[c] = 0.f;
}

// Single block of 1024 threads, up to kSortAssign assignments: [top-k, T <= kSmallTokens],
// count, scan, the stable scatter, per-token counts, x prep.  The scatter ranks each
// assignment among the earlier ones of its expert: up to kMaskTokens tokens, from a bit mask
// per expert over the tokens (its rank is the number of lower tokens set, as no token names
// an expert twice; a token that does takes the other way); otherwise a bitonic sort of the
// keys (expert << 12 | assignment id) in shared memory, whose position i is perm position i.
// Either gives the order of the multi-block path (experts ascending, tokens ascending).
constexpr int kMaskTokens = 128;
constexpr int kMaskWords = kMaskTokens / 32;
__global__ void __launch_bounds__(1024) k_prep_small(PrepArgs p) {
  pdl_wait();
  pdl_launch();
  __shared__ int cnt[kMaxExperts];
  // the one-token top-k's sort keys, then the token masks [E][kMaskWords] or the sort keys
  __shared__ __align__(16) uint32_t sbuf[kSortAssign];
  static_assert(kMaxExperts * kMaskWords <= kSortAssign && kSortAssign * 4 >= 1024 * 8, "sbuf");
  __shared__ SegSmem sg;
  uint64_t* keys = reinterpret_cast<uint64_t*>(sbuf);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, k = p.k, E = p.E;
  if (p.logits) {
    if (T == 1)
      topk_block_sort(p.logits, p.bias, E, k, p.renorm, p.routed_scale, p.idx, p.gate, p.gap, keys);
    else if (warp < T)
      topk_warp(p.logits + (size_t)warp * E, p.bias, E, k, p.renorm, p.routed_scale,
                p.idx + (size_t)warp * k, p.gate + (size_t)warp * k,
                p.gap ? p.gap + warp : nullptr, lane);
  }
  const int P = T * k;
  const bool masks = T <= kMaskTokens;
  cnt[tid] = 0;
  if (masks)
    for (int i = tid; i < E * kMaskWords; i += blockDim.x) sbuf[i] = 0u;
  __syncthreads();  // top-k results (global, this block) are visible from here on
  int NP = 32;  // sort width: a power of two >= P
  while (NP < P) NP <<= 1;
  int dropped = 0, dup = 0;
  for (int a = tid; a < (masks ? P : NP); a += blockDim.x) {
    uint32_t key = 0xffffffffu;
    if (a < P) {
      const int e = p.idx[a];
      if (e >= 0 && e < E) {
        atomicAdd(&cnt[e], 1);
        key = ((uint32_t)e << 12) | (uint32_t)a;
        if (masks) {
          const int t = a / k;
          const uint32_t bit = 1u << (t & 31);
          dup |= (atomicOr(&sbuf[e * kMaskWords + (t >> 5)], bit) & bit) ? 1 : 0;
        }
      } else if (e != kRemoteExpert) {
        ++dropped;
      }
    }
    if (!masks) sbuf[a] = key;
  }
  const bool sort = __syncthreads_or(dup) != 0 || !masks;
  const int c = (tid < E) ? cnt[tid] : 0;
  const int excl = publish_counts(c, dropped, E, p.b, p.status, sg);
  if (!sort) {
    // rank = tokens of this expert below t
    if (tid < E) cnt[tid] = excl;
    __syncthreads();
    for (int a = tid; a < P; a += blockDim.x) {
      const int e = p.idx[a];
      if (e >= 0 && e < E) {
        const int t = a / k;
        const uint32_t* m = sbuf + e * kMaskWords;
        int r = __popc(m[t >> 5] & ((1u << (t & 31)) - 1u));
        for (int w = 0; w < (t >> 5); ++w) r += __popc(m[w]);
        const int pos = cnt[e] + r;
        p.b.perm[pos] = a;
        p.b.inv[a] = pos;
      }
    }
  } else {
    if (masks) {  // the keys were not kept: a second pass
      for (int a = tid; a < NP; a += blockDim.x) {
        uint32_t key = 0xffffffffu;
        if (a < P) {
          const int e = p.idx[a];
          if (e >= 0 && e < E) key = ((uint32_t)e << 12) | (uint32_t)a;
        }
        sbuf[a] = key;
      }
      __syncthreads();
    }
    for (int size = 2; size <= NP; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < NP; i += blockDim.x) {
          const int j = i ^ stride;
          if (j > i) {
            const uint32_t a = sbuf[i], b = sbuf[j];
            if ((a > b) == ((i & size) == 0)) {
              sbuf[i] = b;
              sbuf[j] = a;
            }
          }
        }
        __syncthreads();
      }
    }
    for (int i = tid; i < P; i += blockDim.x) {
      const uint32_t key = sbuf[i];
      if (key != 0xffffffffu) {
        const int a = (int)(key & 0xfffu);
        p.b.perm[i] = a;
        p.b.inv[a] = i;
      }
    }
  }
  for (int t = warp; t < T; t += 32) {
    if (p.x16) prep_x_warp(p.x + (size_t)t * p.L, p.L, p.x16 + (size_t)t * p.L, p.xexp + t, lane);
    token_valid_warp(p.idx + (size_t)t * k, k, E, p.L, p.b.nvalid + t, p.y + (size_t)t * p.L, lane);
  }
}

// Multi-block path, pass 1: per-chunk histograms stored transposed [E][nchunks]; also the
// chunk's tokens' nvalid.
__global__ void __launch_bounds__(256) k_bucket_count(PrepArgs p, int nchunks) {
  pdl_wait();
  pdl_launch();
  __shared__ int hist[kMaxExperts];
  const int T = p.T, k = p.k, E = p.E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int c = blockIdx.x;
  const int t0 = c * kChunkTokens, t1 = min(T, t0 + kChunkTokens);
  int dropped = 0;
  for (int a = t0 * k + threadIdx.x; a < t1 * k; a += blockDim.x) {
    const int e = p.idx[a];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else if (e != kRemoteExpert) ++dropped;
  }
  if (dropped && p.status) atomicAdd(p.status + kStatDropped, dropped);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = t0 + warp; t < t1; t += blockDim.x >> 5)
    token_valid_warp(p.idx + (size_t)t * k, k, E, p.L, p.b.nvalid + t, p.y + (size_t)t * p.L, lane);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) p.b.chunk_base[(size_t)e * nchunks + c] = hist[e];
}

// Pass 2a: per expert (one warp each), the exclusive prefix of its chunk histograms in chunk
// order, in place (positions relative to the expert's first), and its total into counts[e].
__global__ void __launch_bounds__(1024) k_bucket_chunkscan(int E, int nchunks, BucketOut o) {
  pdl_wait();
  pdl_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + warp;
  if (e >= E) return;
  int32_t* cb = o.chunk_base + (size_t)e * nchunks;
  int run = 0;
  for (int c0 = 0; c0 < nchunks; c0 += 32) {
    const int c = c0 + lane;
    const int v = c < nchunks ? cb[c] : 0;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += n;
    }
    if (c < nchunks) cb[c] = run + incl - v;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) o.counts[e] = run;
}

// Pass 2b (one block): the scan over experts (offsets, active list, tile tables).
__global__ void __launch_bounds__(1024) k_bucket_scan(int E, BucketOut o) {
  pdl_wait();
  pdl_launch();
  __shared__ SegSmem sg;
  const int e = threadIdx.x;
  publish_counts(e < E ? o.counts[e] : 0, 0, E, o, nullptr, sg);
}

// Pass 3: stable scatter of one chunk, token by token by one warp (the block's other warps
// help fill the cursors); the chunk's expert indices are loaded before the first token.
__global__ void __launch_bounds__(256) k_bucket_scatter(const int32_t* __restrict__ idx, int T,
                                                        int k, int E, int nchunks, BucketOut o) {
  pdl_wait();
  pdl_launch();
  __shared__ int cur[kMaxExperts];
  const int c = blockIdx.x, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    cur[e] = o.offsets[e] + o.chunk_base[(size_t)e * nchunks + c];
  const int t0 = c * kChunkTokens;
  int ev[kChunkTokens];
#pragma unroll
  for (int i = 0; i < kChunkTokens; ++i)
    ev[i] = (threadIdx.x < 32 && lane < k && t0 + i < T) ? idx[(size_t)(t0 + i) * k + lane] : -1;
  __syncthreads();
  if (threadIdx.x >= 32) return;
#pragma unroll
  for (int i = 0; i < kChunkTokens; ++i) {
    const int e = ev[i];
    if (e >= 0 && e < E) {
      const int a = (t0 + i) * k + lane;
      const int pos = atomicAdd(&cur[e], 1);
      o.perm[pos] = a;
      o.inv[a] = pos;
    }
    __syncwarp();
  }
}

__global__ void __launch_bounds__(256) k_localize_idx(const int32_t* __restrict__ idx, int n, int E,
                                                      int e0, int e1, int32_t* __restrict__ out) {
  pdl_wait();
  pdl_launch();
  const int a = blockIdx.x * blockDim.x + threadIdx.x;
  if (a >= n) return;
  const int e = idx[a];
  out[a] = (e >= e0 && e < e1) ? e - e0 : ((e >= 0 && e < E) ? kRemoteExpert : -1);
}

}  // namespace

cudaError_t launch_localize_idx(const int32_t* idx, int n, int E, int e0, int e1,
                                int32_t* idx_local, cudaStream_t s, bool pdl) {
  return launch_kernel(k_localize_idx, dim3((n + 255) / 256), dim3(256), 0, s, pdl, idx, n, E, e0,
                       e1, idx_local);
}

int bucket_chunks(int T) { return (T + kChunkTokens - 1) / kChunkTokens; }

bool prep_is_fused(int T) { return T <= kSmallTokens; }

cudaError_t launch_prep(const PrepArgs& p, cudaStream_t s, bool pdl) {
  if (p.logits && !prep_is_fused(p.T)) return cudaErrorInvalidValue;
  if ((size_t)p.T * p.k <= (size_t)kSortAssign)
    return launch_kernel(k_prep_small, dim3(1), dim3(1024), 0, s, pdl, p);
  // large batches: the top-k runs as its own grid before this point
  const int nch = bucket_chunks(p.T);
  cudaError_t err = launch_kernel(k_bucket_count, dim3(nch), dim3(256), 0, s, pdl, p, nch);
  if (err != cudaSuccess) return err;
  err = launch_kernel(k_bucket_chunkscan, dim3((p.E + 31) / 32), dim3(1024), 0, s, true, p.E, nch, p.b);
  if (err != cudaSuccess) return err;
  err = launch_kernel(k_bucket_scan, dim3(1), dim3(1024), 0, s, true, p.E, p.b);
  if (err != cudaSuccess) return err;
  err = launch_kernel(k_bucket_scatter, dim3(nch), dim3(256), 0, s, true,
                      static_cast<const int32_t*>(p.idx), p.T, p.k, p.E, nch, p.b);
  if (err != cudaSuccess) return err;
  if (!p.x16) return cudaSuccess;
  return launch_prep_x(p.x, p.T, p.L, p.x16, p.xexp, s, true);
}

}  // namespace k3
