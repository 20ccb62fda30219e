// gemv.cu -- MXFP4 grouped GEMV for the routed experts (decode-sized batches).
//
// README "kimi-k3-in-c", Part II section 4: the expert weights are multiplied straight
// from their packed form and never expanded in memory.  Per expert e and token t:
//   g = W1[e] x_t,  u = W3[e] x_t,  act = silu(g) * u  (or SiTU-GLU)       -- k_gemm1
//   o = W2[e] act,  y[t] = sum_j gate[t][j] * o_j  (slot order)            -- k_gemm2
//
// GB300 design.  A 16-row block of w1 and of w3 (k_gemm1) or a 32-row block of w2
// (k_gemm2) is contiguous in HBM, so a producer warp moves it into a shared-memory ring
// with a few bulk asynchronous copies (completion counted on an mbarrier) while eight
// consumer warps decode the previous blocks.  Each consumer warp owns whole row pairs:
// lane l decodes MX groups l, l+32, l+64, ... of both rows (one 16-byte shared load = 32
// nibbles = one group = one scale byte), and when the group count leaves a tail of at
// most 16 groups, lanes 0-15 take the first row's tail and lanes 16-31 the second's, so no
// lane idles on the K3 shapes (112 = 3*32 + 16 groups, 96 = 3*32).  Nibble pairs become
// exact f16 pairs in hardware (cvt e2m1x2) and meet the activations, held as exact f16 in
// registers (scaled by a power of two per vector), in mixed-precision fused multiply-adds
// with fp32 accumulation; each group's partial is multiplied by its E8M0 scale.  A row's
// sum is a fixed butterfly over the warp, so results do not depend on scheduling.
//
// The combine is fused into k_gemm2: each warp writes gate * o for its rows and token
// into a per-assignment slot buffer, then counts the slot in a per-(token, 4-row) counter;
// the warp that completes a counter adds the token's slots in slot order (deterministic)
// and writes y.  There is no spin-wait anywhere: only the mbarrier waits of the ring,
// each bounded.
#include "launch.h"

namespace k3 {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);

struct G1Args {
  const uint8_t *w1p, *w1s, *w3p, *w3s;
  int L, I, k;
  const __half* x16;
  const int32_t* xexp;
  const int32_t *active, *seg_off, *seg_cnt, *meta, *perm;
  float* act;
  int act_kind;
  float b1, b2;
  int32_t* status;
  int stages;
};

struct G2Args {
  const uint8_t *w2p, *w2s;
  int L, I, k, E;
  const float* act;
  const float* gate;
  const int32_t* idx;
  const int32_t *active, *seg_off, *seg_cnt, *meta, *perm, *nvalid;
  float* ybuf;
  int32_t* cnt;
  float* y;
  int32_t* status;
  int stages;
};

// Lane -> group mapping for a pair of rows with G groups (see the file comment).
struct GroupMap {
  int F;        // full rounds: groups l + 32j, j < F, for both rows
  int tail;     // G % 32
  bool paired;  // 0 < tail <= 16: lanes 0-15 take row A's tail, 16-31 row B's
  __device__ GroupMap(int G) : F(G >> 5), tail(G & 31), paired((G & 31) > 0 && (G & 31) <= 16) {}
  // group of the tail round(s) handled by this lane
  __device__ int tail_group(int lane) const { return 32 * F + (paired ? (lane & 15) : lane); }
  __device__ bool tail_ok(int lane) const { return paired ? (lane & 15) < tail : lane < tail; }
};

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

// acc += scale(s) * dot(group of w, x)
__device__ __forceinline__ void mx_group(const uint8_t* wrow, const uint8_t* srow, int g,
                                         const uint32_t (&x)[16], float& acc) {
  acc = fmaf(dot32_e2m1_f16(lds128(wrow + 16 * g), x), e8m0_to_f32(srow[g]), acc);
}

// Loads the f16 activations of the lane's groups from a prepared [L] f16 row.
template <int NR>
__device__ __forceinline__ void load_x_f16(const __half* row, const GroupMap& gm, int lane,
                                           uint32_t (&xr)[NR][16]) {
#pragma unroll
  for (int j = 0; j < NR; ++j) {
    const bool is_tail = (j == gm.F);
    const int g = is_tail ? gm.tail_group(lane) : lane + 32 * j;
    const bool ok = (j < gm.F) || (is_tail && gm.tail > 0 && gm.tail_ok(lane));
    if (ok) {
      const uint4* p = reinterpret_cast<const uint4*>(row + 32 * g);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = __ldg(p + q);
        xr[j][4 * q] = v.x;
        xr[j][4 * q + 1] = v.y;
        xr[j][4 * q + 2] = v.z;
        xr[j][4 * q + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 16; ++q) xr[j][q] = 0u;
    }
  }
}

// Loads fp32 activations of the lane's groups, finds the warp-wide largest magnitude and
// stores them as f16 scaled by 2^-e; returns e.  Every lane of the warp covers distinct
// groups and together they cover the whole vector, so e is the vector's exponent.
template <int NR>
__device__ __forceinline__ int load_act_f16(const float* row, const GroupMap& gm, int lane,
                                            uint32_t (&xr)[NR][16]) {
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < NR; ++j) {
    const bool is_tail = (j == gm.F);
    const int g = is_tail ? gm.tail_group(lane) : lane + 32 * j;
    const bool ok = (j < gm.F) || (is_tail && gm.tail > 0 && gm.tail_ok(lane));
    if (ok) {
      const float4* p = reinterpret_cast<const float4*>(row + 32 * g);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 v = __ldg(p + q);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      }
    }
  }
  m = warp_max(m);
  const int e = f16_exponent_for(m);
  const Pow2Scale sc(e);
#pragma unroll
  for (int j = 0; j < NR; ++j) {
    const bool is_tail = (j == gm.F);
    const int g = is_tail ? gm.tail_group(lane) : lane + 32 * j;
    const bool ok = (j < gm.F) || (is_tail && gm.tail > 0 && gm.tail_ok(lane));
    if (ok) {
      const float4* p = reinterpret_cast<const float4*>(row + 32 * g);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 v = __ldg(p + q);
        xr[j][2 * q] = pack_half2(sc(v.x), sc(v.y));
        xr[j][2 * q + 1] = pack_half2(sc(v.z), sc(v.w));
      }
    } else {
#pragma unroll
      for (int q = 0; q < 16; ++q) xr[j][q] = 0u;
    }
  }
  return e;
}

// Partial dot products of a row pair (A = row 0, B = row 1 of `w`, stride rowB; scales
// stride G) for this lane's groups.
template <int NR>
__device__ __forceinline__ void row_pair(const uint8_t* w, const uint8_t* s, uint32_t rowB, int G,
                                         const GroupMap& gm, int lane,
                                         const uint32_t (&xr)[NR][16], float& a, float& b) {
#pragma unroll
  for (int j = 0; j < NR; ++j) {
    if (j < gm.F) {
      const int g = lane + 32 * j;
      mx_group(w, s, g, xr[j], a);
      mx_group(w + rowB, s + G, g, xr[j], b);
    } else if (gm.tail > 0) {
      const int g = gm.tail_group(lane);
      if (gm.tail_ok(lane)) {
        if (gm.paired) {
          if (lane < 16) mx_group(w, s, g, xr[j], a);
          else mx_group(w + rowB, s + G, g, xr[j], b);
        } else {
          mx_group(w, s, g, xr[j], a);
          mx_group(w + rowB, s + G, g, xr[j], b);
        }
      }
    }
  }
}

// Sum of a (row A) and b (row B) over the warp: on return lanes 0-15 hold row A's sum and
// lanes 16-31 row B's.
__device__ __forceinline__ float pair_sum(float a, float b, int lane) {
  const bool hi = lane >= 16;
  float keep = hi ? b : a;
  keep += __shfl_xor_sync(kFull, hi ? a : b, 16);
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) keep += __shfl_xor_sync(kFull, keep, o);
  return keep;
}

// Per-stage item description written by the producer before it arms the stage's barrier
// (the barrier's release/acquire orders it for the consumers): the expert slot, row
// block, and the item's first kMetaAsg assignment ids, so consumers start an item without
// a global-memory round trip.
constexpr int kMetaAsg = 8;
struct StageMeta {
  int slot, rb, off, cnt;
  int asg[kMetaAsg];
};

__device__ __forceinline__ void fill_meta(StageMeta& m, int slot, int rb, const int32_t* seg_off,
                                          const int32_t* seg_cnt, const int32_t* perm) {
  m.slot = slot;
  m.rb = rb;
  m.off = seg_off[slot];
  m.cnt = seg_cnt[slot];
  const int n = m.cnt < kMetaAsg ? m.cnt : kMetaAsg;
  for (int i = 0; i < n; ++i) m.asg[i] = perm[m.off + i];
}

__device__ __forceinline__ int item_asg(const StageMeta& m, int tt, const int32_t* perm) {
  return tt < kMetaAsg ? m.asg[tt] : perm[m.off + tt];
}

template <int NR>
__global__ void __launch_bounds__(kThreads, 1) k_gemm1(const G1Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ StageMeta meta[8];
  const int L = a.L, I = a.I;
  const int G = L >> 5;
  const uint32_t rowB = (uint32_t)L >> 1;
  const uint32_t blkB = 16u * rowB;
  const uint32_t sclB = 16u * (uint32_t)G;
  const uint32_t stageB = 2u * blkB + 2u * sclB;
  const int S = a.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * stageB);
  uint64_t* empty = full + S;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch();

  const int NRB = I >> 4;
  const long long n_items = (long long)a.meta[0] * NRB;
  const long long i0 = n_items * blockIdx.x / gridDim.x;
  const long long i1 = n_items * (blockIdx.x + 1) / gridDim.x;

  if (warp == kConsumerWarps) {  // producer
    if (lane == 0) {
      for (long long i = i0; i < i1; ++i) {
        const int it = (int)(i - i0), s = it % S;
        if (it >= S && !mbar_wait(&empty[s], ((it / S) - 1) & 1, a.status)) break;
        const int slot = (int)(i / NRB), rb = (int)(i % NRB);
        fill_meta(meta[s], slot, rb, a.seg_off, a.seg_cnt, a.perm);
        const size_t row0 = (size_t)a.active[slot] * I + (size_t)rb * 16;
        uint8_t* st = smem + (size_t)s * stageB;
        mbar_arrive_expect_tx(&full[s], stageB);
        bulk_g2s(st, a.w1p + row0 * rowB, blkB, &full[s]);
        bulk_g2s(st + blkB, a.w3p + row0 * rowB, blkB, &full[s]);
        bulk_g2s(st + 2 * blkB, a.w1s + row0 * G, sclB, &full[s]);
        bulk_g2s(st + 2 * blkB + sclB, a.w3s + row0 * G, sclB, &full[s]);
      }
    }
    return;
  }

  const GroupMap gm(G);
  int cur_t = -1, xe = 0;
  uint32_t xr[NR][16];
  for (long long i = i0; i < i1; ++i) {
    const int it = (int)(i - i0), s = it % S;
    if (!mbar_wait(&full[s], (it / S) & 1, a.status)) break;  // every consumer warp times out alike
    const StageMeta& md = meta[s];
    const uint8_t* st = smem + (size_t)s * stageB;
    const uint8_t* w1 = st + (size_t)(2 * warp) * rowB;
    const uint8_t* w3 = w1 + blkB;
    const uint8_t* s1 = st + 2 * blkB + (2 * warp) * G;
    const uint8_t* s3 = s1 + sclB;
    const int rb = md.rb, cnt = md.cnt;
    for (int tt = 0; tt < cnt; ++tt) {
      const int asg = item_asg(md, tt, a.perm);
      const int t = asg / a.k;
      if (t != cur_t) {
        load_x_f16<NR>(a.x16 + (size_t)t * L, gm, lane, xr);
        xe = a.xexp[t];
        cur_t = t;
      }
      float gA = 0.f, gB = 0.f, uA = 0.f, uB = 0.f;
      row_pair<NR>(w1, s1, rowB, G, gm, lane, xr, gA, gB);
      row_pair<NR>(w3, s3, rowB, G, gm, lane, xr, uA, uB);
      const float gs = pair_sum(gA, gB, lane);
      const float us = pair_sum(uA, uB, lane);
      if ((lane & 15) == 0) {
        const float av = activation(ldexpf(gs, xe), ldexpf(us, xe), a.act_kind, a.b1, a.b2);
        a.act[(size_t)asg * I + (size_t)rb * 16 + 2 * warp + (lane >> 4)] = av;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

template <int NR>
__global__ void __launch_bounds__(kThreads, 1) k_gemm2(const G2Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ StageMeta meta[8];
  const int L = a.L, I = a.I;
  const int G = I >> 5;
  const uint32_t rowB = (uint32_t)I >> 1;
  const uint32_t blkB = 32u * rowB;
  const uint32_t sclB = 32u * (uint32_t)G;
  const uint32_t stageB = blkB + sclB;
  const int S = a.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * stageB);
  uint64_t* empty = full + S;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch();

  const int NRB = L >> 5;
  const long long n_items = (long long)a.meta[0] * NRB;
  const long long i0 = n_items * blockIdx.x / gridDim.x;
  const long long i1 = n_items * (blockIdx.x + 1) / gridDim.x;

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      for (long long i = i0; i < i1; ++i) {
        const int it = (int)(i - i0), s = it % S;
        if (it >= S && !mbar_wait(&empty[s], ((it / S) - 1) & 1, a.status)) break;
        const int slot = (int)(i / NRB), rb = (int)(i % NRB);
        fill_meta(meta[s], slot, rb, a.seg_off, a.seg_cnt, a.perm);
        const size_t row0 = (size_t)a.active[slot] * L + (size_t)rb * 32;
        uint8_t* st = smem + (size_t)s * stageB;
        mbar_arrive_expect_tx(&full[s], stageB);
        bulk_g2s(st, a.w2p + row0 * rowB, blkB, &full[s]);
        bulk_g2s(st + blkB, a.w2s + row0 * G, sclB, &full[s]);
      }
    }
    return;
  }

  const GroupMap gm(G);
  const int nq = L >> 2;  // 4-row counters per token
  int cur_a = -1, ae = 0;
  float gw = 0.f;
  uint32_t xr[NR][16];
  // The combine counter of the previous (token, 4-row) slot is checked one slot later, so
  // the atomic's round trip overlaps the next slot's arithmetic.
  int pend_t = -1, pend_row0 = 0, pend_prev = 0;
  auto resolve = [&]() {
    if (pend_t < 0) return;
    const int last = __shfl_sync(kFull, (lane == 0) ? (pend_prev == a.nvalid[pend_t] - 1) : 0, 0);
    if (last) {
      // acquire: the other slots' stores (each released by its counter increment) are visible
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      if (lane < 4) {
        float acc = 0.f;
        for (int j = 0; j < a.k; ++j) {
          const int e = a.idx[(size_t)pend_t * a.k + j];
          if (e < 0 || e >= a.E) continue;
          acc += __ldcg(a.ybuf + ((size_t)pend_t * a.k + j) * L + pend_row0 + lane);
        }
        a.y[(size_t)pend_t * L + pend_row0 + lane] = acc;
      }
    }
    pend_t = -1;
  };
  for (long long i = i0; i < i1; ++i) {
    const int it = (int)(i - i0), s = it % S;
    if (!mbar_wait(&full[s], (it / S) & 1, a.status)) break;
    const StageMeta& md = meta[s];
    const uint8_t* st = smem + (size_t)s * stageB;
    const uint8_t* wp = st + (size_t)(4 * warp) * rowB;
    const uint8_t* sp = st + blkB + (4 * warp) * G;
    const int row0 = md.rb * 32 + 4 * warp;  // this warp's 4 rows: row0 .. row0+3
    const int cnt = md.cnt;
    for (int tt = 0; tt < cnt; ++tt) {
      const int asg = item_asg(md, tt, a.perm);
      if (asg != cur_a) {
        ae = load_act_f16<NR>(a.act + (size_t)asg * I, gm, lane, xr);
        gw = a.gate[asg];
        cur_a = asg;
      }
      float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
      row_pair<NR>(wp, sp, rowB, G, gm, lane, xr, o0, o1);
      row_pair<NR>(wp + 2 * rowB, sp + 2 * G, rowB, G, gm, lane, xr, o2, o3);
      const float p01 = pair_sum(o0, o1, lane);  // lanes 0-15: row0, 16-31: row0+1
      const float p23 = pair_sum(o2, o3, lane);  // lanes 0-15: row0+2, 16-31: row0+3
      const float r1 = __shfl_sync(kFull, p01, 16);
      const float r3 = __shfl_sync(kFull, p23, 16);
      resolve();
      const int t = asg / a.k;
      if (lane == 0) {
        *reinterpret_cast<float4*>(a.ybuf + (size_t)asg * L + row0) =
            make_float4(gw * ldexpf(p01, ae), gw * ldexpf(r1, ae), gw * ldexpf(p23, ae),
                        gw * ldexpf(r3, ae));
        // release: the slot's store is ordered before the count
        asm volatile("atom.add.release.gpu.global.s32 %0, [%1], 1;"
                     : "=r"(pend_prev)
                     : "l"(a.cnt + (size_t)t * nq + (row0 >> 2))
                     : "memory");
      }
      pend_t = t;
      pend_row0 = row0;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  resolve();
}

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

template <typename Args>
cudaError_t launch_smem(void (*kern)(Args), const Args& a, int grid, size_t smem, cudaStream_t s,
                        bool pdl) {
  // The opt-in shared-memory limit is set once per kernel and device.
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || configured[dev] < (int)smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = (int)smem;
  }
  return launch_kernel(kern, dim3(grid), dim3(kThreads), smem, s, pdl, a);
}

constexpr size_t kSmemBudget = 200 * 1024;

int choose_stages(size_t stageB) {
  int S = (int)(kSmemBudget / stageB);
  return S > 4 ? 4 : S;
}

}  // namespace

cudaError_t launch_prep_x(const uint16_t* x, int T, int L, __half* x16, int32_t* xexp,
                          cudaStream_t s, bool pdl) {
  return launch_kernel(k_prep_x, dim3(T), dim3(256), 0, s, pdl, x, L, x16, xexp);
}

cudaError_t launch_gemm1(const ExpertPtrs& w, int L, int I, int E, int T, int k,
                         const __half* x16, const int32_t* xexp, const BucketOut& b,
                         float* act, int act_kind, float b1, float b2, int32_t* status,
                         cudaStream_t s, bool pdl) {
  G1Args a{w.w1p, w.w1s, w.w3p, w.w3s, L, I, k, x16, xexp, b.active, b.seg_off, b.seg_cnt,
           b.meta, b.perm, act, act_kind, b1, b2, status, 0};
  const size_t stageB = 17u * (size_t)L;
  a.stages = choose_stages(stageB);
  const size_t smem = a.stages * stageB + 16u * a.stages;
  const long long max_items = (long long)std::min(E, T * k) * (I >> 4);
  const int grid = (int)std::min<long long>(sm_count(), std::max<long long>(1, max_items));
  switch (((L >> 5) + 31) >> 5) {
    case 1: return launch_smem(k_gemm1<1>, a, grid, smem, s, pdl);
    case 2: return launch_smem(k_gemm1<2>, a, grid, smem, s, pdl);
    case 3: return launch_smem(k_gemm1<3>, a, grid, smem, s, pdl);
    case 4: return launch_smem(k_gemm1<4>, a, grid, smem, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm2(const ExpertPtrs& w, int L, int I, int E, int T, int k,
                         const float* act, const float* gate, const int32_t* idx,
                         const BucketOut& b, float* ybuf, int32_t* cnt, float* y,
                         int32_t* status, cudaStream_t s, bool pdl) {
  G2Args a{w.w2p, w.w2s, L, I, k, E, act, gate, idx, b.active, b.seg_off, b.seg_cnt, b.meta,
           b.perm, b.nvalid, ybuf, cnt, y, status, 0};
  const size_t stageB = 17u * (size_t)I;
  a.stages = choose_stages(stageB);
  const size_t smem = a.stages * stageB + 16u * a.stages;
  const long long max_items = (long long)std::min(E, T * k) * (L >> 5);
  const int grid = (int)std::min<long long>(sm_count(), std::max<long long>(1, max_items));
  switch (((I >> 5) + 31) >> 5) {
    case 1: return launch_smem(k_gemm2<1>, a, grid, smem, s, pdl);
    case 2: return launch_smem(k_gemm2<2>, a, grid, smem, s, pdl);
    case 3: return launch_smem(k_gemm2<3>, a, grid, smem, s, pdl);
    case 4: return launch_smem(k_gemm2<4>, a, grid, smem, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_matvec(float* y, const uint16_t* x, const uint8_t* packed,
                          const uint8_t* scales, int in, int rows, cudaStream_t s) {
  return launch_kernel(k_matvec, dim3((rows + 7) / 8), dim3(256), 0, s, false, y, x, packed,
                       scales, in, rows);
}

}  // namespace k3
