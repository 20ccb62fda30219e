// experts.cu -- the routed experts' MXFP4 grouped GEMV (decode-sized batches).
//
// README "kimi-k3-in-c", Part II section 4: the expert weights are multiplied straight from
// their packed form and never expanded in memory.  Per expert e and token t:
//   g = W1[e] x_t,  u = W3[e] x_t,  act = silu(g) * u  (or SiTU-GLU)      -- MODE 0 (GEMM1)
//   ybuf[t*k+j] = gate[t][j] * W2[e] act                                  -- MODE 1 (GEMM2)
//   y[t] = sum_j ybuf[t*k+j]  (slot order, deterministic)                 -- k_combine
//
// GB300 design.  One persistent CTA per SM walks a contiguous range of work items; an item
// is two 16-row tiles of one expert (MODE 0: rows r..r+15 of w1 and of w3; MODE 1: rows
// r..r+31 of w2) and all of that expert's tokens.  A producer warp moves each item's packed
// rows and E8M0 scales from HBM into a shared-memory ring with bulk asynchronous copies
// (cp.async.bulk, completion counted on an mbarrier, rows padded by 16 bytes so the
// consumers' fragment loads are free of bank conflicts), several items ahead of the eight
// consumer warps.  Consumer warp w owns MX groups [w*G/8, (w+1)*G/8) of both tiles.  For each
// group a lane loads 4 packed bytes of row (lane/4) and of row (lane/4)+8, turns each nibble
// pair into an exact f16 pair in hardware (cvt e2m1x2; low nibble = even column) -- these
// pairs are directly the A fragments of two m16n8k16 tensor-core MMAs -- and the tokens'
// activations, stored as f16 scaled by a power of two per vector, are the B fragments (up
// to 8 tokens share every decoded weight).  The fp32 MMA result of each group is multiplied
// by the rows' E8M0 scales and accumulated; products are exact, sums are fp32.  The eight
// warps' partial sums meet in shared memory in a fixed order (deterministic), and the
// epilogue applies SwiGLU (MODE 0) or the gate (MODE 1).
//
// Every wait is bounded: a wait that runs out is counted in the status block, and all
// consumer warps stop at the same item (they share every named barrier).
#include "launch.h"

namespace k3 {
namespace {

constexpr int kGroupWarps = 4;             // consumer warps per stage: 2 tiles x 2 K halves
constexpr int kMaxStages = 3;              // stages = consumer warp groups
constexpr int kThreadsX = 32 * (kMaxStages * kGroupWarps + 1);  // + one producer warp
constexpr int kRows = 16;                  // rows per tile (MMA M)
constexpr int kMaxNT = 8;                  // tokens per tile (MMA N)
constexpr int kMetaAsg = 8;

struct XArgs {
  // MODE 0: A0 = w1, A1 = w3 (rows r..r+15 of each); MODE 1: A0 = A1 = w2 (rows r.., r+16..)
  const uint8_t *p0, *s0, *p1, *s1;
  int K;             // reduction width: L (MODE 0) or I (MODE 1)
  int rows_total;    // rows per expert: I (MODE 0) or L (MODE 1)
  int item_rows;     // 16 (MODE 0) or 32 (MODE 1)
  int k;             // experts per token
  const __half* x16;       // MODE 0 activations [T][L] f16, scaled by 2^-xexp[t]
  const int32_t* xexp;
  const float* act_in;     // MODE 1 activations [T*k][I] fp32
  const float* gate;       // MODE 1 gates [T*k]
  const int32_t *active, *seg_off, *seg_cnt, *meta, *perm;
  float* out;              // MODE 0: act [T*k][I]; MODE 1: ybuf [T*k][L]
  int act_kind;
  float b1, b2;
  int32_t* status;
  int stages, ntx;
};

struct StageMeta {
  int slot, rb, off, cnt;
  int asg[kMetaAsg];
};

// An expert slot of the CTA's item range, as the producer needs it.
struct SlotInfo {
  int expert, off, cnt;
  int asg[kMetaAsg];
};
constexpr int kSlotTable = 32;

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// OR of a flag over one consumer group (4 warps) through the group's named barrier.
__shared__ int g_or_scratch[kMaxStages];
__device__ __forceinline__ int __syncthreads_or_group(int v, uint32_t bar) {
  const int q = (int)bar - 1;
  const int any = __any_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0 && threadIdx.x % (32 * kGroupWarps) == 0) g_or_scratch[q] = 0;
  named_bar(bar, 32 * kGroupWarps);
  if ((threadIdx.x & 31) == 0 && any) atomicOr(&g_or_scratch[q], 1);
  named_bar(bar, 32 * kGroupWarps);
  const int r = g_or_scratch[q];
  named_bar(bar, 32 * kGroupWarps);
  return r;
}

// D = A * B (+ 0): one m16n8k16 MMA with f16 inputs and fp32 accumulation.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One MX group of one 16-row tile against one 8-column activation tile.
//   wa / wb: this lane's 4 packed bytes (8 nibbles) of rows gid and gid+8; the lane's
//   logical K positions 2t,2t+1 / 2t+8,2t+9 of MMA step s are the group's columns
//   8t+4s+{0,1} / 8t+4s+{2,3}, and xb holds the activations of those 8 columns.
__device__ __forceinline__ void group_mma(uint32_t wa, uint32_t wb, const uint4& xb, float (&c)[4]) {
  uint32_t ha[4], hb[4];
  e2m1x8_to_f16x2(wa, ha);
  e2m1x8_to_f16x2(wb, hb);
  c[0] = c[1] = c[2] = c[3] = 0.f;
  mma16816(c, ha[0], hb[0], ha[1], hb[1], xb.x, xb.y);
  mma16816(c, ha[2], hb[2], ha[3], hb[3], xb.z, xb.w);
}

// KC: the reduction width at compile time (0 = read from the arguments); the Kimi-K3
// widths are compiled so that every shared-memory offset in the inner loop is an immediate.
template <int MODE, bool ONE, int KC>
__global__ void __launch_bounds__(kThreadsX, 1) k_experts(const XArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ StageMeta meta[kMaxStages];
  __shared__ SlotInfo slot_tab[kSlotTable];
  __shared__ int xtile_asg[kMaxStages][kMaxNT];  // assignment ids of each group's activation rows
  __shared__ int xtile_exp[kMaxStages][kMaxNT];  // their power-of-two exponents
  __shared__ int abort_flag;

  const int K = KC ? KC : a.K, G = K >> 5, S = a.stages, NTX = a.ntx;
  const uint32_t RS = (uint32_t)(K >> 1) + 16u;       // padded packed-row stride
  const uint32_t tileB = kRows * RS;
  const uint32_t sclB = kRows * (uint32_t)G;
  const uint32_t stageB = 2u * tileB + 2u * sclB;
  const uint32_t RSX = 2u * (uint32_t)K + 64u;        // activation-row stride (bytes)
  uint8_t* xt_all = smem + (size_t)S * stageB;                          // [S][NTX] rows
  float* red_all = reinterpret_cast<float*>(xt_all + (size_t)S * NTX * RSX);  // [S][4][2][16][8]
  uint64_t* full = reinterpret_cast<uint64_t*>(red_all + (size_t)S * 8 * kRows * kMaxNT);
  uint64_t* empty = full + S;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGroupWarps);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  pdl_wait();
  pdl_launch();

  const int NRB = a.rows_total / a.item_rows;
  const long long n_items = (long long)a.meta[0] * NRB;
  const long long i0 = n_items * blockIdx.x / gridDim.x;
  const long long i1 = n_items * (blockIdx.x + 1) / gridDim.x;
  const int producer_warp = kMaxStages * kGroupWarps;

  if (warp == producer_warp) {  // producer: one lane issues the bulk copies
    // The CTA's expert slots, read once: the copy loop then needs no global-memory round
    // trip before it can issue an item.
    const int slot_lo = (int)(i0 / NRB);
    const int n_slots = i1 > i0 ? (int)((i1 - 1) / NRB) - slot_lo + 1 : 0;
    const bool tabled = n_slots <= kSlotTable;
    if (tabled) {
      for (int v = lane; v < n_slots; v += 32) {
        const int sl = slot_lo + v;
        slot_tab[v].expert = a.active[sl];
        slot_tab[v].off = a.seg_off[sl];
        slot_tab[v].cnt = a.seg_cnt[sl];
        const int n = slot_tab[v].cnt < kMetaAsg ? slot_tab[v].cnt : kMetaAsg;
        for (int q = 0; q < n; ++q) slot_tab[v].asg[q] = a.perm[slot_tab[v].off + q];
      }
      __syncwarp();
    }
    if (lane == 0) {
      for (long long i = i0; i < i1; ++i) {
        const int it = (int)(i - i0), s = it % S;
        if (it >= S && !mbar_wait(&empty[s], ((it / S) - 1) & 1, a.status)) break;
        if (*reinterpret_cast<volatile int*>(&abort_flag)) break;
        const int slot = (int)(i / NRB), rb = (int)(i % NRB);
        StageMeta& m = meta[s];
        m.slot = slot;
        m.rb = rb;
        int expert;
        if (tabled) {
          const SlotInfo& si = slot_tab[slot - slot_lo];
          expert = si.expert;
          m.off = si.off;
          m.cnt = si.cnt;
          const int n = m.cnt < kMetaAsg ? m.cnt : kMetaAsg;
          for (int q = 0; q < n; ++q) m.asg[q] = si.asg[q];
        } else {
          expert = a.active[slot];
          m.off = a.seg_off[slot];
          m.cnt = a.seg_cnt[slot];
          const int n = m.cnt < kMetaAsg ? m.cnt : kMetaAsg;
          for (int q = 0; q < n; ++q) m.asg[q] = a.perm[m.off + q];
        }
        const size_t row0 = (size_t)expert * a.rows_total + (size_t)rb * a.item_rows;
        const size_t row1 = MODE == 0 ? row0 : row0 + kRows;
        const uint8_t* p1 = MODE == 0 ? a.p1 : a.p0;
        const uint8_t* s1 = MODE == 0 ? a.s1 : a.s0;
        uint8_t* st = smem + (size_t)s * stageB;
        const uint32_t rowB = (uint32_t)(K >> 1);
        mbar_arrive_expect_tx(&full[s], 2u * kRows * rowB + 2u * sclB);
        for (int r = 0; r < kRows; ++r) {
          bulk_g2s(st + r * RS, a.p0 + (row0 + r) * rowB, rowB, &full[s]);
          bulk_g2s(st + tileB + r * RS, p1 + (row1 + r) * rowB, rowB, &full[s]);
        }
        bulk_g2s(st + 2 * tileB, a.s0 + row0 * G, sclB, &full[s]);
        bulk_g2s(st + 2 * tileB + sclB, s1 + row1 * G, sclB, &full[s]);
      }
    }
    return;
  }

  // consumers: warp group q owns stage q; warp (tl, kh) of the group handles tile tl over
  // the K half kh
  const int q = warp / kGroupWarps, wq = warp % kGroupWarps;
  if (q >= S) return;
  const int gid = lane >> 2, t4 = lane & 3;
  const int gbeg = wq * G / kGroupWarps, gend = (wq + 1) * G / kGroupWarps;
  const int gtid = wq * 32 + lane;  // 0..127 within the group
  const uint32_t bar = 1 + q;       // the group's named barrier
  uint8_t* xt = xt_all + (size_t)q * NTX * RSX;
  float* red = red_all + (size_t)q * 8 * kRows * kMaxNT;
  int loaded[kMaxNT];
#pragma unroll
  for (int n = 0; n < kMaxNT; ++n) loaded[n] = -1;
  int loaded_n = 0;

  for (long long i = i0 + q; i < i1; i += S) {
    const int it = (int)(i - i0), s = q;
    const bool ok = mbar_wait(&full[s], (it / S) & 1, a.status);
    if (!ok) abort_flag = 1;
    const StageMeta& md = meta[s];
    const int cnt = md.cnt, rb = md.rb;
    const uint8_t* st = smem + (size_t)s * stageB;
    // does the stage hold a scale byte of 0 or 255 (the two that are not a plain exponent)?
    int special = 0;
    for (int v = gtid; v < (int)(2 * sclB / 4); v += 32 * kGroupWarps) {
      const uint32_t w = lds32(st + 2 * tileB + 4 * v);
      const uint32_t z = (w - 0x01010101u) & ~w & 0x80808080u;          // a zero byte
      const uint32_t f = ((~w) - 0x01010101u) & w & 0x80808080u;        // a 0xFF byte
      special |= (z | f) != 0u;
    }
    const bool plain_scales = __syncthreads_or_group(special, bar) == 0;
    bool stop = false;
    for (int nt0 = 0; nt0 < cnt && !stop; nt0 += NTX) {
      const int nn = min(NTX, cnt - nt0);
      // ---- the group's activation tile: rows = this n-tile's assignments
      int key[kMaxNT];
      bool same = (nn == loaded_n);
#pragma unroll
      for (int n = 0; n < kMaxNT; ++n) {
        key[n] = -1;
        if (n < nn) {
          const int qq = nt0 + n;
          const int asg = qq < kMetaAsg ? md.asg[qq] : a.perm[md.off + qq];
          key[n] = MODE == 0 ? asg / a.k : asg;
          if (key[n] != loaded[n]) same = false;
        }
      }
      if (!same) {
        named_bar(bar, 32 * kGroupWarps);  // nobody in the group reads the old tile any more
        if (MODE == 0) {
          const int nvec = K >> 3;  // 16-byte pieces per row
          for (int v = gtid; v < nn * nvec; v += 32 * kGroupWarps) {
            const int n = v / nvec, c = v - n * nvec;
            const int tok = n == 0 ? key[0] : (n == 1 ? key[1] : (n == 2 ? key[2] : (n == 3 ? key[3] :
                            (n == 4 ? key[4] : (n == 5 ? key[5] : (n == 6 ? key[6] : key[7]))))));
            const uint4 val = __ldg(reinterpret_cast<const uint4*>(a.x16 + (size_t)tok * K) + c);
            *reinterpret_cast<uint4*>(xt + (size_t)n * RSX + 16 * c) = val;
          }
          if (wq == 0) {
#pragma unroll
            for (int n = 0; n < kMaxNT; ++n)
              if (lane == n && n < nn) xtile_exp[q][n] = a.xexp[key[n]];
          }
        } else {
          // warp wq converts rows wq, wq+4: fp32 activations -> f16 scaled by the row's exponent
#pragma unroll
          for (int n = 0; n < kMaxNT; ++n) {
            if (n % kGroupWarps != wq || n >= nn) continue;
            const float4* src = reinterpret_cast<const float4*>(a.act_in + (size_t)key[n] * K);
            float m = 0.f;
            for (int c = lane; c < (K >> 2); c += 32) {
              const float4 v = __ldg(src + c);
              m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
            m = warp_max(m);
            const int e = f16_exponent_for(m);
            const Pow2Scale sc(e);
            for (int c = lane; c < (K >> 2); c += 32) {
              const float4 v = __ldg(src + c);
              uint2 o;
              o.x = pack_half2(sc(v.x), sc(v.y));
              o.y = pack_half2(sc(v.z), sc(v.w));
              *reinterpret_cast<uint2*>(xt + (size_t)n * RSX + 8 * c) = o;
            }
            if (lane == 0) xtile_exp[q][n] = e;
          }
        }
        if (wq == 0) {
#pragma unroll
          for (int n = 0; n < kMaxNT; ++n)
            if (lane == n && n < nn) xtile_asg[q][n] = key[n];
        }
        named_bar(bar, 32 * kGroupWarps);
#pragma unroll
        for (int n = 0; n < kMaxNT; ++n) loaded[n] = key[n];
        loaded_n = nn;
      }
      // ---- both tiles over this warp's K quarter
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint8_t* xrow = xt + (size_t)min(gid, nn - 1) * RSX + 16 * t4;
      const uint8_t* wrow = st + gid * RS + 4 * t4;
      const uint8_t* srow = st + 2 * tileB + gid * G;
      if (plain_scales) {
        // every scale byte of the stage is in 1..254: 2^(s-127) is the byte in the exponent
#pragma unroll 4
        for (int g = gbeg; g < gend; ++g) {
          const uint4 xb = *reinterpret_cast<const uint4*>(xrow + 64 * g);
#pragma unroll
          for (int tl = 0; tl < 2; ++tl) {
            const uint8_t* tb = wrow + tl * tileB + 16 * g;
            const uint8_t* sr = srow + tl * sclB + g;
            const float sa = __uint_as_float((uint32_t)sr[0] << 23);
            const float sbv = __uint_as_float((uint32_t)sr[8 * G] << 23);
            float c[4];
            group_mma(lds32(tb), lds32(tb + 8 * RS), xb, c);
            acc[tl][0] = fmaf(c[0], sa, acc[tl][0]);
            acc[tl][2] = fmaf(c[2], sbv, acc[tl][2]);
            if (!ONE) {
              acc[tl][1] = fmaf(c[1], sa, acc[tl][1]);
              acc[tl][3] = fmaf(c[3], sbv, acc[tl][3]);
            }
          }
        }
      } else {
        for (int g = gbeg; g < gend; ++g) {
          const uint4 xb = *reinterpret_cast<const uint4*>(xrow + 64 * g);
#pragma unroll
          for (int tl = 0; tl < 2; ++tl) {
            const uint8_t* tb = wrow + tl * tileB + 16 * g;
            const uint8_t* sr = srow + tl * sclB + g;
            const float sa = e8m0_to_f32(sr[0]), sbv = e8m0_to_f32(sr[8 * G]);
            float c[4];
            group_mma(lds32(tb), lds32(tb + 8 * RS), xb, c);
            acc[tl][0] = fmaf(c[0], sa, acc[tl][0]);
            acc[tl][2] = fmaf(c[2], sbv, acc[tl][2]);
            if (!ONE) {
              acc[tl][1] = fmaf(c[1], sa, acc[tl][1]);
              acc[tl][3] = fmaf(c[3], sbv, acc[tl][3]);
            }
          }
        }
      }
      // ---- the four K quarters of both tiles meet in the group's buffer [wq][tile][row][col]
#pragma unroll
      for (int tl = 0; tl < 2; ++tl) {
        float* r = red + ((size_t)wq * 2 + tl) * (kRows * kMaxNT);
        r[gid * kMaxNT + 2 * t4] = acc[tl][0];
        r[(gid + 8) * kMaxNT + 2 * t4] = acc[tl][2];
        if (!ONE) {
          r[gid * kMaxNT + 2 * t4 + 1] = acc[tl][1];
          r[(gid + 8) * kMaxNT + 2 * t4 + 1] = acc[tl][3];
        }
      }
      named_bar(bar, 32 * kGroupWarps);
      if (*reinterpret_cast<volatile int*>(&abort_flag)) {
        stop = true;
        break;
      }
      const int RC = kRows * kMaxNT;
      if (MODE == 0) {
        // thread -> (row, token column); SwiGLU of (w1 row, w3 row)
        const int row = gtid >> 3, n = gtid & 7;
        if (n < nn) {
          float g = 0.f, u = 0.f;
#pragma unroll
          for (int w = 0; w < kGroupWarps; ++w) {
            g += red[(2 * w + 0) * RC + row * kMaxNT + n];
            u += red[(2 * w + 1) * RC + row * kMaxNT + n];
          }
          const int xe = xtile_exp[q][n];
          const int asg = nt0 + n < kMetaAsg ? md.asg[nt0 + n] : a.perm[md.off + nt0 + n];
          const float av = activation(ldexpf(g, xe), ldexpf(u, xe), a.act_kind, a.b1, a.b2);
          a.out[(size_t)asg * a.rows_total + (size_t)rb * kRows + row] = av;
        }
      } else {
        // thread -> (row, token column) of each tile; gate * o into the assignment's slot
        const int row = gtid >> 3, n = gtid & 7;
        if (n < nn) {
          const int asg = xtile_asg[q][n];
          const float gw = a.gate[asg];
          const int e = xtile_exp[q][n];
          float o0 = 0.f, o1 = 0.f;
#pragma unroll
          for (int w = 0; w < kGroupWarps; ++w) {
            o0 += red[(2 * w + 0) * RC + row * kMaxNT + n];
            o1 += red[(2 * w + 1) * RC + row * kMaxNT + n];
          }
          float* dst = a.out + (size_t)asg * a.rows_total + (size_t)rb * 2 * kRows + row;
          dst[0] = gw * ldexpf(o0, e);
          dst[kRows] = gw * ldexpf(o1, e);
        }
      }
      named_bar(bar, 32 * kGroupWarps);  // the buffer is free for the next n-tile
    }
    if (stop) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// y[t][c] = sum over valid j of ybuf[t*k+j][c], in slot order (deterministic).  Slots are
// taken kBatch at a time: their experts first, then their rows (independent loads in
// flight), then added in order.  Small batches take 16 (the rows were just written and sit
// in L2: the time is the loads' latency); large ones 4 (HBM-bound: 16 costs registers and
// with them resident blocks, 143 -> 208 us at 4096 tokens).
template <int kBatch>
__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ ybuf,
                                                 const int32_t* __restrict__ idx, int k, int E,
                                                 int L, float* __restrict__ y) {
  pdl_wait();
  pdl_launch();
  const int t = blockIdx.y;
  const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
  if (c4 * 4 >= L) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < k; j0 += kBatch) {
    int e[kBatch];
#pragma unroll
    for (int jj = 0; jj < kBatch; ++jj)
      e[jj] = j0 + jj < k ? __ldg(idx + (size_t)t * k + j0 + jj) : -1;
    float4 v[kBatch];
    bool ok[kBatch];
#pragma unroll
    for (int jj = 0; jj < kBatch; ++jj) {
      ok[jj] = e[jj] >= 0 && e[jj] < E;
      if (ok[jj])
        v[jj] = __ldcs(reinterpret_cast<const float4*>(ybuf + ((size_t)t * k + j0 + jj) * L) + c4);
    }
#pragma unroll
    for (int jj = 0; jj < kBatch; ++jj) {
      if (ok[jj]) {
        acc.x += v[jj].x;
        acc.y += v[jj].y;
        acc.z += v[jj].z;
        acc.w += v[jj].w;
      }
    }
  }
  reinterpret_cast<float4*>(y + (size_t)t * L)[c4] = acc;
}

template <int MODE, bool ONE, int KC>
cudaError_t launch_k(const XArgs& a, int grid, size_t smem, cudaStream_t s, bool pdl) {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || configured[dev] < (int)smem) {
    cudaError_t e = cudaFuncSetAttribute(k_experts<MODE, ONE, KC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = (int)smem;
  }
  return launch_kernel(k_experts<MODE, ONE, KC>, dim3(grid), dim3(kThreadsX), smem, s, pdl, a);
}

template <int MODE, bool ONE>
cudaError_t launch_mode(const XArgs& a, int grid, size_t smem, cudaStream_t s, bool pdl) {
  if (MODE == 0 && a.K == 3584) return launch_k<MODE, ONE, 3584>(a, grid, smem, s, pdl);
  if (MODE == 1 && a.K == 3072) return launch_k<MODE, ONE, 3072>(a, grid, smem, s, pdl);
  return launch_k<MODE, ONE, 0>(a, grid, smem, s, pdl);
}

constexpr size_t kSmemMax = 225 * 1024;  // dynamic shared memory (static use stays below 2 KB)

// Ring depth (= consumer warp groups) and activation-tile height for a reduction width K
// and batch T.
bool plan(int K, int T, int* stages, int* ntx, size_t* smem) {
  const size_t G = K >> 5;
  const size_t stageB = 2 * kRows * ((size_t)(K >> 1) + 16) + 2 * kRows * G;
  const size_t xrow = 2 * (size_t)K + 64;
  for (int nt = T < kMaxNT ? T : kMaxNT; nt >= 1; nt = (nt == 1 ? 0 : (nt + 1) / 2)) {
    for (int S = kMaxStages; S >= 2; --S) {
      const size_t per = stageB + (size_t)nt * xrow + 8 * kRows * kMaxNT * sizeof(float) + 16;
      if ((size_t)S * per + 64 <= kSmemMax) {
        *stages = S;
        *ntx = nt;
        *smem = (size_t)S * per + 64;
        return true;
      }
    }
    if (nt == 1) break;
  }
  return false;
}

cudaError_t launch_experts(int mode, XArgs a, int E, int T, cudaStream_t s, bool pdl) {
  int stages, ntx;
  size_t smem;
  if (!plan(a.K, T, &stages, &ntx, &smem)) return cudaErrorInvalidValue;
  a.stages = stages;
  a.ntx = ntx;
  const long long max_items = (long long)std::min(E, T * a.k) * (a.rows_total / a.item_rows);
  const int grid = (int)std::min<long long>(sm_count(), std::max<long long>(1, max_items));
  const bool one = (ntx == 1);
  if (mode == 0)
    return one ? launch_mode<0, true>(a, grid, smem, s, pdl) : launch_mode<0, false>(a, grid, smem, s, pdl);
  return one ? launch_mode<1, true>(a, grid, smem, s, pdl) : launch_mode<1, false>(a, grid, smem, s, pdl);
}

}  // namespace

cudaError_t launch_gemm1(const ExpertPtrs& w, int L, int I, int E, int T, int k,
                         const __half* x16, const int32_t* xexp, const BucketOut& b,
                         float* act, int act_kind, float b1, float b2, int32_t* status,
                         cudaStream_t s, bool pdl) {
  XArgs a{};
  a.p0 = w.w1p; a.s0 = w.w1s; a.p1 = w.w3p; a.s1 = w.w3s;
  a.K = L; a.rows_total = I; a.item_rows = kRows; a.k = k;
  a.x16 = x16; a.xexp = xexp;
  a.active = b.active; a.seg_off = b.seg_off; a.seg_cnt = b.seg_cnt; a.meta = b.meta; a.perm = b.perm;
  a.out = act; a.act_kind = act_kind; a.b1 = b1; a.b2 = b2; a.status = status;
  return launch_experts(0, a, E, T, s, pdl);
}

cudaError_t launch_gemm2(const ExpertPtrs& w, int L, int I, int E, int T, int k,
                         const float* act, const float* gate, const BucketOut& b, float* ybuf,
                         int32_t* status, cudaStream_t s, bool pdl) {
  XArgs a{};
  a.p0 = w.w2p; a.s0 = w.w2s; a.p1 = w.w2p; a.s1 = w.w2s;
  a.K = I; a.rows_total = L; a.item_rows = 2 * kRows; a.k = k;
  a.act_in = act; a.gate = gate;
  a.active = b.active; a.seg_off = b.seg_off; a.seg_cnt = b.seg_cnt; a.meta = b.meta; a.perm = b.perm;
  a.out = ybuf; a.status = status;
  return launch_experts(1, a, E, T, s, pdl);
}

cudaError_t launch_combine(const float* ybuf, const int32_t* idx, int T, int k, int E, int L,
                           float* y, cudaStream_t s, bool pdl) {
  dim3 grid(((L >> 2) + 255) / 256, T);
  if (T <= 256) return launch_kernel(k_combine<16>, grid, dim3(256), 0, s, pdl, ybuf, idx, k, E, L, y);
  return launch_kernel(k_combine<4>, grid, dim3(256), 0, s, pdl, ybuf, idx, k, E, L, y);
}

}  // namespace k3
