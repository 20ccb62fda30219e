// moe_tc.cu -- the routed experts on the block-scaled tensor cores (kind::mxf4).
//
// README "kimi-k3-in-c", Part II sections 4 and 9: every selected expert multiplies its
// packed E2M1 weights, one E8M0 scale per 32, straight from the checkpoint bytes:
//   g = W1[e] x,  u = W3[e] x,  act = silu(g) u (or SiTU-GLU),  o = W2[e] act,
//   y[t] = sum_j gate[t][j] o_j.
// Here the weights go from HBM to shared memory by TMA (128-byte swizzle) and from there
// straight into tcgen05.mma kind::mxf4 (E2M1 x E2M1, UE8M0 block scales, fp32 accumulation
// in tensor memory): the CUDA cores never touch a weight nibble.  The second operand is the
// activation written as kTerms MXFP4 terms per token (mxq.cuh), one MMA column per term; the
// hardware applies each term's scales, so a token's product is the sum of its columns.
//
// Work: tiles of 128 weight rows x (up to 16 of an expert's tokens) x the full reduction,
// cut into units of 512 reduction elements.  The grid is one CTA per SM; CTA c takes units
// [U c / G, U (c+1) / G) of the whole list (balanced to within one unit whatever the
// routing).  A tile cut between CTAs is finished by the CTA holding its first unit: the
// others leave their partial sums and a flag, and it adds them in CTA order (deterministic).
//
// Roles (320 threads): warps 0-3 epilogue (TMEM lane quarters 0-3), warps 4-7 move each
// stage's scales into TMEM (a 0xFF scale byte, "no value", becomes 0 there), warp 8 issues
// the TMA copies into a 4-stage ring, warp 9 allocates TMEM and issues the MMAs.  Every
// wait is bounded; one that runs out sets the status block's timeout count and the CTA
// stops issuing new work.
#include "launch.h"
#include "mxq.cuh"
#include "tc.cuh"
#include "tmap.h"

namespace k3 {
namespace {

constexpr int kStages = 4;
constexpr int kKStage = 512;                                 // reduction elements per stage
constexpr int kMmas = kKStage / 64;                          // MMAs per stage (K = 64 each)
constexpr int kTokTile = kTcTokTile;                         // tokens per tile
constexpr int kNMax = kTokTile * kTerms;                     // B rows (MMA N) per tile
constexpr int kRowsTile = 128;                               // MMA M
constexpr uint32_t kABytes = kRowsTile * (kKStage / 2);      // 32768
constexpr uint32_t kBBytes = kNMax * (kKStage / 2);          // 16384
constexpr uint32_t kSABytes = kRowsTile * (kKStage / 32);    // 2048
constexpr uint32_t kSBBytes = kNMax * (kKStage / 32);        // 1024
constexpr uint32_t kOffB = kABytes, kOffSA = kABytes + kBBytes, kOffSB = kOffSA + kSABytes;
constexpr uint32_t kStageBytes = kOffSB + kSBBytes;          // 52224 = 51 x 1024
constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + 1024;
constexpr int kThreads = 320;
constexpr int kSfWarp0 = 4, kProdWarp = 8, kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: accumulators in [0, 256), buffer b at 128 b, matrix m at + 64 m; the scale
// ring in [256, 512), stage s at 256 + 64 s: A scales of MMA j at + 4 j (+ lane quarter),
// B scales at + 32 + 4 j (+ 1 for B rows 32..63).
constexpr uint32_t kAccCols = 128, kSfBase = 256, kSfStageCols = 64;
constexpr int kEpiBar = 1;  // named barrier of the four epilogue warps

static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");

struct TcArgs {
  int K, R, KC, RT, k;
  const int32_t *active, *seg_off, *seg_cnt, *meta, *perm, *ntile_base;
  // GEMM1: activation terms out ([P * kTerms][I/2] codes, [P * kTerms][I/32] scales)
  uint8_t *act_q, *act_sf;
  int I, act_kind;
  float b1, b2;
  // GEMM2: gate-weighted per-assignment outputs [T*k][L]
  const float* gate;
  float* ybuf;
  // split tiles: partial sums [grid][2 * npart][128] and flags [grid]
  float* part;
  int npart;
  int32_t* flags;
  int32_t* status;
};

struct Cursor {
  int a, n, rt, kc, tile;
};

__device__ __forceinline__ void cursor_at(Cursor& c, long long u, const TcArgs& a) {
  const long long t = u / a.KC;
  c.kc = (int)(u - t * a.KC);
  c.tile = (int)t;
  const int ntg = (int)(t / a.RT);
  c.rt = (int)(t - (long long)ntg * a.RT);
  int lo = 0, hi = a.meta[0] - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.ntile_base[mid] <= ntg) lo = mid;
    else hi = mid - 1;
  }
  c.a = lo;
  c.n = ntg - a.ntile_base[lo];
}

__device__ __forceinline__ void cursor_next(Cursor& c, const TcArgs& a) {
  if (++c.kc < a.KC) return;
  c.kc = 0;
  ++c.tile;
  if (++c.rt < a.RT) return;
  c.rt = 0;
  if (++c.n < (a.seg_cnt[c.a] + kTokTile - 1) / kTokTile) return;
  c.n = 0;
  ++c.a;
}

struct TileInfo {
  int expert, pos0, ntok, N;
};
__device__ __forceinline__ TileInfo tile_info(const Cursor& c, const TcArgs& a) {
  TileInfo t;
  t.expert = a.active[c.a];
  t.pos0 = a.seg_off[c.a] + c.n * kTokTile;
  t.ntok = min(kTokTile, a.seg_cnt[c.a] - c.n * kTokTile);
  t.N = ((t.ntok * kTerms + 15) / 16) * 16;
  return t;
}

// bytes 0xFF -> 0x00 (an E8M0 "no value" becomes the smallest scale: the group adds nothing
// measurable, as the pages' decoder's zero group)
__device__ __forceinline__ uint32_t clear_ff_bytes(uint32_t w) {
  const uint32_t t = ~w;
  const uint32_t y = ((t & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | t;  // bit 7 clear iff the byte of t is 0
  const uint32_t ff = (~y & 0x80808080u) >> 7;
  return w & ~(ff * 0xFFu);
}

__device__ __forceinline__ int bar_or(uint32_t id, uint32_t n, int v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v), "r"(id), "r"(n)
      : "memory");
  return (int)r;
}

__device__ __forceinline__ void st_release(int32_t* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// 16 TMEM columns of this warp's lane quarter into registers (load and wait in one asm, so
// no register is read before the data is there)
__device__ __forceinline__ void tmem_load16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "{\n\ttcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
      "%10, %11, %12, %13, %14, %15}, [%16];\n\ttcgen05.wait::ld.sync.aligned;\n\t}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    k_moe_tc(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mS0,
             const __grid_constant__ CUtensorMap mA1, const __grid_constant__ CUtensorMap mS1,
             const __grid_constant__ CUtensorMap mB, const __grid_constant__ CUtensorMap mSB,
             const TcArgs a) {
  constexpr int NM = MODE == 0 ? 2 : 1;  // weight matrices per unit (w1 and w3, or w2)
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[kStages], sfready[kStages], empty[kStages];
  __shared__ __align__(8) uint64_t accfull[2], accempty[2], drained;
  __shared__ uint32_t tbase;
  __shared__ int abort_flag;
  __shared__ int flag_ok;
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) &
                                           ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sfready[s], 4);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], 4);
    }
    mbar_init(&drained, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  pdl_wait();
  const long long U = (long long)a.ntile_base[a.meta[0]] * a.RT * a.KC;
  const long long u0 = U * blockIdx.x / gridDim.x, u1 = U * (blockIdx.x + 1) / gridDim.x;
  const bool busy = u1 > u0;
  if (warp == kMmaWarp && busy) {
    tc::tmem_alloc(&tbase, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  pdl_launch();
  if (!busy) return;
  const uint32_t t0 = tbase;
  volatile int* abort_v = &abort_flag;

  if (warp == kProdWarp) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tc::tma_prefetch_map(&mA0);
      tc::tma_prefetch_map(&mS0);
      tc::tma_prefetch_map(&mB);
      tc::tma_prefetch_map(&mSB);
      Cursor c;
      cursor_at(c, u0, a);
      int it = 0;
      for (long long u = u0; u < u1 && !*abort_v; ++u, cursor_next(c, a)) {
        const TileInfo ti = tile_info(c, a);
        const int nbox = ti.N / 16;
        const int arow = ti.expert * a.R + c.rt * kRowsTile;
        for (int m = 0; m < NM; ++m, ++it) {
          const int s = it % kStages;
          if (it >= kStages && !mbar_wait(&empty[s], ((it / kStages) - 1) & 1, a.status)) {
            *abort_v = 1;
            break;
          }
          uint8_t* st = sm + (size_t)s * kStageBytes;
          const CUtensorMap* mA = m == 0 ? &mA0 : &mA1;
          const CUtensorMap* mS = m == 0 ? &mS0 : &mS1;
          mbar_arrive_expect_tx(&full[s], kABytes + kSABytes + (uint32_t)nbox * (2 * 2048 + 256));
          tc::tma_load_2d(st, mA, c.kc * 256, arow, &full[s]);
          tc::tma_load_2d(st + 16384, mA, c.kc * 256 + 128, arow, &full[s]);
          tc::tma_load_2d(st + kOffSA, mS, c.kc * 16, arow, &full[s]);
          for (int b = 0; b < nbox; ++b) {
            const int brow = ti.pos0 * kTerms + 16 * b;
            tc::tma_load_2d(st + kOffB + b * 2048, &mB, c.kc * 256, brow, &full[s]);
            tc::tma_load_2d(st + kOffB + 8192 + b * 2048, &mB, c.kc * 256 + 128, brow, &full[s]);
            tc::tma_load_2d(st + kOffSB + b * 256, &mSB, c.kc * 16, brow, &full[s]);
          }
        }
      }
      if (*abort_v) {
        // copies still in flight land before the CTA leaves: wait for each stage's last fill
        for (int d = 1; d <= kStages && d <= it; ++d) {
          const int i = it - d;
          mbar_wait(&full[i % kStages], (i / kStages) & 1, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp >= kSfWarp0 && warp < kSfWarp0 + 4) {
    // ---------------------------------------------------------------- scales -> TMEM
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    Cursor c;
    cursor_at(c, u0, a);
    int it = 0;
    bool stop = false;
    for (long long u = u0; u < u1 && !stop; ++u, cursor_next(c, a)) {
      const int N = tile_info(c, a).N;
      for (int m = 0; m < NM; ++m, ++it) {
        const int s = it % kStages;
        const bool ok = !*abort_v && mbar_wait(&full[s], (it / kStages) & 1, lane == 0 ? a.status : nullptr);
        if (!__all_sync(0xffffffffu, ok)) {
          *abort_v = 1;
          stop = true;
          break;
        }
        const uint8_t* st = sm + (size_t)s * kStageBytes;
        const uint32_t ring = t0 + lane_off + kSfBase + (uint32_t)s * kSfStageCols;
        const uint4 sa = *reinterpret_cast<const uint4*>(st + kOffSA + 16 * (32 * q + lane));
        const uint32_t wa[4] = {clear_ff_bytes(sa.x), clear_ff_bytes(sa.y), clear_ff_bytes(sa.z),
                                clear_ff_bytes(sa.w)};
#pragma unroll
        for (int j = 0; j < kMmas; ++j)
          tc::tmem_st_x1(ring + 4 * j + q, (wa[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
        const uint4 sb0 = *reinterpret_cast<const uint4*>(st + kOffSB + 16 * lane);
        const uint32_t wb0[4] = {sb0.x, sb0.y, sb0.z, sb0.w};
#pragma unroll
        for (int j = 0; j < kMmas; ++j)
          tc::tmem_st_x1(ring + 32 + 4 * j, (wb0[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
        if (N > 32) {
          const uint4 sb1 = *reinterpret_cast<const uint4*>(st + kOffSB + 16 * (32 + lane));
          const uint32_t wb1[4] = {sb1.x, sb1.y, sb1.z, sb1.w};
#pragma unroll
          for (int j = 0; j < kMmas; ++j)
            tc::tmem_st_x1(ring + 33 + 4 * j, (wb1[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfready[s]);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      Cursor c;
      cursor_at(c, u0, a);
      int it = 0, tcount = 0;
      for (long long u = u0; u < u1 && !*abort_v; ++u, cursor_next(c, a)) {
        const bool first = (u == u0) || c.kc == 0;
        const bool last = (u == u1 - 1) || c.kc == a.KC - 1;
        const int b = tcount & 1;
        if (first && tcount >= 2 && !mbar_wait(&accempty[b], ((tcount >> 1) - 1) & 1, a.status)) {
          *abort_v = 1;
          break;
        }
        const uint32_t idesc = tc::idesc_mxf4(kRowsTile, tile_info(c, a).N, 0, 0);
        bool ok = true;
        for (int m = 0; m < NM; ++m, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(&full[s], ph, a.status) || !mbar_wait(&sfready[s], ph, a.status)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t st = tc::smem_addr(sm + (size_t)s * kStageBytes);
          const uint32_t d = t0 + (uint32_t)b * kAccCols + 64u * m;
          const uint32_t sfr = t0 + kSfBase + (uint32_t)s * kSfStageCols;
#pragma unroll
          for (int j = 0; j < kMmas; ++j) {
            const uint32_t koff = (uint32_t)(j >> 2) * 16384u + (uint32_t)(j & 3) * 32u;
            const uint32_t kboff = (uint32_t)(j >> 2) * 8192u + (uint32_t)(j & 3) * 32u;
            const uint64_t ad = tc::smem_desc(st + koff, 16, 1024, tc::kLayout128B);
            const uint64_t bd = tc::smem_desc(st + kOffB + kboff, 16, 1024, tc::kLayout128B);
            tc::mma_mxf4(d, ad, bd, idesc, sfr + 4 * j, sfr + 32 + 4 * j,
                         (first && j == 0) ? 0u : 1u);
          }
          tc::mma_commit(&empty[s]);
        }
        if (!ok) {
          *abort_v = 1;
          break;
        }
        if (last) {
          tc::mma_commit(&accfull[b]);
          ++tcount;
        }
      }
      tc::mma_commit(&drained);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue (warps 0-3)
    const int q = warp;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const int row = 32 * q + lane;  // row within the tile
    int tcount = 0;
    long long u = u0;
    while (u < u1) {
      Cursor c;
      cursor_at(c, u, a);
      const TileInfo ti = tile_info(c, a);
      const long long tu0 = (long long)c.tile * a.KC, tu1 = tu0 + a.KC;
      const bool head = tu0 >= u0;
      const int b = tcount & 1;
      const int bad = (*abort_v || !mbar_wait(&accfull[b], (tcount >> 1) & 1, a.status)) ? 1 : 0;
      if (bar_or(kEpiBar, 128, bad)) {
        *abort_v = 1;
        break;
      }
      tc::fence_after_sync();
      float acc[NM][kNMax];
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int c0 = 0; c0 < kNMax; c0 += 16) {
          float v[16];
          if (c0 < ti.N) {
            tmem_load16(t0 + lane_off + (uint32_t)b * kAccCols + 64u * m + c0, v);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[m][c0 + i] = v[i];
        }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[b]);
      ++tcount;

      float* my_part = a.part + (size_t)blockIdx.x * 2 * a.npart * kRowsTile;
      if (!head) {
        // leave the partial sums for the tile's first CTA
#pragma unroll
        for (int m = 0; m < NM; ++m)
#pragma unroll
          for (int cc = 0; cc < kNMax; ++cc)
            if (cc < ti.N) my_part[((size_t)m * a.npart + cc) * kRowsTile + row] = acc[m][cc];
        __threadfence();
        named_bar(kEpiBar, 128);
        if (threadIdx.x == 0) st_release(a.flags + blockIdx.x, 1);
      } else {
        bool failed = false;
        if (tu1 > u1) {
          for (int oc = blockIdx.x + 1; oc < (int)gridDim.x; ++oc) {
            const long long ou0 = U * oc / gridDim.x;
            if (ou0 >= tu1) break;
            if (U * (oc + 1) / gridDim.x == ou0) continue;  // an idle CTA leaves nothing
            if (threadIdx.x == 0) {
              int ok = 0;
              for (uint32_t i = 0; i < kWaitPolls && !ok; ++i) ok = ld_acquire(a.flags + oc) == 1;
              if (!ok && a.status) atomicAdd(a.status + kStatTimeout, 1);
              flag_ok = ok;
            }
            named_bar(kEpiBar, 128);
            const bool got = flag_ok != 0;
            named_bar(kEpiBar, 128);  // flag_ok is rewritten by the next wait
            if (!got) {
              *abort_v = 1;
              failed = true;
              break;
            }
            const float* op = a.part + (size_t)oc * 2 * a.npart * kRowsTile;
#pragma unroll
            for (int m = 0; m < NM; ++m)
#pragma unroll
              for (int cc = 0; cc < kNMax; ++cc)
                if (cc < ti.N) acc[m][cc] += __ldcg(op + ((size_t)m * a.npart + cc) * kRowsTile + row);
          }
        }
        if (failed) break;
        const int r_exp = c.rt * kRowsTile + row;  // row within the expert
        if (MODE == 0) {
          // SwiGLU (or SiTU-GLU) per token, then its kTerms MXFP4 terms for the second GEMM;
          // this warp's 32 rows are one group of 32 along the second GEMM's reduction
          const bool in_range = c.rt * kRowsTile + 32 * q < a.R;
#pragma unroll
          for (int j = 0; j < kTokTile; ++j) {
            if (j >= ti.ntok) break;
            float g = 0.f, uu = 0.f;
#pragma unroll
            for (int t = 0; t < kTerms; ++t) {
              g += acc[0][j * kTerms + t];
              uu += acc[NM - 1][j * kTerms + t];
            }
            const float act = activation(g, uu, a.act_kind, a.b1, a.b2);
            uint32_t words[kTerms], sf[kTerms];
            mx_split_group(act, words, sf);
            if (in_range) {
              const size_t p = (size_t)(ti.pos0 + j);
              const int grp = (c.rt * kRowsTile + 32 * q) >> 5;
#pragma unroll
              for (int t = 0; t < kTerms; ++t) {
                const size_t r2 = p * kTerms + t;
                if ((lane & 7) == 0)
                  *reinterpret_cast<uint32_t*>(a.act_q + r2 * (size_t)(a.I >> 1) + grp * 16 +
                                               4 * (lane >> 3)) = words[t];
                if (lane == 0) a.act_sf[r2 * (size_t)(a.I >> 5) + grp] = (uint8_t)sf[t];
              }
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < kTokTile; ++j) {
            if (j >= ti.ntok) break;
            float o = 0.f;
#pragma unroll
            for (int t = 0; t < kTerms; ++t) o += acc[0][j * kTerms + t];
            const int asg = a.perm[ti.pos0 + j];
            if (r_exp < a.R) a.ybuf[(size_t)asg * a.R + r_exp] = a.gate[asg] * o;
          }
        }
      }
      u = min(u1, tu1);
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncthreads();
  if (warp == kMmaWarp) {
    if (lane == 0) mbar_wait(&drained, 0, a.status);
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(t0, kTmemCols);
  }
}

// x (bf16, one row per token) -> kTerms MXFP4 terms per (token, expert) position, in the
// bucket order: rows p * kTerms + t of xq [P*kTerms][L/2] and xsf [P*kTerms][L/32].  Grid
// (T, L/512), 16 warps: warp w handles group 16 * blockIdx.y + w of token blockIdx.x.
__global__ void __launch_bounds__(512) k_split_x(const uint16_t* __restrict__ x, int L, int k,
                                                 int E, const int32_t* __restrict__ idx,
                                                 const int32_t* __restrict__ inv,
                                                 uint8_t* __restrict__ xq,
                                                 uint8_t* __restrict__ xsf) {
  pdl_wait();
  pdl_launch();
  const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = blockIdx.y * 16 + warp;
  const float v = __uint_as_float((uint32_t)x[(size_t)t * L + 32 * grp + lane] << 16);
  uint32_t words[kTerms], sf[kTerms];
  mx_split_group(v, words, sf);
  for (int j = 0; j < k; ++j) {
    const int asg = t * k + j;
    const int e = idx[asg];
    if (e < 0 || e >= E) continue;
    const size_t p = (size_t)inv[asg];
#pragma unroll
    for (int tt = 0; tt < kTerms; ++tt) {
      const size_t r = p * kTerms + tt;
      if ((lane & 7) == 0)
        *reinterpret_cast<uint32_t*>(xq + r * (size_t)(L >> 1) + grp * 16 + 4 * (lane >> 3)) = words[tt];
      if (lane == 0) xsf[r * (size_t)(L >> 5) + grp] = (uint8_t)sf[tt];
    }
  }
}

template <int MODE>
cudaError_t launch_tc(const CUtensorMap (&maps)[6], const TcArgs& a, int grid, cudaStream_t s,
                      bool pdl) {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_moe_tc<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  return launch_kernel(k_moe_tc<MODE>, dim3(grid), dim3(kThreads), kSmemBytes, s, pdl, maps[0],
                       maps[1], maps[2], maps[3], maps[4], maps[5], a);
}

}  // namespace

bool tc_path_supported(int L, int I) { return L % kKStage == 0 && I % kKStage == 0; }

int tc_grid() { return sm_count() < kTcMaxGrid ? sm_count() : kTcMaxGrid; }

size_t tc_part_floats(int T) {
  return (size_t)kTcMaxGrid * 2 * tc_npart(T) * kRowsTile;
}

int tc_npart(int T) {
  const int tok = T < kTokTile ? T : kTokTile;
  return ((tok * kTerms + 15) / 16) * 16;
}

cudaError_t launch_split_x(const uint16_t* x, int T, int L, int k, int E, const int32_t* idx,
                           const int32_t* inv, uint8_t* xq, uint8_t* xsf, cudaStream_t s,
                           bool pdl) {
  return launch_kernel(k_split_x, dim3(T, L / kKStage), dim3(512), 0, s, pdl, x, L, k, E, idx,
                       inv, xq, xsf);
}

cudaError_t launch_tc_gemm1(const ExpertPtrs& w, int L, int I, int E, int T, int k,
                            const uint8_t* xq, const uint8_t* xsf, const BucketOut& b,
                            uint8_t* act_q, uint8_t* act_sf, int act_kind, float b1, float b2,
                            float* part, int32_t* flags, int32_t* status, cudaStream_t s,
                            bool pdl) {
  const uint64_t P4 = (uint64_t)T * k * kTerms;
  CUtensorMap maps[6];
  if (!make_map_2d(&maps[0], w.w1p, L / 2, (uint64_t)E * I, 128, 128, true) ||
      !make_map_2d(&maps[1], w.w1s, L / 32, (uint64_t)E * I, 16, 128, false) ||
      !make_map_2d(&maps[2], w.w3p, L / 2, (uint64_t)E * I, 128, 128, true) ||
      !make_map_2d(&maps[3], w.w3s, L / 32, (uint64_t)E * I, 16, 128, false) ||
      !make_map_2d(&maps[4], xq, L / 2, P4, 128, 16, true) ||
      !make_map_2d(&maps[5], xsf, L / 32, P4, 16, 16, false))
    return cudaErrorInvalidValue;
  TcArgs a{};
  a.K = L; a.R = I; a.KC = L / kKStage; a.RT = (I + kRowsTile - 1) / kRowsTile; a.k = k;
  a.active = b.active; a.seg_off = b.seg_off; a.seg_cnt = b.seg_cnt; a.meta = b.meta;
  a.perm = b.perm; a.ntile_base = b.ntile_base;
  a.act_q = act_q; a.act_sf = act_sf; a.I = I; a.act_kind = act_kind; a.b1 = b1; a.b2 = b2;
  a.part = part; a.npart = tc_npart(T); a.flags = flags; a.status = status;
  return launch_tc<0>(maps, a, tc_grid(), s, pdl);
}

cudaError_t launch_tc_gemm2(const ExpertPtrs& w, int L, int I, int E, int T, int k,
                            const uint8_t* act_q, const uint8_t* act_sf, const float* gate,
                            const BucketOut& b, float* ybuf, float* part, int32_t* flags,
                            int32_t* status, cudaStream_t s, bool pdl) {
  const uint64_t P4 = (uint64_t)T * k * kTerms;
  CUtensorMap maps[6];
  if (!make_map_2d(&maps[0], w.w2p, I / 2, (uint64_t)E * L, 128, 128, true) ||
      !make_map_2d(&maps[1], w.w2s, I / 32, (uint64_t)E * L, 16, 128, false) ||
      !make_map_2d(&maps[4], act_q, I / 2, P4, 128, 16, true) ||
      !make_map_2d(&maps[5], act_sf, I / 32, P4, 16, 16, false))
    return cudaErrorInvalidValue;
  maps[2] = maps[0];
  maps[3] = maps[1];
  TcArgs a{};
  a.K = I; a.R = L; a.KC = I / kKStage; a.RT = (L + kRowsTile - 1) / kRowsTile; a.k = k;
  a.active = b.active; a.seg_off = b.seg_off; a.seg_cnt = b.seg_cnt; a.meta = b.meta;
  a.perm = b.perm; a.ntile_base = b.ntile_base;
  a.gate = gate; a.ybuf = ybuf;
  a.part = part; a.npart = tc_npart(T); a.flags = flags; a.status = status;
  return launch_tc<1>(maps, a, tc_grid(), s, pdl);
}

}  // namespace k3
