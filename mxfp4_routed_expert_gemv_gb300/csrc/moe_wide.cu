// moe_wide.cu -- the routed experts of a large batch on the block-scaled tensor cores.
//
// README "kimi-k3-in-c", Part II sections 4 and 9: every selected expert multiplies its
// packed E2M1 weights (one E8M0 scale per 32) straight from the checkpoint bytes:
//   g = W1[e] x,  u = W3[e] x,  act = silu(g) u (or SiTU-GLU),  o = W2[e] act,
//   ybuf[assignment] = gate * o   (the slots are summed by k_combine, in slot order).
//
// When many tokens share an expert (a prefill: about 700 per active expert, some experts
// chosen by every token) the work is a grouped GEMM, and the shape of a tile decides how
// often each byte is brought into shared memory.  Here a tile is 128 positions of one expert
// (its tokens, in bucket order) as the MMA's M and 256 weight rows as its N, over the whole
// reduction:
//   * the activation's kTerms MXFP4 terms (mxq.cuh) are folded into the reduction: per
//     K-step of 64 the tile issues one MMA per term, same weights, same accumulator, so a
//     token costs one TMEM column whatever the number of terms, and the weight tile in
//     shared memory feeds kTerms MMAs;
//   * GEMM1's 256 rows are 128 rows of w1 and the same 128 rows of w3, so g and u of a row
//     meet in one thread of the epilogue (SwiGLU with no exchange), and the thread holds
//     whole groups of 32 act values of its position: it writes their MXFP4 terms alone.
// Tiles run expert by expert, and within an expert row block by row block with the token
// tiles fastest, CTA c taking tiles c, c + G, ...: the CTAs working at one time share a few
// weight blocks and one expert's activation terms, which stay in L2.
//
// Scales travel by TMA as well.  The activation terms' E8M0 bytes are stored stage-major on
// this path (k_split_x_wide and GEMM1's epilogue write them so): for each 128-wide stage of
// the reduction, one 16-byte row per position holding its 4 groups' kTerms scale bytes
// (group-major: one 4-byte word per group), so a stage's scales are one 2 KB box.  The weights' scales stay in the checkpoint layout and
// come as 16-byte boxes of 512-wide chunks (four stages) into a two-slot ring.
//
// Pipeline (448 threads, one CTA per SM): warp 8 issues the TMA copies of a stage (K = 128:
// the kTerms term tiles of the positions, 64-byte swizzle, their scales, and the 256 weight
// rows; the weight scales once per four stages), warps 10-13 move the scales from shared
// memory into TMEM (each warp its lane quarter), warp 9 allocates TMEM and issues the MMAs
// (tcgen05.mma kind::mxf4, M = 128, N = 256, fp32 accumulators in TMEM), warps 0-7 run the
// epilogue.  GEMM1's epilogue keeps act (fp32) in registers and frees the accumulator
// before it splits act into terms, so the split overlaps the next tile's MMAs; four stages
// in both GEMMs.  Every wait is bounded; one that runs out counts a timeout in the status
// block and the CTA stops.
#include "launch.h"
#include "mxq.cuh"
#include "tc.cuh"
#include "tmap.h"

namespace k3 {
namespace {

constexpr int kWM = kTcWideTok;                          // MMA M (rows of the A tile)
constexpr int kWN = 256;                                 // weight rows per tile (MMA N)
constexpr int kWsK = 512;                                // reduction per weight-scale box
constexpr uint32_t kWsBytes = kWN * 16;                  // one weight-scale ring slot: 4 KB
constexpr int kThreadsW = 448;
constexpr int kEpiWarpsW = 8, kProdWarpW = 8, kMmaWarpW = 9, kSfWarpW0 = 10;
constexpr uint32_t kAccColsW = kWN;                      // one fp32 accumulator, N columns
constexpr uint32_t kTmemColsW = 512;

// The two tile shapes.  Folded (TR false): 128 positions are the MMA's rows and each
// activation term is its own MMA into the same accumulator (kTerms A tiles per stage; stages
// of K = 128, 64-byte swizzle).  Rows (TR true): the 128 MMA rows are 32 positions x kTerms
// terms (the per-position term rows as stored), one MMA per K-step, and the epilogue adds a
// position's term rows (stages of K = 256, 128-byte swizzle: a stage of this shape has four
// times fewer MMAs per byte, so it is made twice as long, with rows of 128 bytes).
// TMEM scale ring, per stage: A scales of term t, K-step j at 4 (t kKSteps + j): 4 columns,
// row m reads lane m of column + m/32; B (weight) scales of K-step j at kSfB + 8 j: 8
// columns, row n reads column + n/32 in every lane quarter.
template <bool TR>
struct WMode {
  static constexpr int kPos = TR ? kTcRowTok : kTcWideTok;        // positions per tile
  static constexpr int kTermMmas = TR ? 1 : kTerms;               // MMAs per K-step
  static constexpr int kKS = TR ? 256 : 128;                      // reduction per stage
  static constexpr int kKSteps = kKS / 64;
  static constexpr uint32_t kRowB = kKS / 2;                      // bytes of a row per stage
  static constexpr uint32_t kSbo = 8 * kRowB;                     // 8-row group stride
  static constexpr uint32_t kLayout = TR ? tc::kLayout128B : tc::kLayout64B;
  static constexpr uint32_t kATile = kWM * kRowB;                 // one 128-row A tile
  static constexpr uint32_t kABytes = kATile * kTermMmas;         // A tiles of a stage
  static constexpr uint32_t kBBytes = kWN * kRowB;                // the weight tile
  static constexpr int kAsBoxes = kKS / 128;                      // 16-byte scale rows per position
  static constexpr uint32_t kAsBytes = kPos * 16 * kAsBoxes;      // the positions' scales
  static constexpr uint32_t kStage =
      ((kABytes + kBBytes + kAsBytes + 1023) / 1024) * 1024;      // 49 KB or 50 KB
  static constexpr int kStagesPerWs = kWsK / kKS;                 // stages per weight-scale box
  static constexpr uint32_t kSfB = 4 * kKSteps * kTermMmas;
  static constexpr uint32_t kSfCols = kSfB + 8 * kKSteps;
  static_assert(kPos * (TR ? kTerms : 1) == kWM, "A tile rows");
};
constexpr int kEpiBarW = 1;      // named barrier of the 256 epilogue threads

template <int PH, bool TR>
struct WLay {
  using M = WMode<TR>;
  static constexpr int kStages = 4;
  static constexpr size_t kSmemBytes = (size_t)kStages * M::kStage + 2 * kWsBytes + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared-memory budget");
  static_assert(kAccColsW + kStages * M::kSfCols <= kTmemColsW, "TMEM budget");
};

struct WArgs {
  int K;            // reduction width: L (GEMM1) or I (GEMM2)
  int R;            // weight rows per expert: I (GEMM1, w1 and w3) or L (GEMM2)
  int RB;           // row blocks per expert: R / 128 (GEMM1) or R / 256 (GEMM2)
  int P;            // position rows of the activation terms (T * k)
  const int32_t *meta, *perm;
  const int4* desc;         // [tiles] expert, first position, positions, rb | groups << 8
  uint8_t *act_q, *act_sf;  // GEMM1 output: act terms [P * kTerms][I / 2], scales stage-major
  int I;
  int act_kind;
  float b1, b2;
  const float* gate;        // GEMM2: [T * k]
  float* ybuf;              // GEMM2 output [T * k][L]
  int L;
  int32_t* status;
};

struct WMaps {
  CUtensorMap a;      // activation terms: folded, 3-D [P][kTerms][K / 2], boxes of 128
                      // positions of one term; rows, 2-D [P * kTerms][K / 2], boxes of 128 rows
  CUtensorMap as;     // their scales, stage-major: [K / 128 * P][16 B], boxes of kPos rows
  CUtensorMap w0, w1; // weights: w1 and w3 (boxes of 128 rows) or w2 (twice, 256 rows)
  CUtensorMap s0, s1; // weight scales [E * R][K / 32 B], boxes of 16 B (512-wide chunks)
};

struct WTile {
  int expert, pos0, ntok, rb, groups;
};

__device__ __forceinline__ WTile unpack_tile(int4 d) {
  WTile w;
  w.expert = d.x;
  w.pos0 = d.y;
  w.ntok = d.z;
  w.rb = d.w & 255;
  w.groups = d.w >> 8;
  return w;
}

__device__ __forceinline__ int bar_or_w(uint32_t id, uint32_t n, int v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v), "r"(id), "r"(n)
      : "memory");
  return (int)r;
}

// Byte offset of the 4-byte word of group `grp` at position `pos` (byte t: term t's E8M0
// scale) in the stage-major layout of activation-term scales: [K / 128][P][4 groups][kTerms].
__host__ __device__ __forceinline__ size_t wide_sf_offset(int grp, int pos, int P) {
  return (((size_t)(grp >> 2) * P + pos) * 4 + (grp & 3)) * kTerms;
}
static_assert(kTerms == 4, "one 32-bit word of scales per group");

// Rows mode: a position's kTerms term rows are 4 consecutive lanes (a quad, t4 = lane % 4).
// On entry each lane holds 32 columns of its term row; on exit v[0 .. 7] holds the sums over
// the four terms of columns 8 t4 .. 8 t4 + 7, added as (t0 + t2) + (t1 + t3): a reduce-scatter
// in two exchanges (16 values with the lane 2 apart, then 8 with the neighbour).
__device__ __forceinline__ void quad_reduce_scatter32(float (&v)[32], int t4) {
  const bool h2 = (t4 & 2) != 0, h1 = (t4 & 1) != 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float send = h2 ? v[i] : v[i + 16];
    const float keep = h2 ? v[i + 16] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = h1 ? v[i] : v[i + 8];
    const float keep = h1 ? v[i + 8] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
  }
}

// The MXFP4 terms of one group of 32 act values (consumed) into the per-position rows and
// the stage-major scale word.
__device__ __forceinline__ void store_act_group(const WArgs& f, float (&r)[32], size_t pos, int grp) {
  uint32_t words[kTerms][4], sfb[kTerms];
  mx_split_lane32(r, words, sfb);
#pragma unroll
  for (int tt = 0; tt < kTerms; ++tt) {
    const size_t r2 = pos * kTerms + tt;
    *reinterpret_cast<uint4*>(f.act_q + r2 * (size_t)(f.I >> 1) + grp * 16) =
        make_uint4(words[tt][0], words[tt][1], words[tt][2], words[tt][3]);
  }
  *reinterpret_cast<uint32_t*>(f.act_sf + wide_sf_offset(grp, (int)pos, f.P)) =
      sfb[0] | (sfb[1] << 8) | (sfb[2] << 16) | (sfb[3] << 24);
}

// bytes 0xFF -> 0x00 (an E8M0 "no value" becomes the smallest scale: the group adds nothing
// measurable, as the README decoder's zero group)
__device__ __forceinline__ uint32_t clear_ff(uint32_t w) {
  const uint32_t t = ~w;
  const uint32_t y = ((t & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | t;
  const uint32_t ff = (~y & 0x80808080u) >> 7;
  return w & ~(ff * 0xFFu);
}

template <int PH, bool TR>
__global__ void __launch_bounds__(kThreadsW, 1) k_moe_wide(const __grid_constant__ WMaps mp,
                                                           const WArgs f) {
  using Y = WLay<PH, TR>;
  using M = WMode<TR>;
  constexpr int S = Y::kStages;
  constexpr uint32_t kStageW = M::kStage;
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[S], sfready[S], empty[S];
  __shared__ __align__(8) uint64_t accfull, accempty, drained, wsfull[2], wsempty[2];
  __shared__ uint32_t tbase;
  __shared__ int abort_flag;
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) &
                                           ~uintptr_t(1023));
  uint8_t* wsring = sm + (size_t)S * kStageW;  // two weight-scale slots
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sfready[s], 4);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&accfull, 1);
    mbar_init(&accempty, 1);
    mbar_init(&drained, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&wsfull[i], 1);
      mbar_init(&wsempty[i], 4);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == kMmaWarpW) {
    tc::tmem_alloc(&tbase, kTmemColsW);
    tc::tmem_relinquish();
  }
  if (warp == kProdWarpW && lane == 0) {
    tc::tma_prefetch_map(&mp.a);
    tc::tma_prefetch_map(&mp.as);
    tc::tma_prefetch_map(&mp.w0);
    tc::tma_prefetch_map(&mp.w1);
    tc::tma_prefetch_map(&mp.s0);
    tc::tma_prefetch_map(&mp.s1);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // Only the producer's activation-term copies read the preceding launch's output (the tile
  // table comes from the preparation, which had completed before that launch passed its own
  // wait), and nothing this kernel writes is read by it: only the producer waits.
  pdl_launch();
  const uint32_t t0 = tbase;
  volatile int* abort_v = &abort_flag;
  const int ntiles = f.meta[TR ? 4 : 3] * f.RB;
  const int KC = f.K / M::kKS;

  if (warp == kProdWarpW) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // a stage reads 64 or 128 bytes of each weight row and the tensor maps fill L2 in
      // 256-byte pieces, so a row's next bytes are read from L2 by the following stages:
      // weights keep normal priority (evict-first would drop them before that)
      const uint64_t pol = tc::make_policy_evict_normal();
      int it = 0, ch = 0;  // stages and weight-scale chunks issued
      bool stop = false;
      int4 next = cta < ntiles ? __ldg(f.desc + cta) : make_int4(0, 0, 0, 0);
      if (cta < ntiles) {
        // while the preceding launch finishes, the first stages' weights into L2 (they are
        // constants, and the tile table was complete before that launch started)
        const WTile w0 = unpack_tile(next);
        const int wrow0 = w0.expert * f.R + w0.rb * (PH == 0 ? 128 : 256);
        for (int kc = 0; kc < S && kc < KC; ++kc) {
          tc::tma_prefetch_l2_2d(&mp.w0, kc * (int)M::kRowB, wrow0);
          if (PH == 0) tc::tma_prefetch_l2_2d(&mp.w1, kc * (int)M::kRowB, wrow0);
        }
      }
      pdl_wait();
      for (int t = cta; t < ntiles && !stop; t += G) {
        const WTile wt = unpack_tile(next);
        if (t + G < ntiles) next = __ldg(f.desc + t + G);  // in flight during this tile
        const int wrow = wt.expert * f.R + wt.rb * (PH == 0 ? 128 : 256);
        // rows: only the boxes of 8 positions (32 term rows) that hold the tile's tokens;
        // the other A rows keep older bytes, which reach only D rows the epilogue skips
        const int nbox = TR ? (wt.ntok + 7) / 8 : 1;
        for (int kc = 0; kc < KC; ++kc, ++it) {
          const int s = it % S;
          if (*abort_v ||
              (it >= S && !mbar_wait_ab(&empty[s], ((it / S) - 1) & 1, f.status, abort_v))) {
            *abort_v = 1;
            stop = true;
            break;
          }
          if (kc % M::kStagesPerWs == 0) {
            // the weight scales of the next kWsK reduction elements into slot ch % 2, once the
            // scale warps are done with the chunk that last used it
            const int slot = ch & 1;
            if (ch >= 2 && !mbar_wait_ab(&wsempty[slot], ((ch >> 1) - 1) & 1, f.status, abort_v)) {
              *abort_v = 1;
              stop = true;
              break;
            }
            uint8_t* ws = wsring + slot * kWsBytes;
            mbar_arrive_expect_tx(&wsfull[slot], kWsBytes);
            if (PH == 0) {
              tc::tma_load_2d(ws, &mp.s0, (kc / M::kStagesPerWs) * 16, wrow, &wsfull[slot]);
              tc::tma_load_2d(ws + kWsBytes / 2, &mp.s1, (kc / M::kStagesPerWs) * 16, wrow,
                              &wsfull[slot]);
            } else {
              tc::tma_load_2d(ws, &mp.s0, (kc / M::kStagesPerWs) * 16, wrow, &wsfull[slot]);
            }
            ++ch;
          }
          // one barrier for the whole stage: activation terms, their scales and the weights
          // (separate barriers for the activation and the weight copies measured slower)
          uint8_t* st = sm + (size_t)s * kStageW;
          mbar_arrive_expect_tx(&full[s], (TR ? nbox * (M::kATile / 4) : M::kABytes) + M::kBBytes +
                                              M::kAsBytes);
          const int x = kc * (int)M::kRowB;
          if (TR) {
            for (int b = 0; b < nbox; ++b)
              tc::tma_load_2d(st + b * (M::kATile / 4), &mp.a, x, (wt.pos0 + 8 * b) * kTerms, &full[s]);
          } else {
#pragma unroll
            for (int tt = 0; tt < kTerms; ++tt)
              tc::tma_load_3d(st + tt * M::kATile, &mp.a, x, tt, wt.pos0, &full[s]);
          }
#pragma unroll
          for (int r = 0; r < M::kAsBoxes; ++r)
            tc::tma_load_2d(st + M::kABytes + M::kBBytes + r * (M::kPos * 16), &mp.as, 0,
                            (kc * M::kAsBoxes + r) * f.P + wt.pos0, &full[s]);
          uint8_t* sb = st + M::kABytes;
          if (PH == 0) {
            tc::tma_load_2d_hint(sb, &mp.w0, x, wrow, &full[s], pol);
            tc::tma_load_2d_hint(sb + M::kBBytes / 2, &mp.w1, x, wrow, &full[s], pol);
          } else {
            tc::tma_load_2d_hint(sb, &mp.w0, x, wrow, &full[s], pol);
          }
        }
      }
      if (*abort_v) {
        // copies still in flight land before the CTA leaves
        for (int d = 1; d <= S && d <= it; ++d) {
          const int i = it - d;
          mbar_wait(&full[i % S], (i / S) & 1, nullptr);
        }
        for (int d = 1; d <= 2 && d <= ch; ++d) {
          const int c = ch - d;
          mbar_wait(&wsfull[c & 1], (c >> 1) & 1, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp >= kSfWarpW0) {
    // --------------------------------------------------------- scales -> TMEM (4 warps)
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    int it = 0, ch = -1;
    bool stop = false;
    for (int t = cta; t < ntiles && !stop; t += G) {
      for (int kc = 0; kc < KC; ++kc, ++it) {
        const int s = it % S;
        const uint32_t par = (it / S) & 1;
        // the stage's data has landed: the MMAs that last read this TMEM scale slot are done
        bool ok = !*abort_v &&
                  mbar_wait_ab(&full[s], par, lane == 0 ? f.status : nullptr, abort_v);
        if (kc % M::kStagesPerWs == 0) {
          ++ch;
          ok = ok && mbar_wait_ab(&wsfull[ch & 1], (ch >> 1) & 1, lane == 0 ? f.status : nullptr,
                                  abort_v);
        }
        if (!__all_sync(0xffffffffu, ok)) {
          *abort_v = 1;
          stop = true;
          break;
        }
        const uint8_t* st = sm + (size_t)s * kStageW;
        // this lane's A row: a position (folded), or a position's term row (rows)
        const int arow = 32 * q + lane;
        const uint8_t* ws = wsring + (ch & 1) * kWsBytes + (kc % M::kStagesPerWs) * (M::kKS / 32);
        const uint32_t ring = t0 + lane_off + kAccColsW + (uint32_t)s * M::kSfCols;
#pragma unroll
        for (int r = 0; r < M::kAsBoxes; ++r) {  // each 16-byte row: 4 groups = 2 K-steps
          const uint4 as = *reinterpret_cast<const uint4*>(
              st + M::kABytes + M::kBBytes + r * (M::kPos * 16) + 16 * (TR ? (arow >> 2) : arow));
          // word g of the row holds group g's term bytes; term t's word gathers byte t of each
#pragma unroll
          for (int tt = 0; tt < M::kTermMmas; ++tt) {
            const uint32_t term = TR ? (uint32_t)(arow & 3) : (uint32_t)tt;
            const uint32_t sel = term | ((term + 4) << 4);
            const uint32_t a = clear_ff(
                __byte_perm(__byte_perm(as.x, as.y, sel), __byte_perm(as.z, as.w, sel), 0x5410));
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
              tc::tmem_st_x1(ring + 4 * (tt * M::kKSteps + 2 * r + jj) + q, (a >> (16 * jj)) & 0xFFFFu);
          }
        }
#pragma unroll
        for (int r = 0; r < M::kKSteps / 2; ++r) {  // a weight-scale word: 2 K-steps
          uint32_t wv[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            wv[c] = clear_ff(*reinterpret_cast<const uint32_t*>(ws + 16 * (32 * c + lane) + 4 * r));
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            uint32_t v[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) v[c] = (wv[c] >> (16 * jj)) & 0xFFFFu;
            tc::tmem_st_x8(ring + M::kSfB + 8 * (2 * r + jj), v);
          }
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sfready[s]);
          if (kc % M::kStagesPerWs == M::kStagesPerWs - 1)
            mbar_arrive(&wsempty[ch & 1]);  // done with this chunk's slot
        }
      }
    }
  } else if (warp == kMmaWarpW) {
    // ---------------------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_mxf4(kWM, kWN, 0, 0);
      int it = 0, tl = 0;
      bool stop = false;
      for (int t = cta; t < ntiles && !stop; t += G, ++tl) {
        if (tl >= 1 && !mbar_wait_ab(&accempty, (tl - 1) & 1, f.status, abort_v)) {
          *abort_v = 1;
          break;
        }
        tc::fence_after_sync();
        for (int kc = 0; kc < KC; ++kc, ++it) {
          const int s = it % S;
          const uint32_t par = (it / S) & 1;
          // the scale warps arrive on sfready only after they have seen the stage's copies
          // land (full), so this one wait covers both
          if (*abort_v || !mbar_wait_ab(&sfready[s], par, f.status, abort_v)) {
            *abort_v = 1;
            stop = true;
            break;
          }
          tc::fence_after_sync();
          const uint32_t st = tc::smem_addr(sm + (size_t)s * kStageW);
          const uint32_t sfr = t0 + kAccColsW + (uint32_t)s * M::kSfCols;
#pragma unroll
          for (int j = 0; j < M::kKSteps; ++j) {
            const uint64_t bd = tc::smem_desc(st + M::kABytes + 32 * j, 16, M::kSbo, M::kLayout);
#pragma unroll
            for (int tt = 0; tt < M::kTermMmas; ++tt) {
              const uint64_t ad = tc::smem_desc(st + tt * M::kATile + 32 * j, 16, M::kSbo, M::kLayout);
              tc::mma_mxf4(t0, ad, bd, idesc, sfr + 4 * (tt * M::kKSteps + j), sfr + M::kSfB + 8 * j,
                           (kc == 0 && j == 0 && tt == 0) ? 0u : 1u);
            }
          }
          tc::mma_commit(&empty[s]);
        }
        if (!stop) tc::mma_commit(&accfull);
      }
      tc::mma_commit(&drained);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-7)
    const int q = warp & 3, hf = warp >> 2;
    const int m = 32 * q + lane;                  // position within the tile
    const uint32_t tacc = t0 + ((uint32_t)(32 * q) << 16);
    const int et = threadIdx.x;                   // 0 .. 255
    int tl = 0;
    for (int t = cta; t < ntiles; t += G, ++tl) {
      const WTile wt = unpack_tile(__ldg(f.desc + t));
      const int bad = (*abort_v || !mbar_wait_ab(&accfull, tl & 1, f.status, abort_v)) ? 1 : 0;
      if (bar_or_w(kEpiBarW, 32 * kEpiWarpsW, bad)) {
        *abort_v = 1;
        break;
      }
      tc::fence_after_sync();
      if (TR) {
        // rows mode: lane = (position 8 q + lane / 4, term lane % 4)
        const int t4 = lane & 3;
        const int mpos = 8 * q + (lane >> 2);  // position within the tile
        if (PH == 0) {
          // chunk c = 2 hf + cc: rows 32 c .. 32 c + 31 of w1 (g) and w3 (u); the term rows
          // added (lane t4 then holds rows 32 c + 8 t4 .. + 7), SwiGLU
          float act[2][8], us[2][8];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * hf + cc;
            uint32_t gr[32], ur[32];
            tc::tmem_ld_x32(tacc + 32 * c, gr);
            tc::tmem_ld_x32(tacc + 128 + 32 * c, ur);
            tc::tmem_ld_wait();
            float g[32], u[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              g[i] = __uint_as_float(gr[i]);
              u[i] = __uint_as_float(ur[i]);
            }
            quad_reduce_scatter32(g, t4);
            quad_reduce_scatter32(u, t4);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              act[cc][i] = g[i];
              us[cc][i] = u[i];
            }
          }
          // the accumulator is read: the next tile's MMAs may start while this one finishes
          tc::fence_before_sync();
          named_bar(kEpiBarW, 32 * kEpiWarpsW);
          if (et == 0) mbar_arrive(&accempty);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              act[cc][i] = activation_fast(act[cc][i], us[cc][i], f.act_kind, f.b1, f.b2);
          // the quad splits each chunk's group of 32 act values (every lane takes part in the
          // shuffles; only positions of the tile store)
          const bool mine = mpos < wt.ntok;
          const size_t pos = (size_t)(wt.pos0 + mpos);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int grp = wt.rb * 4 + 2 * hf + cc;
            uint32_t wq[kTerms], sfb[kTerms];
            mx_split_quad8(act[cc], wq, sfb);
            if (mine) {
#pragma unroll
              for (int tt = 0; tt < kTerms; ++tt)
                *reinterpret_cast<uint32_t*>(f.act_q + (pos * kTerms + tt) * (size_t)(f.I >> 1) +
                                             grp * 16 + 4 * t4) = wq[tt];
              if (t4 == 0)
                *reinterpret_cast<uint32_t*>(f.act_sf + wide_sf_offset(grp, (int)pos, f.P)) =
                    sfb[0] | (sfb[1] << 8) | (sfb[2] << 16) | (sfb[3] << 24);
            }
          }
        } else {
          // o for output rows 256 rb + 128 hf .. + 127 of this warp's 8 positions, 32 at a
          // time; after the term sum lane t4 holds 8 of the 32, stored times the gate
          int a = 0;
          float gt = 0.f;
          const bool mine = mpos < wt.ntok;
          if (mine) {
            a = __ldg(f.perm + wt.pos0 + mpos);
            gt = __ldg(f.gate + a);
          }
          float* yrow = f.ybuf + (size_t)a * f.L + (size_t)wt.rb * 256 + 128 * hf + 8 * t4;
          float o[4][8];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t vr[32];
            tc::tmem_ld_x32(tacc + 128 * hf + 32 * c, vr);
            tc::tmem_ld_wait();
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(vr[i]);
            quad_reduce_scatter32(v, t4);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[c][i] = v[i];
          }
          // the accumulator is read: the next tile's MMAs may start during the stores
          tc::fence_before_sync();
          named_bar(kEpiBarW, 32 * kEpiWarpsW);
          if (et == 0) mbar_arrive(&accempty);
          if (mine) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              *reinterpret_cast<float4*>(yrow + 32 * c) =
                  make_float4(gt * o[c][0], gt * o[c][1], gt * o[c][2], gt * o[c][3]);
              *reinterpret_cast<float4*>(yrow + 32 * c + 4) =
                  make_float4(gt * o[c][4], gt * o[c][5], gt * o[c][6], gt * o[c][7]);
            }
          }
        }
      } else if (PH == 0) {
        // g in columns 0..127, u in 128..255 (rows 128 rb .. 128 rb + 127 of w1 / w3); this
        // thread: position m, rows 64 hf .. 64 hf + 63 (two groups of 32), 16 at a time, act
        // kept in registers; the accumulator is released before the groups' MXFP4 split
        // (the activation of the first two pieces is taken while the accumulator is held,
        // the last two are read raw and activated after it is released: the activation's
        // special-function work, not the reads, sets how long the MMAs wait)
        float act[64];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c16 = 4 * hf + cc;  // 16-row piece
          uint32_t g[16], u[16];
          tc::tmem_ld_x16(tacc + 16 * c16, g);
          tc::tmem_ld_x16(tacc + 128 + 16 * c16, u);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            act[16 * cc + i] =
                activation_fast(__uint_as_float(g[i]), __uint_as_float(u[i]), f.act_kind, f.b1, f.b2);
        }
        uint32_t g2[2][16], u2[2][16];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          tc::tmem_ld_x16(tacc + 16 * (4 * hf + 2 + cc), g2[cc]);
          tc::tmem_ld_x16(tacc + 128 + 16 * (4 * hf + 2 + cc), u2[cc]);
        }
        tc::tmem_ld_wait();
        tc::fence_before_sync();
        named_bar(kEpiBarW, 32 * kEpiWarpsW);
        if (et == 0) mbar_arrive(&accempty);  // the next tile's MMAs may start
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int i = 0; i < 16; ++i)
            act[32 + 16 * cc + i] = activation_fast(__uint_as_float(g2[cc][i]),
                                                    __uint_as_float(u2[cc][i]), f.act_kind, f.b1, f.b2);
        if (m < wt.ntok) {
#pragma unroll
          for (int jg = 0; jg < 2; ++jg)
            store_act_group(f, *reinterpret_cast<float(*)[32]>(act + 32 * jg),
                            (size_t)(wt.pos0 + m), wt.rb * 4 + 2 * hf + jg);
        }
      } else {
        // o for the 256 output rows 256 rb .. 256 rb + 255, times the assignment's gate;
        // this warp takes columns 128 hf .. 128 hf + 127 of its 32 positions, read as 16
        // positions x 32 columns at a time (16x256b: four lanes hold 8 consecutive columns of
        // one position), so that each 8-byte store of four lanes fills a 32-byte sector of
        // one assignment's row with no exchange across the warp.  The next piece is read
        // while this one is stored; the accumulator is released once the last is read.
        const int t4 = lane & 3, r8 = lane >> 2;
        int ar[4];
        float gr[4];
        bool ok[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // rows 16 (i / 2) + 8 (i % 2) + lane / 4 of the warp's 32
          const int mm = 32 * q + 16 * (i >> 1) + 8 * (i & 1) + r8;
          ok[i] = mm < wt.ntok;
          ar[i] = ok[i] ? __ldg(f.perm + wt.pos0 + mm) : 0;
          gr[i] = ok[i] ? __ldg(f.gate + ar[i]) : 0.f;
        }
        const size_t col0 = (size_t)wt.rb * 256 + 128 * hf + 2 * t4;
        uint32_t u[2][16];
        tc::tmem_ld_16x256b_x4(tacc + 128 * hf, u[0]);
        tc::tmem_ld_wait_regs(u[0]);
#pragma unroll
        for (int pc = 0; pc < 8; ++pc) {  // piece: lanes 16 (pc / 4) .., columns 32 (pc % 4) ..
          if (pc < 7) {
            const int nx = pc + 1;
            tc::tmem_ld_16x256b_x4(tacc + ((uint32_t)(16 * (nx >> 2)) << 16) + 128 * hf + 32 * (nx & 3),
                                   u[nx & 1]);
          }
          const int h = pc >> 2, c = pc & 3;
#pragma unroll
          for (int e = 0; e < 2; ++e) {  // row lane / 4 (e = 0) or lane / 4 + 8 (e = 1)
            const int i = 2 * h + e;
            if (ok[i]) {
              float* yr = f.ybuf + (size_t)ar[i] * f.L + col0 + 32 * c;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                *reinterpret_cast<float2*>(yr + 8 * j) =
                    make_float2(gr[i] * __uint_as_float(u[pc & 1][4 * j + 2 * e]),
                                gr[i] * __uint_as_float(u[pc & 1][4 * j + 2 * e + 1]));
            }
          }
          if (pc < 7) tc::tmem_ld_wait_regs(u[(pc + 1) & 1]);
          if (pc == 6) {
            tc::fence_before_sync();
            named_bar(kEpiBarW, 32 * kEpiWarpsW);
            if (et == 0) mbar_arrive(&accempty);
          }
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncthreads();
  if (warp == kMmaWarpW) {
    if (lane == 0) mbar_wait(&drained, 0, f.status);
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(t0, kTmemColsW);
  }
}

// x (bf16, one row per token) -> kTerms MXFP4 terms per (token, expert) position for the
// large-batch path: codes in rows p * kTerms + t of xq [P * kTerms][L / 2] (as k_split_x),
// scales stage-major (wide_sf_offset).  One block per token, four threads per group of 32
// (eight elements each, split together by mx_split_quad8 with the hardware E2M1 rounding):
// each thread then writes its 4 code bytes of every term, and the group's first thread its
// scale word, to each valid slot's position (a warp's stores of a term row are 128
// contiguous bytes).
__global__ void __launch_bounds__(1024) k_split_x_wide(const uint16_t* __restrict__ x, int L, int k,
                                                       int E, int P, const int32_t* __restrict__ idx,
                                                       const int32_t* __restrict__ inv,
                                                       uint8_t* __restrict__ xq,
                                                       uint8_t* __restrict__ xsf) {
  __shared__ int spos[kMaxTopk];  // each slot's position, or -1
  pdl_wait();
  pdl_launch();
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    const int a = t * k + threadIdx.x;
    const int e = idx[a];
    spos[threadIdx.x] = (e >= 0 && e < E) ? inv[a] : -1;
  }
  const int grp = threadIdx.x >> 2, t4 = threadIdx.x & 3;  // blockDim.x == 4 (L / 32)
  const uint4 raw =
      __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * L + 32 * grp + 8 * t4));
  float r[8] = {bf16lo(raw.x), bf16hi(raw.x), bf16lo(raw.y), bf16hi(raw.y),
                bf16lo(raw.z), bf16hi(raw.z), bf16lo(raw.w), bf16hi(raw.w)};
  uint32_t w[kTerms], sf[kTerms];
  mx_split_quad8(r, w, sf);
  const uint32_t sfword = sf[0] | (sf[1] << 8) | (sf[2] << 16) | (sf[3] << 24);
  __syncthreads();  // spos
  const size_t row = (size_t)(L >> 1);
  for (int j = 0; j < k; ++j) {
    const int pos = spos[j];
    if (pos < 0) continue;
    uint8_t* dst = xq + (size_t)pos * kTerms * row + grp * 16 + 4 * t4;
#pragma unroll
    for (int tt = 0; tt < kTerms; ++tt) *reinterpret_cast<uint32_t*>(dst + tt * row) = w[tt];
    if (t4 == 0) *reinterpret_cast<uint32_t*>(xsf + wide_sf_offset(grp, pos, P)) = sfword;
  }
}

template <int PH, bool TR>
cudaError_t launch_wide_phase(const WMaps& mp, const WArgs& f, cudaStream_t s, bool pdl) {
  static int configured[64] = {0};
  constexpr size_t smem = WLay<PH, TR>::kSmemBytes;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_moe_wide<PH, TR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  const int grid = sm_count() < kTcMaxGrid ? sm_count() : kTcMaxGrid;
  return launch_kernel(k_moe_wide<PH, TR>, dim3(grid), dim3(kThreadsW), smem, s, pdl, mp, f);
}

}  // namespace

bool wide_path_supported(int L, int I) { return L % 512 == 0 && I % 512 == 0; }

cudaError_t launch_split_x_wide(const uint16_t* x, int T, int L, int k, int E, const int32_t* idx,
                                const BucketOut& b, uint8_t* xq, uint8_t* xsf, cudaStream_t s,
                                bool pdl) {
  if (k > kMaxTopk || L / 8 > 1024) return cudaErrorInvalidValue;
  return launch_kernel(k_split_x_wide, dim3(T), dim3(L / 8), 0, s, pdl, x, L, k, E, T * k,
                       idx, static_cast<const int32_t*>(b.inv), xq, xsf);
}

// Token groups of the table a call of T tokens reads (rows: kTcRowTok positions per group).
static size_t wide_groups(int E, int T, int k, bool rows) {
  const int pos = rows ? kTcRowTok : kTcWideTok;
  return ((size_t)T * k + pos - 1) / pos + E + 1;
}

size_t wide_desc_count(int L, int I, int E, int T, int k) {
  // a workspace for T tokens serves every call of up to T tokens: the larger of the two tables
  const int Tr = T < kWideMinTokens ? T : kWideMinTokens - 1;
  size_t g = wide_groups(E, Tr, k, true);
  const size_t gw = wide_groups(E, T, k, false);
  g = g > gw ? g : gw;
  return g * (size_t)(I / 128) + g * (size_t)(L / 256);
}

void wide_desc_setup(BucketOut& b, int4* desc, int L, int I, int E, int T, int k, bool rows) {
  b.wdesc = desc;
  b.wrb0 = I / 128;
  b.wrb1 = L / 256;
  b.wdesc1 = (int32_t)(wide_groups(E, T, k, rows) * (size_t)b.wrb0);
  b.wmode = rows ? 2 : 1;
}

cudaError_t launch_wide_experts(const ExpertPtrs& w, int L, int I, int E, int T, int k, bool rows,
                                const uint8_t* xq, const uint8_t* xsf, const BucketOut& b,
                                uint8_t* act_q, uint8_t* act_sf, int act_kind, float b1, float b2,
                                const float* gate, float* ybuf, int32_t* status, cudaStream_t s,
                                void (*between)(cudaStream_t)) {
  const uint64_t P = (uint64_t)T * k;
  const int pos_tile = rows ? kTcRowTok : kTcWideTok;
  // the preparation wrote the tile descriptors (wide_desc_setup)
  if (!b.wdesc || b.wmode != (rows ? 2 : 1) || b.wrb0 != I / 128 || b.wrb1 != L / 256)
    return cudaErrorInvalidValue;
  int4* desc0 = b.wdesc;
  int4* desc1 = b.wdesc + b.wdesc1;
  WMaps m0, m1;
  const auto sw64 = CU_TENSOR_MAP_SWIZZLE_64B, none = CU_TENSOR_MAP_SWIZZLE_NONE;
  // activation terms: boxes of 128 positions of one term (folded, 64-byte rows) or of 128
  // term rows (rows, 128-byte rows); weights: rows of the same width
  const auto sw = rows ? CU_TENSOR_MAP_SWIZZLE_128B : sw64;
  const uint32_t rowb = rows ? 128 : 64;
  auto amap = [&](CUtensorMap* m, const void* base, int K) {
    return rows ? make_map_2d_sw(m, base, K / 2, P * kTerms, rowb, kWM / 4, sw)
                : make_map_3d(m, base, K / 2, kTerms, K / 2, P, (uint64_t)kTerms * (K / 2), rowb,
                              kWM, sw);
  };
  if (!amap(&m0.a, xq, L) ||
      !make_map_2d_sw(&m0.as, xsf, 16, (uint64_t)(L / 128) * P, 16, pos_tile, none) ||
      !make_map_2d_sw(&m0.w0, w.w1p, L / 2, (uint64_t)E * I, rowb, 128, sw) ||
      !make_map_2d_sw(&m0.w1, w.w3p, L / 2, (uint64_t)E * I, rowb, 128, sw) ||
      !make_map_2d_sw(&m0.s0, w.w1s, L / 32, (uint64_t)E * I, 16, 128, none) ||
      !make_map_2d_sw(&m0.s1, w.w3s, L / 32, (uint64_t)E * I, 16, 128, none) ||
      !amap(&m1.a, act_q, I) ||
      !make_map_2d_sw(&m1.as, act_sf, 16, (uint64_t)(I / 128) * P, 16, pos_tile, none) ||
      !make_map_2d_sw(&m1.w0, w.w2p, I / 2, (uint64_t)E * L, rowb, 256, sw) ||
      !make_map_2d_sw(&m1.s0, w.w2s, I / 32, (uint64_t)E * L, 16, 256, none))
    return cudaErrorInvalidValue;
  m1.w1 = m1.w0;
  m1.s1 = m1.s0;
  WArgs f{};
  f.P = (int)P;
  f.meta = b.meta;
  f.perm = b.perm;
  f.act_q = act_q;
  f.act_sf = act_sf;
  f.I = I;
  f.L = L;
  f.act_kind = act_kind;
  f.b1 = b1;
  f.b2 = b2;
  f.gate = gate;
  f.ybuf = ybuf;
  f.status = status;
  // GEMM1: w1 and w3 -> act terms
  f.K = L;
  f.R = I;
  f.RB = I / 128;
  f.desc = desc0;
  cudaError_t e = rows ? launch_wide_phase<0, true>(m0, f, s, true)
                       : launch_wide_phase<0, false>(m0, f, s, true);
  if (e != cudaSuccess) return e;
  if (between) between(s);
  // GEMM2: w2 -> gate * o per assignment
  f.K = I;
  f.R = L;
  f.RB = L / 256;
  f.desc = desc1;
  return rows ? launch_wide_phase<1, true>(m1, f, s, true) : launch_wide_phase<1, false>(m1, f, s, true);
}

}  // namespace k3
