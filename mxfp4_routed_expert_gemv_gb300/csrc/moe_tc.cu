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
// Two launches of one persistent kernel: phase 0 (w1, w3 -> act terms) and phase 1 (w2 ->
// gate * o per assignment).  A phase is a list of tiles of 128 weight rows x (up to 16 of an
// expert's tokens) x the full reduction, cut into units of 512 (or 1024) reduction elements; CTA c (one
// per SM) takes units [U c / G, U (c+1) / G), balanced to one unit whatever the routing.  A
// tile cut by a range boundary is finished by the CTA holding its first unit (its "head"),
// which processes it last; the others process their part first and leave it in global
// memory with a flag.  While the head's last MMAs run, a helper thread waits for those flags
// and bulk-copies the parts into shared memory, so the end of the kernel does no global round
// trip.  Parts are added in CTA order (deterministic).
//
// Roles (352 threads): warps 0-3 epilogue (TMEM lane quarters 0-3), warps 4-7 move each
// stage's scales into TMEM (a 0xFF scale byte, "no value", becomes 0 there), warp 8 issues
// the weight TMA copies into the ring (one 64 KB unit per stage, see Lay), warp 10 the
// activation copies (and then fetches the parts of a shared last tile), warp 9 allocates
// TMEM and issues the MMAs.  Every wait is bounded; one that runs out sets the status
// block's timeout count and the CTA stops.  Each phase (and unit shape) is its own kernel.
#include "launch.h"
#include "mxq.cuh"
#include "tc.cuh"
#include "tmap.h"
#include "topk.cuh"

namespace k3 {
namespace {

constexpr int kKStage = 512;                                 // reduction elements per stage
constexpr int kMmas = kKStage / 64;                          // MMAs per stage (K = 64 each)
constexpr int kTokTile = kTcTokTile;                         // tokens per tile
constexpr int kRowsTile = 128;                               // MMA M
constexpr uint32_t kABytes = kRowsTile * (kKStage / 2);      // 32768: two 16 KB swizzle columns
constexpr uint32_t kSABytes = kRowsTile * (kKStage / 32);    // 2048
constexpr int kThreads = 352;
constexpr int kSfWarp0 = 4, kProdWarp = 8, kMmaWarp = 9, kBWarp = 10;
constexpr uint32_t kTmemCols = 512;
constexpr int kEpiBar = 1;  // named barrier of the four epilogue warps

// Shared-memory and TMEM layout for tiles of at most NMAX activation rows (MMA N: 16 for
// batches of up to 4 tokens, 64 otherwise), NM weight matrices per unit (2 in the first
// GEMM, w1 and w3; 1 in the second) and KS 512-chunks of the reduction per unit (1, or 2 in
// the second GEMM when its reduction allows).  A ring stage holds one whole unit: NM x KS
// weight blocks of 128 x 512, so a stage is 64 KB of weights either way (fewer, larger TMA
// batches stream HBM faster than more, smaller ones).  Block (m, ks) is sub-block
// sb = m KS + ks.
//   stage: A of sub-block sb at sb * 32 KB | B of chunk ks (two 128-byte columns of NMAX
//          rows) | A scales of sb, 128 x 16 B each | B scales of ks, NMAX x 16 B each,
//          padded to a multiple of 1 KB;
//   TMEM:  accumulator buffer b at b * kAccCols, matrix m at + m * kMatCols; the scale ring
//          from kSfBase, stage s at + kSfStageCols s: A scales of sb, MMA j at + 32 sb + 4 j
//          (+ lane quarter), B scales of ks at + 32 (NM KS + ks) + 4 j (+ 1 for B rows 32..63);
//   fix:   the parts a head tile adds, after the ring (kFixBytes), then the act buffer.
template <int NMAX, int NM, int KS, int BR>
struct Lay {
  // BR activation rows are stored per chunk: NMAX, or 8 for one token (its 4 term rows; the
  // MMA's rows 8..15 read the same 8 rows again, columns that are never used), which keeps
  // a third ring stage in reach of the second GEMM
  static constexpr uint32_t kBKatom = BR * 128;
  static constexpr uint32_t kBBytes = 2 * kBKatom;
  static constexpr uint32_t kSBBytes = BR * (kKStage / 32);
  static constexpr uint32_t kOffB = NM * KS * kABytes, kOffSA = kOffB + KS * kBBytes;
  static constexpr uint32_t kOffSB = kOffSA + NM * KS * kSABytes;
  static constexpr uint32_t kStageBytes = ((kOffSB + KS * kSBBytes + 1023) / 1024) * 1024;
  static constexpr int kStages =
      NM * KS == 2 ? ((NMAX <= 16 && NM == 2) || BR == 8 ? 3 : 2) : (NMAX <= 16 ? 5 : 4);
  static constexpr uint32_t kFixBytes = (NMAX <= 16 && NM == 2) || BR == 8 ? 4096 : 16384;
  static constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + kFixBytes + 1024;
  static constexpr uint32_t kMatCols = NMAX <= 16 ? 32 : 64;
  static constexpr uint32_t kAccCols = 2 * kMatCols;
  static constexpr uint32_t kSfBase = 2 * kAccCols;
  static constexpr uint32_t kSfStageCols = 32 * (NM * KS + KS);
  static_assert(kSfBase + kStages * kSfStageCols <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared-memory budget");
  static_assert(NMAX % 16 == 0 && NMAX <= 64, "tile height");
};

struct FArgs {
  int ph;                  // 0: w1, w3 -> act terms; 1: w2 -> gate * o
  int one_token;           // T == 1: phase-0 activation rows are 0 .. kTerms-1
  // route_one: one token, no preparation launch.  Phase-0 CTAs each route the token from the
  // router's logits; CTA 0 publishes idx, gate, gap and the route words; phase-1 CTAs read
  // the route words.
  int route_one;
  const float *logits, *bias;
  int E, renorm;
  float routed_scale;
  int32_t* idx_out;
  float *gate_out, *gap_out;
  unsigned long long* route_words;  // [k] the routing, one self-flagged word per expert
  float* y;                // one routed token: y [L], summed by the second GEMM
  int32_t* ycount;         // [L / 128] slots written per 128-row tile of y (zeroed)
  int k, L, I, act_kind;
  float b1, b2;
  int KC, RT, R;           // reduction chunks, row tiles, rows per expert
  const int32_t *meta, *perm;
  const int32_t* nbase;     // [active experts + 1] first token group of each active expert
  const int4* tiles;        // per token group: expert, first position, token count
  uint8_t *act_q, *act_sf;  // phase-0 output = phase-1 activation operand
  const float* gate;
  float* ybuf;              // [T*k][L]
  float* part;              // [kTcMaxGrid] parts of shared tiles (one per CTA)
  int npart;                // tokens per part
  int32_t* flags;           // [kTcMaxGrid] part written (zeroed before the launch)
  int32_t* status;
  uint32_t flag_polls;      // polls a wait on a flag or routing word makes before it gives up
};

// Units [lo(c), lo(c+1)) of U go to CTA c of G: lo(c) = floor(U c / G), from U = q G + r as
// q c + floor(r c / G), in 32-bit arithmetic (U < 2^31, r c < G^2).
struct Split {
  int U, q, r, G;
  __device__ __forceinline__ Split(int U_, int G_) : U(U_), q(U_ / G_), r(U_ % G_), G(G_) {}
  __device__ __forceinline__ int lo(int c) const { return q * c + (r * c) / G; }
};

int tc_grid_size() { return sm_count() < kTcMaxGrid ? sm_count() : kTcMaxGrid; }

// floats of one CTA's part: NM matrices x npart tokens x 128 rows, element (m, j, r) at
// (m * npart + j) * 128 + r
__device__ __forceinline__ size_t part_floats(int NM, int npart) {
  return (size_t)NM * npart * 128;
}

struct TileInfo {
  int rt, expert, pos0, ntok, N;
  bool shared_rows;  // other tiles of this launch read the same weight rows
};
// Tiles in order: expert by expert (active experts ascending), and within an expert with n
// token groups, row tile by row tile, each row tile once per group (tile = base + rt n + g),
// so that the n tiles reading the same 128 weight rows follow each other and the rows come
// from L2 after the first.  A cursor walks a CTA's tiles in increasing order: it finds the
// expert block of its first tile by bisection over the groups' prefix (nbase, from the
// preparation), then steps block by block.  One routed token: one group per expert, from
// the CTA's own table.
struct TileCursor {
  int a = -1, gb = 0, n = 1, t_lo = 0, t_hi = 0;
  template <bool ONE>
  __device__ __forceinline__ TileInfo get(int tile, const FArgs& f, const int4* own) {
    TileInfo t;
    int ntg;
    if constexpr (ONE) {
      ntg = tile / f.RT;
      t.rt = tile - ntg * f.RT;
      n = 1;
    } else {
      if (a < 0) {  // bisection: the last active expert whose first tile is <= tile
        int lo = 0, hi = f.meta[0] - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (__ldg(f.nbase + mid) * f.RT <= tile) lo = mid; else hi = mid - 1;
        }
        a = lo - 1;
      }
      while (a < 0 || tile >= t_hi) {
        ++a;
        gb = __ldg(f.nbase + a);
        n = __ldg(f.nbase + a + 1) - gb;
        t_lo = gb * f.RT;
        t_hi = t_lo + n * f.RT;
      }
      const int local = tile - t_lo;
      t.rt = local / n;
      ntg = gb + (local - t.rt * n);
    }
    const int4 g = ONE ? own[ntg] : __ldg(f.tiles + ntg);
    t.expert = g.x;
    t.pos0 = g.y;
    t.ntok = g.z;
    t.N = ((t.ntok * kTerms + 15) / 16) * 16;
    t.shared_rows = n > 1;
    return t;
  }
};

__device__ __forceinline__ void st_release(int32_t* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Release-acquire add at GPU scope: its release covers what a CTA barrier before it
// ordered, its acquire what a barrier after it orders.
__device__ __forceinline__ int atom_add_acq_rel(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One token's routing for an expert-GEMM CTA (every thread calls it).  Phase 0: the CTA
// routes the token itself from the router's logits (the ring, free until the producers
// start, is the scratch); CTA 0 also publishes the result, the routing as one self-flagged
// 64-bit word per expert (no fence: each word carries its own ready bit).  Phase 1: the
// words CTA 0 of phase 0 published, one load each once written.  Out (shared): tiles[i] =
// (expert, i, 1) for the chosen experts in ascending order, perm[i] = the choice index of
// tile i, gate[j] = gate of choice j.  Returns the number of token groups (0 after a timeout).
template <int PH>
__device__ __forceinline__ int route_one_token(const FArgs& f, uint8_t* scratch, int4* tiles,
                                               int* perm, float* gate, bool publish) {
  __shared__ int ngroups;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, k = f.k;
  if (PH == 0) {
    const OneTokenChoice c = topk_one_token<3>(
        f.logits, f.bias, f.E, k, f.renorm, f.routed_scale, publish ? f.gap_out : nullptr,
        reinterpret_cast<unsigned long long*>(scratch), reinterpret_cast<float*>(scratch + 4096));
    if (warp == 0) {
      if (lane < k) {
        gate[lane] = c.g;
        tiles[c.rank] = make_int4(c.e, c.rank, 1, 0);
        perm[c.rank] = lane;
        if (publish) {
          f.idx_out[lane] = c.e;
          f.gate_out[lane] = c.g;
          const unsigned long long w =
              ((unsigned long long)__float_as_uint(c.g) << 32) |
              (0x80000000u | ((uint32_t)lane << 16) | (uint32_t)c.e);
          asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(f.route_words + c.rank),
                       "l"(w)
                       : "memory");
        }
      }
      if (lane == 0) ngroups = k;
    }
  } else if (warp == 0) {
    // lane i: the word of the i-th chosen expert (ascending index), polled until written
    unsigned long long w = 0ull;
    if (lane < k) {
      for (uint32_t q = 0; q < f.flag_polls; ++q) {
        asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(f.route_words + lane)
                     : "memory");
        if (w & 0x80000000ull) break;
        __nanosleep(64);
      }
    }
    const bool got = __all_sync(0xffffffffu, lane >= k || (w & 0x80000000ull) != 0ull);
    if (got && lane < k) {
      const int e = (int)(w & 0xFFFFu), j = (int)((w >> 16) & 0x7FFFu);
      tiles[lane] = make_int4(e, lane, 1, 0);
      perm[lane] = j;
      gate[j] = __uint_as_float((uint32_t)(w >> 32));
    }
    if (lane == 0) {
      ngroups = got ? k : 0;
      if (!got && f.status) atomicAdd(f.status + kStatTimeout, 1);
    }
  }
  __syncthreads();
  return ngroups;
}

// bytes 0xFF -> 0x00 (an E8M0 "no value" becomes the smallest scale: the group adds nothing
// measurable, as the zero group of the README "kimi-k3-in-c" decoder, Part II section 4)
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

// generic-proxy global writes seen through an acquire -> later bulk/TMA (async proxy) reads
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Maps: phase 0: [0] w1 [1] w1 scales [2] w3 [3] w3 scales [4] x terms [5] their scales;
// phase 1: [0] w2 [1] w2 scales [2] w2 [3] w2 scales [4] act terms [5] their scales.
// Per phase: [0..1] first weight matrix and its scales, [2..3] the second (phase 0: w3;
// phase 1: w2 again), [4..5] activation terms and scales.
// N consecutive 32-bit TMEM columns of this warp's lane quarter into registers (N = 4 or 16),
// waiting for the load.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 4 || N == 16, "column count");
  if constexpr (N == 4) {
    asm volatile(
        "{\n\ttcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t}"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(taddr)
        : "memory");
  } else {
    tc::tmem_ld_x16(taddr, r);
    tc::tmem_ld_wait();
  }
}

struct Maps {
  CUtensorMap m[6];
};

// The CTA's range in tiles: the first tile (maybe shared, part at the front), whole tiles,
// the last tile (maybe shared, this CTA its head: parts of later CTAs are added to it).
struct Range {
  int u0, u1;
  int t_first, t_last;
  bool tail_first;   // the first tile started in an earlier CTA: leave a part
  bool head_last;    // the last tile continues in later CTAs: add their parts
};
__device__ __forceinline__ Range make_range(const Split& sp, int KC, int c) {
  Range r;
  r.u0 = sp.lo(c);
  r.u1 = sp.lo(c + 1);
  r.t_first = (int)(r.u0 / KC);
  r.t_last = r.u1 > r.u0 ? (int)((r.u1 - 1) / KC) : r.t_first - 1;
  r.tail_first = r.u1 > r.u0 && r.u0 % KC != 0;
  r.head_last = r.u1 > r.u0 && r.u1 % KC != 0 && (r.t_last != r.t_first || !r.tail_first);
  return r;
}

template <int NMAX, int PH, int KS, bool ONE>
__global__ void __launch_bounds__(kThreads, 1) k_moe_tc(const __grid_constant__ Maps mp,
                                                        const FArgs f) {
  constexpr int NM = PH == 0 ? 2 : 1;  // weight matrices per unit: w1 and w3, or w2
  constexpr int TB = NMAX / 16;        // tokens per epilogue step
  constexpr int BR = ONE ? 8 : NMAX;   // activation rows stored per chunk
  using Y = Lay<NMAX, NM, KS, BR>;
  constexpr int kStages = Y::kStages;
  constexpr uint32_t kStageBytes = Y::kStageBytes, kBKatom = Y::kBKatom;
  constexpr uint32_t kOffB = Y::kOffB, kOffSA = Y::kOffSA, kOffSB = Y::kOffSB;
  constexpr uint32_t kBBytes = Y::kBBytes, kSBBytes = Y::kSBBytes;
  constexpr uint32_t kAccCols = Y::kAccCols, kMatCols = Y::kMatCols, kSfBase = Y::kSfBase;
  constexpr uint32_t kSfStageCols = Y::kSfStageCols, kFixBytes = Y::kFixBytes;
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t fullA[kStages], fullB[kStages], sfready[kStages], empty[kStages];
  __shared__ __align__(8) uint64_t accfull[2], accempty[2], drained, fixfull;
  __shared__ uint32_t tbase;
  __shared__ int abort_flag, y_last;
  __shared__ int4 own_tiles[32];  // route_one: this CTA's table of token groups
  __shared__ int own_perm[32];
  __shared__ float own_gate[32];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) &
                                           ~uintptr_t(1023));
  float* fix = reinterpret_cast<float*>(sm + (size_t)kStages * kStageBytes);
  // many tokens per tile: each lane splits one token's group (no cross-lane work); one token
  // per tile: the warp splits the group together
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&fullA[s], 1);
      mbar_init(&fullB[s], 1);
      mbar_init(&sfready[s], 4);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], 4);
    }
    mbar_init(&drained, 1);
    mbar_init(&fixfull, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&tbase, kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == kProdWarp && lane == 0)
    for (int i = 0; i < 6; ++i) tc::tma_prefetch_map(&mp.m[i]);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // Phase 0 reads what the preparation (or the router) wrote: everyone waits for the previous
  // launch.  Phase 1 starts streaming its weights at once: the routing it reads (or the
  // logits it routes from) was complete before phase 0 passed this point (phase 0 lets this
  // launch start only after its own wait), and only the activation terms come from phase 0,
  // so only the thread that loads them waits.
  // (A single routed token has k token groups whatever the routing, so its CTAs lay out
  // their ranges before the wait and route after it.)
  if (!ONE) {
    if (PH == 0) pdl_wait();
    pdl_launch();
  }
  const uint32_t t0 = tbase;
  volatile int* abort_v = &abort_flag;
  const int ngroups = ONE ? f.k : f.meta[2];

  const Split sp(ngroups * f.RT * f.KC, G);
  const Range rg = make_range(sp, f.KC, cta);
  const int ntiles = rg.t_last - rg.t_first + 1;  // tiles this CTA touches (0 if idle)
  // the later CTAs whose parts the head tile needs, and where their parts land in `fix`
  int fix_c0 = cta + 1, fix_c1 = cta;  // [fix_c0, fix_c1]
  if (rg.head_last) {
    const int tend = (rg.t_last + 1) * f.KC;
    while (fix_c1 + 1 < G && sp.lo(fix_c1 + 1) < tend) ++fix_c1;
  }
  const size_t pf = part_floats(NM, f.npart);
  // this phase's parts (the phases have separate regions: phase 1 may start before phase 0
  // has finished with its parts)
  float* const parts = f.part + (PH == 0 ? 0 : (size_t)kTcMaxGrid * part_floats(2, f.npart));
  // an idle CTA (empty range, when there are fewer units than CTAs) leaves no part
  auto idle = [&](int c) { return sp.lo(c + 1) == sp.lo(c); };
  int nfix = 0;
  for (int c = fix_c0; c <= fix_c1; ++c) nfix += idle(c) ? 0 : 1;
  const bool fix_smem = (size_t)nfix * pf * 4 <= kFixBytes;
  if (ONE) {
    if (PH == 0) pdl_wait();
    pdl_launch();
    if (route_one_token<PH>(f, sm, own_tiles, own_perm, own_gate, PH == 0 && cta == 0) == 0)
      *abort_v = 1;  // the routing words never came: every role stops at its first wait
  }

  if (warp == kProdWarp || warp == kBWarp) {
    // ------------------------------------- TMA: weights (warp 8), activations (warp 10)
    if (lane == 0) {
      const bool wts = warp == kProdWarp;
      if (!wts && PH == 1) pdl_wait();  // the activation terms are phase 0's output
      // weights read once per call go evict-first; rows that several token groups read
      // (consecutive tiles) stay at normal priority for the reuse
      const uint64_t once = tc::make_policy_evict_first(), reused = tc::make_policy_evict_normal();
      int it = 0;
      bool stop = false;
      TileCursor cur;
      for (int ti_ = 0; ti_ < ntiles && !stop; ++ti_) {
        const int tile = rg.t_first + ti_;
        const TileInfo ti = cur.get<ONE>(tile, f, own_tiles);
        const int kb = ti_ == 0 ? rg.u0 - tile * f.KC : 0;
        const int ke = ti_ == ntiles - 1 ? rg.u1 - tile * f.KC : f.KC;
        const int nbox = ONE ? 1 : ti.N / 16;  // boxes of BR (one token) or 16 rows
        const int arow = ti.expert * f.R + ti.rt * kRowsTile;
        for (int kc = kb; kc < ke && !stop; ++kc, ++it) {
          const int s = it % kStages;
          if (*abort_v ||
              (it >= kStages &&
               !mbar_wait_ab(&empty[s], ((it / kStages) - 1) & 1, f.status, abort_v))) {
            *abort_v = 1;
            stop = true;
            break;
          }
          uint8_t* st = sm + (size_t)s * kStageBytes;
          if (wts) {
            const uint64_t pol = ti.shared_rows ? reused : once;
            mbar_arrive_expect_tx(&fullA[s], NM * KS * (kABytes + kSABytes));
#pragma unroll
            for (int m = 0; m < NM; ++m) {
#pragma unroll
              for (int ks = 0; ks < KS; ++ks) {
                const int sb = m * KS + ks, x = (kc * KS + ks) * 256;
                uint8_t* sa = st + sb * kABytes;
                tc::tma_load_2d_hint(sa, &mp.m[2 * m], x, arow, &fullA[s], pol);
                tc::tma_load_2d_hint(sa + 16384, &mp.m[2 * m], x + 128, arow, &fullA[s], pol);
                tc::tma_load_2d_hint(st + kOffSA + sb * kSABytes, &mp.m[2 * m + 1],
                                     (kc * KS + ks) * 16, arow, &fullA[s], pol);
              }
            }
          } else {
            // one token: its terms are rows 0 .. kTerms-1 whatever the position (the router
            // launch writes only those; the per-position layout repeats them)
            const int brow0 = f.one_token ? 0 : ti.pos0 * kTerms;
            constexpr uint32_t kBox = (ONE ? 8 : 16) * 128, kSBox = (ONE ? 8 : 16) * 16;
            mbar_arrive_expect_tx(&fullB[s], (uint32_t)(KS * nbox) * (2 * kBox + kSBox));
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              uint8_t* sbk = st + kOffB + ks * kBBytes;
              const int x = (kc * KS + ks) * 256;
              for (int b = 0; b < nbox; ++b) {
                tc::tma_load_2d(sbk + b * kBox, &mp.m[4], x, brow0 + 16 * b, &fullB[s]);
                tc::tma_load_2d(sbk + kBKatom + b * kBox, &mp.m[4], x + 128, brow0 + 16 * b,
                                &fullB[s]);
                tc::tma_load_2d(st + kOffSB + ks * kSBBytes + b * kSBox, &mp.m[5],
                                (kc * KS + ks) * 16, brow0 + 16 * b, &fullB[s]);
              }
            }
          }
        }
      }
      if (!wts && !stop && rg.head_last && fix_smem) {
        // parts of the shared last tile: wait for each later CTA's flag, then bulk-copy its
        // part into `fix` (it lands while this CTA's last MMAs run).  Each copy adds its bytes
        // to the barrier's count before it starts and the one arrival comes after the last
        // copy (or the wait that gave up), so the phase completes once every copy that was
        // started has landed, whether or not all of them were.
        bool ok = true;
        int slot = 0;
        for (int c = fix_c0; c <= fix_c1 && ok; ++c) {
          if (idle(c)) continue;
          int got = 0;
          for (uint32_t q = 0; q < f.flag_polls && !got && !*abort_v; ++q) {
            got = ld_acquire(f.flags + c) == 1;
            if (!got) __nanosleep(256);
          }
          if (!got) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          mbar_expect_tx(&fixfull, (uint32_t)(pf * 4));
          bulk_g2s(fix + (size_t)slot * pf, parts + (size_t)c * pf, (uint32_t)(pf * 4), &fixfull);
          ++slot;
        }
        mbar_arrive(&fixfull);
        if (!ok) {
          if (!*abort_v && f.status) atomicAdd(f.status + kStatTimeout, 1);
          *abort_v = 1;
          stop = true;
          mbar_wait(&fixfull, 0, nullptr);  // the copies already started land first
        }
      }
      if (*abort_v) {
        // copies still in flight land before the CTA leaves: wait for each stage's last fill
        for (int d = 1; d <= kStages && d <= it; ++d) {
          const int i = it - d;
          mbar_wait(wts ? &fullA[i % kStages] : &fullB[i % kStages], (i / kStages) & 1, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp >= kSfWarp0 && warp < kSfWarp0 + 4) {
    // ---------------------------------------------------------------- scales -> TMEM
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    int it = 0;
    bool stop = false;
    TileCursor cur;
    for (int ti_ = 0; ti_ < ntiles && !stop; ++ti_) {
      const int tile = rg.t_first + ti_;
      const int N = cur.get<ONE>(tile, f, own_tiles).N;
      const int kb = ti_ == 0 ? rg.u0 - tile * f.KC : 0;
      const int ke = ti_ == ntiles - 1 ? rg.u1 - tile * f.KC : f.KC;
      for (int kc = kb; kc < ke && !stop; ++kc, ++it) {
        const int s = it % kStages;
        const uint32_t par = (it / kStages) & 1;
        const bool ok = !*abort_v &&
                        mbar_wait_ab(&fullA[s], par, lane == 0 ? f.status : nullptr, abort_v) &&
                        mbar_wait_ab(&fullB[s], par, lane == 0 ? f.status : nullptr, abort_v);
        if (!__all_sync(0xffffffffu, ok)) {
          *abort_v = 1;
          stop = true;
          break;
        }
        const uint8_t* st = sm + (size_t)s * kStageBytes;
        const uint32_t ring = t0 + lane_off + kSfBase + (uint32_t)s * kSfStageCols;
#pragma unroll
        for (int sb = 0; sb < NM * KS; ++sb) {
          const uint4 sa =
              *reinterpret_cast<const uint4*>(st + kOffSA + sb * kSABytes + 16 * (32 * q + lane));
          const uint32_t wa[4] = {clear_ff_bytes(sa.x), clear_ff_bytes(sa.y),
                                  clear_ff_bytes(sa.z), clear_ff_bytes(sa.w)};
#pragma unroll
          for (int j = 0; j < kMmas; ++j)
            tc::tmem_st_x1(ring + 32 * sb + 4 * j + q, (wa[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
        }
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint32_t rb = ring + 32 * (NM * KS + ks);
          const uint8_t* sbs = st + kOffSB + ks * kSBBytes;
          const uint4 sb0 = lane < BR ? *reinterpret_cast<const uint4*>(sbs + 16 * lane)
                                      : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t wb0[4] = {sb0.x, sb0.y, sb0.z, sb0.w};
#pragma unroll
          for (int j = 0; j < kMmas; ++j)
            tc::tmem_st_x1(rb + 4 * j, (wb0[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
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
      int it = 0;
      bool stop = false;
      TileCursor cur;
      for (int ti_ = 0; ti_ < ntiles && !stop; ++ti_) {
        const int tile = rg.t_first + ti_;
        const int kb = ti_ == 0 ? rg.u0 - tile * f.KC : 0;
        const int ke = ti_ == ntiles - 1 ? rg.u1 - tile * f.KC : f.KC;
        const int b = ti_ & 1;
        if (ti_ >= 2 && !mbar_wait_ab(&accempty[b], ((ti_ >> 1) - 1) & 1, f.status, abort_v)) {
          *abort_v = 1;
          stop = true;
          break;
        }
        const uint32_t idesc = tc::idesc_mxf4(kRowsTile, cur.get<ONE>(tile, f, own_tiles).N, 0, 0);
        for (int kc = kb; kc < ke && !stop; ++kc, ++it) {
          const int s = it % kStages;
          const uint32_t par = (it / kStages) & 1;
          // the scale warps arrive on sfready only after they have seen both of the stage's
          // copies land, so this one wait covers all three barriers
          if (*abort_v || !mbar_wait_ab(&sfready[s], par, f.status, abort_v)) {
            *abort_v = 1;
            stop = true;
            break;
          }
          tc::fence_after_sync();
          const uint32_t st = tc::smem_addr(sm + (size_t)s * kStageBytes);
          const uint32_t sfr = t0 + kSfBase + (uint32_t)s * kSfStageCols;
#pragma unroll
          for (int m = 0; m < NM; ++m) {
            const uint32_t d = t0 + (uint32_t)b * kAccCols + kMatCols * m;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              const int sb = m * KS + ks;
#pragma unroll
              for (int j = 0; j < kMmas; ++j) {
                const uint32_t koff =
                    sb * kABytes + (uint32_t)(j >> 2) * 16384u + (uint32_t)(j & 3) * 32u;
                const uint32_t kboff =
                    ks * kBBytes + (uint32_t)(j >> 2) * kBKatom + (uint32_t)(j & 3) * 32u;
                const uint64_t ad = tc::smem_desc(st + koff, 16, 1024, tc::kLayout128B);
                // one token: SBO 0, the second 8-row group reads the first again
                const uint64_t bd =
                    tc::smem_desc(st + kOffB + kboff, 16, BR == 8 ? 0 : 1024, tc::kLayout128B);
                tc::mma_mxf4(d, ad, bd, idesc, sfr + 32 * sb + 4 * j,
                             sfr + 32 * (NM * KS + ks) + 4 * j,
                             (kc == kb && ks == 0 && j == 0) ? 0u : 1u);
              }
            }
          }
          tc::mma_commit(&empty[s]);
        }
        if (!stop) tc::mma_commit(&accfull[b]);
      }
      tc::mma_commit(&drained);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---------------------------------------------------------------- epilogue (warps 0-3)
    // Token by token (a short loop, not unrolled: this code runs once per tile, at the end
    // of the kernel for the last one, and stays small): each token's kTerms columns come
    // straight from TMEM and are summed in column order.
    const int q = warp;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const int row = 32 * q + lane;  // row within the tile
    TileCursor cur;
    for (int ti_ = 0; ti_ < ntiles; ++ti_) {
      const int tile = rg.t_first + ti_;
      const TileInfo ti = cur.get<ONE>(tile, f, own_tiles);
      const int b = ti_ & 1;
      const bool write_part = ti_ == 0 && rg.tail_first;          // leave a part for the head
      const bool add_parts = ti_ == ntiles - 1 && rg.head_last;    // add the later CTAs' parts
      int bad = (*abort_v || !mbar_wait_ab(&accfull[b], (ti_ >> 1) & 1, f.status, abort_v)) ? 1 : 0;
      if (add_parts && !bad) {
        if (fix_smem) {
          // the helper's copies complete this phase; if it gave up it set abort_v, and the
          // bounded wait ends here as well
          bad = (*abort_v || !mbar_wait_ab(&fixfull, 0, f.status, abort_v)) ? 1 : 0;
        } else if (threadIdx.x == 0) {
          // parts too large for `fix`: wait for their flags here, read them from global below
          for (int c = fix_c0; c <= fix_c1 && !bad; ++c) {
            if (idle(c)) continue;
            int got = 0;
            for (uint32_t qq = 0; qq < f.flag_polls && !got && !*abort_v; ++qq) {
              got = ld_acquire(f.flags + c) == 1;
              if (!got) __nanosleep(256);
            }
            if (!got) {
              if (!*abort_v && f.status) atomicAdd(f.status + kStatTimeout, 1);
              bad = 1;
            }
          }
        }
      }
      if (bar_or(kEpiBar, 128, bad)) {
        *abort_v = 1;
        break;
      }
      tc::fence_after_sync();
      const uint32_t tacc = t0 + lane_off + (uint32_t)b * kAccCols;
      const int grp = (ti.rt * kRowsTile + 32 * q) >> 5;            // phase 0: act group
      const bool in_range = ti.rt * kRowsTile + 32 * q < f.R;
      float* mine = parts + (size_t)cta * pf;
      // TB tokens at a time: one TMEM load of their 4 TB columns per matrix, then their
      // epilogues side by side
#pragma unroll 1
      for (int j0 = 0; j0 < ti.ntok; j0 += TB) {
        float v[TB][2];
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          uint32_t r[4 * TB];
          tmem_ld_cols<4 * TB>(tacc + kMatCols * m + (uint32_t)(j0 * kTerms), r);
#pragma unroll
          for (int jj = 0; jj < TB; ++jj)
            v[jj][m] = ((__uint_as_float(r[4 * jj]) + __uint_as_float(r[4 * jj + 1])) +
                        __uint_as_float(r[4 * jj + 2])) +
                       __uint_as_float(r[4 * jj + 3]);
        }
        const int nj = min(TB, ti.ntok - j0);
        if (write_part) {
#pragma unroll
          for (int jj = 0; jj < TB; ++jj)
            if (jj < nj)
              for (int m = 0; m < NM; ++m)
                mine[((size_t)m * f.npart + j0 + jj) * kRowsTile + row] = v[jj][m];
          continue;
        }
        if (add_parts) {
#pragma unroll
          for (int jj = 0; jj < TB; ++jj) {
            if (jj >= nj) break;
            for (int m = 0; m < NM; ++m) {
              const size_t off = ((size_t)m * f.npart + j0 + jj) * kRowsTile + row;
              int slot = 0;
              for (int c = fix_c0; c <= fix_c1; ++c) {
                if (idle(c)) continue;
                v[jj][m] += fix_smem ? fix[(size_t)slot * pf + off]
                                     : __ldcg(parts + (size_t)c * pf + off);
                ++slot;
              }
            }
          }
        }
        if (PH == 0) {
          // SwiGLU (or SiTU-GLU), then each token's kTerms MXFP4 terms for phase 1; this
          // warp's 32 rows are one group of 32 along phase 1's reduction
          float act[TB];
#pragma unroll
          for (int jj = 0; jj < TB; ++jj)
            act[jj] = activation(v[jj][0], v[jj][NM - 1], f.act_kind, f.b1, f.b2);
          uint32_t words[TB][kTerms], sfb[TB][kTerms];
          mx_split_groups<TB>(act, words, sfb);
          if (in_range) {
#pragma unroll
            for (int jj = 0; jj < TB; ++jj) {
              if (jj >= nj) break;
              const size_t p = (size_t)(ti.pos0 + j0 + jj);
#pragma unroll
              for (int t = 0; t < kTerms; ++t) {
                const size_t r2 = p * kTerms + t;
                if ((lane & 7) == 0)
                  *reinterpret_cast<uint32_t*>(f.act_q + r2 * (size_t)(f.I >> 1) + grp * 16 +
                                               4 * (lane >> 3)) = words[jj][t];
                if (lane == 0) f.act_sf[r2 * (size_t)(f.I >> 5) + grp] = (uint8_t)sfb[jj][t];
              }
            }
          }
        } else {
          const int r_exp = ti.rt * kRowsTile + row;  // row within the expert
#pragma unroll
          for (int jj = 0; jj < TB; ++jj) {
            if (jj >= nj) break;
            const int asg = ONE ? own_perm[ti.pos0 + j0 + jj] : f.perm[ti.pos0 + j0 + jj];
            const float gj = ONE ? own_gate[asg] : f.gate[asg];
            if (r_exp < f.R) f.ybuf[(size_t)asg * f.L + r_exp] = gj * v[jj][0];
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[b]);
      if (write_part) {
        __threadfence();
        named_bar(kEpiBar, 128);
        if (threadIdx.x == 0) st_release(f.flags + cta, 1);
      }
      if constexpr (ONE && PH == 1) {
        if (!write_part) {
          // the combine: count this slot for its 128-row tile of y; the CTA that writes the
          // k-th slot of a tile sums the token's slots there in slot order (as k_combine)
          named_bar(kEpiBar, 128);  // orders every row's slot write before the release
          if (threadIdx.x == 0) y_last = atom_add_acq_rel(f.ycount + ti.rt, 1) == f.k - 1;
          named_bar(kEpiBar, 128);
          const int r = ti.rt * kRowsTile + row;
          if (y_last && r < f.R) {
            float sv[kMaxTopk];
#pragma unroll
            for (int sl = 0; sl < kMaxTopk; ++sl)
              sv[sl] = sl < f.k ? __ldcg(f.ybuf + (size_t)sl * f.L + r) : 0.f;
            float acc = 0.f;
#pragma unroll
            for (int sl = 0; sl < kMaxTopk; ++sl)
              if (sl < f.k) acc += sv[sl];
            f.y[r] = acc;
          }
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncthreads();
  if (warp == kMmaWarp) {
    if (lane == 0) mbar_wait(&drained, 0, f.status);
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(t0, kTmemCols);
  }
}

// x (bf16, one row per token) -> kTerms MXFP4 terms per (token, expert) position, in the
// bucket order: rows p * kTerms + t of xq [P*kTerms][L/2] and xsf [P*kTerms][L/32].  Grid
// (T, L/512): one CTA per token and 512-wide slice; warp w splits group 16 * blockIdx.y + w
// of the token once and writes the terms to each of the token's valid positions (inv of
// its slots; slots whose expert index is out of range have none).
__global__ void __launch_bounds__(512) k_split_x(const uint16_t* __restrict__ x, int L, int k,
                                                 int E, const int32_t* __restrict__ idx,
                                                 const int32_t* __restrict__ inv,
                                                 uint8_t* __restrict__ xq,
                                                 uint8_t* __restrict__ xsf) {
  pdl_wait();
  pdl_launch();
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = blockIdx.y * 16 + warp;
  const float v = __uint_as_float((uint32_t)x[(size_t)t * L + 32 * grp + lane] << 16);
  uint32_t words[kTerms], sf[kTerms];
  mx_split_group(v, words, sf);
  for (int j = 0; j < k; ++j) {
    const int a = t * k + j;
    const int e = idx[a];
    if (e < 0 || e >= E) continue;
    const int pos = inv[a];
#pragma unroll
    for (int tt = 0; tt < kTerms; ++tt) {
      const size_t r = (size_t)pos * kTerms + tt;
      if ((lane & 7) == 0)
        *reinterpret_cast<uint32_t*>(xq + r * (size_t)(L >> 1) + grp * 16 + 4 * (lane >> 3)) = words[tt];
      if (lane == 0) xsf[r * (size_t)(L >> 5) + grp] = (uint8_t)sf[tt];
    }
  }
}

template <int NMAX, int PH, int KS, bool ONE>
cudaError_t launch_tc_n(const Maps& mp, FArgs f, cudaStream_t s, bool pdl) {
  static int configured[64] = {0};
  constexpr size_t smem = Lay<NMAX, PH == 0 ? 2 : 1, KS, ONE ? 8 : NMAX>::kSmemBytes;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_moe_tc<NMAX, PH, KS, ONE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  f.KC /= KS;  // units of KS chunks per tile
  return launch_kernel(k_moe_tc<NMAX, PH, KS, ONE>, dim3(tc_grid_size()), dim3(kThreads), smem,
                       s, pdl, mp, f);
}

// Each phase is its own kernel (a launch holds only its phase's code, and a single routed
// token's kernels hold only its in-kernel routing); the second GEMM takes two 512-chunks per
// unit when its reduction (f.KC chunks) divides evenly.
template <int NMAX, bool ONE>
cudaError_t launch_tc_phase(const Maps& mp, const FArgs& f, cudaStream_t s, bool pdl) {
  if (f.ph == 0) return launch_tc_n<NMAX, 0, 1, ONE>(mp, f, s, pdl);
  if (f.KC % 2 == 0) return launch_tc_n<NMAX, 1, 2, ONE>(mp, f, s, pdl);
  return launch_tc_n<NMAX, 1, 1, ONE>(mp, f, s, pdl);
}
// Batches of up to 4 tokens have at most 4 tokens per expert: 16-row activation tiles.
cudaError_t launch_tc(const Maps& mp, const FArgs& f, int T, cudaStream_t s, bool pdl) {
  if (f.route_one) return launch_tc_phase<16, true>(mp, f, s, pdl);  // one token
  // one or two tokens (their terms fill at most 16 MMA columns); batches of 3 tokens or more
  // take the large-batch kernels (moe_wide.cu), which run on every shape this path takes
  if (T * kTerms > 16) return cudaErrorInvalidValue;
  return launch_tc_phase<16, false>(mp, f, s, pdl);
}

}  // namespace

bool tc_path_supported(int L, int I) { return L % kKStage == 0 && I % kKStage == 0; }

int tc_grid() { return tc_grid_size(); }

int tc_npart(int T) { return T < kTokTile ? T : kTokTile; }  // tokens per tile, at most

size_t tc_part_floats(int T) { return (size_t)kTcMaxGrid * 3 * tc_npart(T) * kRowsTile; }

cudaError_t launch_split_x(const uint16_t* x, int T, int L, int k, int E, const int32_t* idx,
                           const BucketOut& b, uint8_t* xq, uint8_t* xsf, cudaStream_t s,
                           bool pdl) {
  return launch_kernel(k_split_x, dim3(T, L / kKStage), dim3(512), 0, s, pdl, x, L, k, E, idx,
                       static_cast<const int32_t*>(b.inv), xq, xsf);
}

cudaError_t launch_tc_experts(const ExpertPtrs& w, int L, int I, int E, int T, int k,
                              const uint8_t* xq, const uint8_t* xsf, const BucketOut& b,
                              uint8_t* act_q, uint8_t* act_sf, int act_kind, float b1, float b2,
                              const float* gate, float* ybuf, float* part, int32_t* status,
                              cudaStream_t s, bool pdl, void (*between)(cudaStream_t),
                              const RouteOne* ro) {
  // activation boxes: 8 rows for one routed token (its 4 term rows), else 16
  const uint32_t brows = ro ? 8 : 16;
  const uint64_t P4 = (uint64_t)T * k * kTerms;
  Maps m0, m1;
  if (!make_map_2d(&m0.m[0], w.w1p, L / 2, (uint64_t)E * I, 128, 128, true) ||
      !make_map_2d(&m0.m[1], w.w1s, L / 32, (uint64_t)E * I, 16, 128, false) ||
      !make_map_2d(&m0.m[2], w.w3p, L / 2, (uint64_t)E * I, 128, 128, true) ||
      !make_map_2d(&m0.m[3], w.w3s, L / 32, (uint64_t)E * I, 16, 128, false) ||
      !make_map_2d(&m0.m[4], xq, L / 2, P4, 128, brows, true) ||
      !make_map_2d(&m0.m[5], xsf, L / 32, P4, 16, brows, false) ||
      !make_map_2d(&m1.m[0], w.w2p, I / 2, (uint64_t)E * L, 128, 128, true) ||
      !make_map_2d(&m1.m[1], w.w2s, I / 32, (uint64_t)E * L, 16, 128, false) ||
      !make_map_2d(&m1.m[4], act_q, I / 2, P4, 128, brows, true) ||
      !make_map_2d(&m1.m[5], act_sf, I / 32, P4, 16, brows, false))
    return cudaErrorInvalidValue;
  m1.m[2] = m1.m[0];
  m1.m[3] = m1.m[1];
  // unit counts stay below 2^31 (32-bit range arithmetic in the kernel)
  const uint64_t groups = (uint64_t)T * k / kTokTile + E + 1;
  if (groups * ((L + kRowsTile - 1) / kRowsTile) * (L / kKStage) >= (1ull << 31) ||
      groups * ((I + kRowsTile - 1) / kRowsTile) * (L / kKStage) >= (1ull << 31) ||
      groups * ((L + kRowsTile - 1) / kRowsTile) * (I / kKStage) >= (1ull << 31))
    return cudaErrorInvalidValue;
  FArgs f{};
  f.k = k; f.L = L; f.I = I; f.act_kind = act_kind; f.b1 = b1; f.b2 = b2;
  f.meta = b.meta; f.perm = b.perm; f.tiles = b.tiles; f.nbase = b.ntile_base;
  f.act_q = act_q; f.act_sf = act_sf; f.gate = gate; f.ybuf = ybuf;
  f.part = part; f.npart = tc_npart(T);
  f.status = status;
  f.flag_polls = flag_wait_polls();
  if (ro) {
    f.route_one = 1;
    f.logits = ro->logits; f.bias = ro->bias; f.E = E;
    f.renorm = ro->renorm; f.routed_scale = ro->routed_scale;
    f.idx_out = ro->idx; f.gate_out = ro->gate; f.gap_out = ro->gap;
    f.route_words = reinterpret_cast<unsigned long long*>(b.flags + kTcRouteTable);
    f.y = ro->y; f.ycount = b.flags + kTcYCount;
  }
  // phase 0 (w1, w3), then phase 1 (w2): the second launch reads what the first wrote, across
  // the kernel boundary (its CTAs wait in griddepcontrol.wait until the first has completed)
  f.ph = 0;
  f.one_token = T == 1;
  f.KC = L / kKStage; f.RT = (I + kRowsTile - 1) / kRowsTile; f.R = I;
  f.flags = b.flags;
  cudaError_t e = launch_tc(m0, f, T, s, pdl);
  if (e != cudaSuccess) return e;
  if (between) between(s);
  f.ph = 1;
  f.one_token = 0;
  f.KC = I / kKStage; f.RT = (L + kRowsTile - 1) / kRowsTile; f.R = L;
  f.flags = b.flags + kTcMaxGrid;
  return launch_tc(m1, f, T, s, true);
}

}  // namespace k3
