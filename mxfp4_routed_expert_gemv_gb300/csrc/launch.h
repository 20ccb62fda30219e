// launch.h -- internal launch helpers and the launchers each kernel file exports.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace k3 {

// Kernels launched through the library since load (host-side count).
extern std::atomic<int64_t> g_launches;

// Launch `kern` with an optional programmatic-dependent-launch attribute, so that the
// kernel's CTAs may be scheduled while the previous kernel on the stream drains; every
// kernel here calls griddepcontrol.wait before it reads what earlier kernels wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Multiprocessor count of the current device (cached per device).
int sm_count();

// Polls a kernel's wait on a flag or routing word written by another CTA makes before it
// gives up and counts a timeout (k3moe_set_flag_wait_polls; kWaitPolls unless changed).
uint32_t flag_wait_polls();

// router.cu
// With xq set (T == 1 only) the launch also writes x's kTerms MXFP4 terms into rows
// 0 .. kTerms-1 of xq / xsf.
// part: [router_splits(T, E, H)][T][E] floats of partial logits when that is > 1 (the
// top-k launch sums them into logits first).
cudaError_t launch_router_logits(const uint16_t* h, const uint16_t* wr, int T, int E, int H,
                                 float* logits, cudaStream_t s, bool pdl,
                                 const uint16_t* x = nullptr, int L = 0, uint8_t* xq = nullptr,
                                 uint8_t* xsf = nullptr, int32_t* zero = nullptr,
                                 int nzero = 0, int32_t* status = nullptr, float* part = nullptr);
// From this many tokens the router logits run as a tensor-core GEMM (router.cu), when the
// hidden width allows (router_tc_supported); up to kRouterSplitMaxTokens its reduction is
// split across CTAs (router_splits ranges).
constexpr int kRouterTcMinTokens = 3;
constexpr int kRouterSplitMaxTokens = 1024;
inline bool router_tc_supported(int H) { return H >= 64 && H % 8 == 0; }
int router_splits(int T, int E, int H);
// logits[t][e] = sum over z of part[z][t][e] in z order, for e = i0, i0 + step, ... < E
// (The loads of eight ranges are issued before their sums, which stay in range order: the
// partials come from L2, and one dependent load per range would chain ks latencies.)
__device__ __forceinline__ void sum_router_parts(const float* part, int ks, int T, int E, int t,
                                                 float* logits, int i0, int step) {
  const size_t zs = (size_t)T * E;
  for (int e = i0; e < E; e += step) {
    const float* pe = part + (size_t)t * E + e;
    float acc = 0.f;
    int z = 0;
    for (; z + 8 <= ks; z += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __ldcg(pe + (size_t)(z + j) * zs);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc += v[j];
    }
    for (; z < ks; ++z) acc += __ldcg(pe + (size_t)z * zs);
    logits[(size_t)t * E + e] = acc;
  }
}
// The same for one token with a whole block, EPT experts per thread (E <= EPT blockDim.x):
// the loads of all the thread's experts for eight ranges are in flight together.
template <int EPT>
__device__ __forceinline__ void sum_router_parts_block(const float* part, int ks, int T, int E,
                                                       int t, float* logits) {
  const size_t zs = (size_t)T * E;
  const float* pt = part + (size_t)t * E;
  float acc[EPT];
  bool on[EPT];
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    acc[j] = 0.f;
    on[j] = threadIdx.x + j * blockDim.x < (unsigned)E;
  }
  for (int z = 0; z < ks; z += 8) {
    float v[EPT][8];
#pragma unroll
    for (int j = 0; j < EPT; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        v[j][i] = (on[j] && z + i < ks) ? __ldcg(pt + (size_t)(z + i) * zs + threadIdx.x + j * blockDim.x) : 0.f;
#pragma unroll
    for (int j = 0; j < EPT; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (z + i < ks) acc[j] += v[j][i];
  }
#pragma unroll
  for (int j = 0; j < EPT; ++j)
    if (on[j]) logits[(size_t)t * E + threadIdx.x + j * blockDim.x] = acc[j];
}
cudaError_t launch_topk(float* logits, const float* part, int ks, const float* bias, int T, int E,
                        int k, int renorm, float routed_scale, int32_t* idx, float* gate,
                        float* gap, cudaStream_t s, bool pdl);

// Tensor-core expert path (moe_tc.cu): tokens per tile, and the largest grid it launches.
constexpr int kTcTokTile = 16;
// Large batches (moe_wide.cu): positions of one expert per tile, and the batch size from
// which the layer takes that path; batches from kRowsMinTokens below that take the same
// kernels with the activation terms as MMA rows, kTcRowTok positions per tile.
constexpr int kTcWideTok = 128;
constexpr int kWideMinTokens = 256;
constexpr int kTcRowTok = 32;
constexpr int kRowsMinTokens = 3;
constexpr int kTcMaxGrid = 160;
// Flags of the tensor-core path, zeroed before each call: [0, kTcMaxGrid) parts of the first
// GEMM's shared tiles written, [kTcMaxGrid, 2 kTcMaxGrid) the same for the second GEMM.
constexpr int kTcFlags = 2 * kTcMaxGrid;
// One routed token: after the flags, per 128-row tile of y, the slots written so far (the
// second GEMM sums the token's slots into y where the count completes; L <= 4096).
constexpr int kTcYCount = kTcFlags;
// Then (8-byte aligned) the single-token routing as one 64-bit word per chosen expert, in
// ascending expert order: gate bits << 32 | 1 << 31 | choice index << 16 | expert.  A word
// is its own ready flag (zeroed words have bit 31 clear).
constexpr int kTcRouteTable = kTcYCount + 4096 / 128;
static_assert(kTcRouteTable % 2 == 0, "route table alignment");
constexpr int kTcFlagWords = kTcRouteTable + 2 * 32;

// bucket.cu
// An expert index that names an expert held by another device (expert-range calls): skipped
// without counting a drop.
constexpr int32_t kRemoteExpert = INT32_MIN;
// idx_local[a] = idx[a] - e0 for e0 <= idx[a] < e1, kRemoteExpert for another index in
// [0, E), and -1 (a counted drop) outside [0, E).
cudaError_t launch_localize_idx(const int32_t* idx, int n, int E, int e0, int e1,
                                int32_t* idx_local, cudaStream_t s, bool pdl);
struct BucketOut {
  int32_t* counts;      // [E]
  int32_t* offsets;     // [E+1]
  int32_t* perm;        // [T*k]  assignment ids sorted by (expert, token)
  int32_t* active;      // [E]    expert ids with at least one token, ascending
  int32_t* seg_off;     // [E]    perm offset of each active expert's tokens
  int32_t* seg_cnt;     // [E]    number of tokens of each active expert
  int32_t* meta;        // [16]   [0] active experts, [1] valid assignments, [2] token groups,
                        //        [3] large-batch token groups, [4] kTcRowTok token groups
  int32_t* chunk_base;  // [E][nchunks] scratch of the multi-block path
  int32_t* nvalid;      // [T]    valid assignments per token
  int32_t* inv;         // [T*k]  perm position of each valid assignment id
  int32_t* ntile_base;  // [E+1]  tensor-core tiles (kTcTokTile tokens) before each active expert
  int32_t* flags;       // [kTcFlagWords] tensor-core path flags and counts (zeroed per call)
  int4* tiles;          // [P/16 + E + 1] per token group: expert, first position, tokens, 0
  int32_t* nbase_w;     // [E+1]  large-batch groups (kTcWideTok tokens) before each active expert
  int4* tiles_w;        // [P/kTcWideTok + E + 1] the same table for groups of kTcWideTok tokens
  int32_t* nbase_r;     // [E+1]  the same for groups of kTcRowTok tokens
  int4* tiles_r;        // [P/kTcRowTok + E + 1]
  // Large-batch expert GEMMs (moe_wide.cu): when wdesc is set, the preparation also writes
  // their tile descriptors, one per (token group, row block) of each GEMM: wrb0 / wrb1 row
  // blocks, the second GEMM's at wdesc + wdesc1; groups of kTcRowTok (wmode 2) or
  // kTcWideTok (wmode 1) tokens.
  int4* wdesc;
  int32_t wdesc1, wrb0, wrb1, wmode;
};

// Everything the per-call preparation touches.  logits == nullptr: idx/gate come from the
// caller (no top-k); otherwise the fused decode-size kernel also runs the router's top-k.
struct PrepArgs {
  const float* logits;
  const float* bias;
  int E, k, renorm;
  float routed_scale;
  int32_t* idx;
  float* gate;
  float* gap;
  int T, L;
  const uint16_t* x;
  __half* x16;
  int32_t* xexp;
  BucketOut b;
  float* y;
  int32_t* status;
};
int bucket_chunks(int T);
bool prep_is_fused(int T);
cudaError_t launch_prep(const PrepArgs& p, cudaStream_t s, bool pdl);

// gemv.cu
struct ExpertPtrs {
  const uint8_t *w1p, *w1s, *w3p, *w3s, *w2p, *w2s;
};
cudaError_t launch_prep_x(const uint16_t* x, int T, int L, __half* x16, int32_t* xexp,
                          cudaStream_t s, bool pdl);
cudaError_t launch_matvec(float* y, const uint16_t* x, const uint8_t* packed,
                          const uint8_t* scales, int in, int rows, cudaStream_t s);

// experts.cu
cudaError_t launch_gemm1(const ExpertPtrs& w, int L, int I, int E, int T, int k,
                         const __half* x16, const int32_t* xexp, const BucketOut& b,
                         float* act, int act_kind, float b1, float b2, int32_t* status,
                         cudaStream_t s, bool pdl);
cudaError_t launch_gemm2(const ExpertPtrs& w, int L, int I, int E, int T, int k,
                         const float* act, const float* gate, const BucketOut& b, float* ybuf,
                         int32_t* status, cudaStream_t s, bool pdl);
cudaError_t launch_combine(const float* ybuf, const int32_t* idx, int T, int k, int E, int L,
                           float* y, cudaStream_t s, bool pdl);

// moe_tc.cu
bool tc_path_supported(int L, int I);
int tc_grid();
int tc_npart(int T);
size_t tc_part_floats(int T);
cudaError_t launch_split_x(const uint16_t* x, int T, int L, int k, int E, const int32_t* idx,
                           const BucketOut& b, uint8_t* xq, uint8_t* xsf, cudaStream_t s,
                           bool pdl);
// One token routed inside the expert GEMMs (no preparation launch): the router's logits and
// the top-k parameters; CTA 0 of the first GEMM publishes idx / gate / gap (and the tile
// table, in BucketOut's tiles / perm, for the second GEMM).  Needs E <= 1056, k <= 31 or k == E.
struct RouteOne {
  const float *logits, *bias;
  int renorm;
  float routed_scale;
  int32_t* idx;
  float *gate, *gap;
  float* y;  // [L]: the second GEMM sums the slots here (no combine launch)
};
// moe_wide.cu: the expert GEMMs of a batch (positions as the MMA's M, 256 weight rows as N);
// reads the per-position x terms (launch_split_x_wide) and the group table of its tile size:
// rows == false, 128 positions per tile with the terms folded into the reduction (large
// batches); rows == true, 32 positions x 4 terms as the 128 MMA rows (small batches).
bool wide_path_supported(int L, int I);
// x into per-position terms for the large-batch path (scales in its stage-major layout)
cudaError_t launch_split_x_wide(const uint16_t* x, int T, int L, int k, int E, const int32_t* idx,
                                const BucketOut& b, uint8_t* xq, uint8_t* xsf, cudaStream_t s,
                                bool pdl);
// Tile descriptors of both expert GEMMs (workspace int4 entries) for any call of up to T
// tokens; wide_desc_setup points b at them for a call of T tokens (the preparation writes them).
size_t wide_desc_count(int L, int I, int E, int T, int k);
void wide_desc_setup(BucketOut& b, int4* desc, int L, int I, int E, int T, int k, bool rows);
cudaError_t launch_wide_experts(const ExpertPtrs& w, int L, int I, int E, int T, int k, bool rows,
                                const uint8_t* xq, const uint8_t* xsf, const BucketOut& b,
                                uint8_t* act_q, uint8_t* act_sf, int act_kind, float b1, float b2,
                                const float* gate, float* ybuf, int32_t* status, cudaStream_t s,
                                void (*between)(cudaStream_t));
cudaError_t launch_tc_experts(const ExpertPtrs& w, int L, int I, int E, int T, int k,
                              const uint8_t* xq, const uint8_t* xsf, const BucketOut& b,
                              uint8_t* act_q, uint8_t* act_sf, int act_kind, float b1, float b2,
                              const float* gate, float* ybuf, float* part, int32_t* status,
                              cudaStream_t s, bool pdl, void (*between)(cudaStream_t),
                              const RouteOne* ro = nullptr);

// dense.cu (the LatentMoE wrapper): z = bf16(down . h) and act = activation(sh1 . h,
// sh3 . h); yn = the RMSNorm of y (or y); out = up . yn + sh2 . act.
cudaError_t launch_dense_in(const uint16_t* h, int T, int H, const uint16_t* down, int L,
                            uint16_t* z, const uint16_t* sh1, const uint16_t* sh3, int SI,
                            float* act, int act_kind, float b1, float b2, cudaStream_t s,
                            bool pdl);
cudaError_t launch_latent_norm(const float* y, int T, int L, int norm, const float* w, float eps,
                               float* yn, cudaStream_t s, bool pdl);
cudaError_t launch_dense_out(const float* yn, int T, int L, const uint16_t* up, int H,
                             const float* act, const uint16_t* sh2, int SI, float* out,
                             cudaStream_t s, bool pdl);

// stack.cu
cudaError_t launch_stack_link(const float* y, int T, int L, int norm, float eps, uint16_t* x_out,
                              uint16_t* h_out, cudaStream_t s);

}  // namespace k3
