/*
 * k3moe.h -- C ABI of the MXFP4 routed-expert MoE layer on one GB300 (sm_103a).
 *
 * The layer (Kimi-K3 shape) is the one stated by the "kimi-k3-in-c" README, Part II
 * section 9 "Picking 16 experts of 896" (router and per-token MoE), with experts stored as
 * MXFP4 as in Part II section 4 "Reduction one: the experts already ship at half a byte"
 * and the tensor shapes of "K3_ARTIFACT_AUDIT" (llm-atlas) section 4.3:
 *
 *   logit[t][e] = sum_i h[t][i] * Wr[e][i]                 router GEMV (bf16 in, fp32 sum)
 *   sc = sigmoid(logit); ch = sc + bias[e]                 bias steers selection only
 *   idx[t][0..k) = top-k of ch, descending; a tie goes to the lower expert index
 *   gate[t][j] = routed_scale * sc[idx_j] / sum_j sc[idx_j]      (renorm on)
 *   y[t] = sum_j gate[t][j] * W2[e_j] act(W1[e_j] x[t], W3[e_j] x[t])
 *   MXFP4 weight w = E2M1[nibble] * 2^(scale - 127), one E8M0 scale per 32 consecutive
 *   weights of a row, low nibble = even column, scale byte 255 -> the group is zero.
 *   act = SwiGLU: silu(g) * u   (or SiTU-GLU, README section 9, when selected)
 *
 * Conventions for every entry point:
 *   - Device pointers unless stated otherwise.  The caller owns every buffer.  No entry
 *     point allocates device or host memory; scratch comes from the caller's workspace
 *     `ws` of at least k3moe_workspace_size() bytes (device memory, 256-byte aligned).
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *     stream) and the call returns after enqueueing; results are ready when the stream
 *     reaches that point.  k3moe_layer_host is the exception: it synchronises the stream
 *     (k3moe_layer_host_async does so only when its host buffers are not all mapped).
 *   - T == 0 is a no-op that returns K3MOE_OK once the configuration is valid (empty
 *     tensors may carry NULL pointers).
 *   - Host-side argument checks run first.  On any failure the call returns a non-zero
 *     k3moe_status and enqueues nothing ("refuse, never guess": README Part II section 2).
 *   - Device-side anomalies are counted into an optional device status block
 *     (int32 status[4]): [0] assignments skipped because their expert index was out of
 *     range, [1] bounded waits that ran out, [2..3] reserved.  The library only adds to
 *     it (atomically); the caller zeroes it.  This follows the README's "counted, never
 *     silent" expert-drop rule (Part II section 9).
 *   - Pointers to bf16/fp32 tensors and to expert bytes must be 16-byte aligned.
 *   - Row-major, contiguous tensors throughout.
 *
 * Thread safety: calls on different streams with disjoint workspaces may run
 * concurrently.  Two calls that share a workspace must be ordered on the GPU.
 */
#ifndef K3MOE_H
#define K3MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define K3MOE_ABI_VERSION 1

typedef enum k3moe_status {
    K3MOE_OK = 0,
    K3MOE_ERR_INVALID = 1,     /* null pointer, negative size, k > E, bad enum value     */
    K3MOE_ERR_UNSUPPORTED = 2, /* a shape the kernels do not handle (see k3moe_cfg)      */
    K3MOE_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned                       */
    K3MOE_ERR_WORKSPACE = 4,   /* ws is NULL/misaligned or smaller than required         */
    K3MOE_ERR_CUDA = 5,        /* a CUDA launch or copy failed                           */
    K3MOE_ERR_TIMEOUT = 6,     /* (device status only) a bounded wait ran out            */
    K3MOE_ERR_DROPPED = 7,     /* (device status only) expert index out of range         */
    K3MOE_ERR_TOO_LARGE = 8    /* request exceeds the library's static scratch capacity  */
} k3moe_status;

typedef enum k3moe_act {
    K3MOE_ACT_SWIGLU = 0, /* act = silu(g) * u                                            */
    K3MOE_ACT_SITU = 1    /* act = b1*tanh(g/b1)*sigmoid(g) * b2*tanh(u/b2)  (README s.9) */
} k3moe_act;

/* Layer configuration; every field is required.  Supported: 1 <= topk <= min(E, 32),
 * 1 <= n_experts <= 1024, group == 32, hidden % 8 == 0, latent and inter multiples of 32
 * with latent <= 4096 and inter <= 4096.  Kimi K3: 7168, 896, 16, 3584, 3072, 32. */
typedef struct k3moe_cfg {
    int32_t hidden;       /* router input width H                                     */
    int32_t n_experts;    /* E                                                        */
    int32_t topk;         /* k                                                        */
    int32_t latent;       /* L: expert input / output width                           */
    int32_t inter;        /* I: expert intermediate width                             */
    int32_t group;        /* MX group size (must be 32)                               */
    int32_t renorm;       /* 1: gates renormalised over the chosen k; 0: not          */
    float routed_scale;   /* gates are multiplied by this (2.5 in the K3 workloads)   */
    int32_t act;          /* k3moe_act                                                */
    float situ_b1;        /* SiTU caps (4.0, 25.0); ignored for SwiGLU                */
    float situ_b2;
} k3moe_cfg;

/* The stacked expert tensors of one layer, checkpoint row layout (device memory):
 *   w1_packed, w3_packed: uint8 [E][inter][latent/2]    nibble pairs, low = even column
 *   w1_scale,  w3_scale:  uint8 [E][inter][latent/32]   E8M0
 *   w2_packed:            uint8 [E][latent][inter/2]
 *   w2_scale:             uint8 [E][latent][inter/32]
 * For Kimi K3 that is 17,547,264 bytes per expert (audit section 4.3). */
typedef struct k3moe_experts {
    const uint8_t *w1_packed, *w1_scale;
    const uint8_t *w3_packed, *w3_scale;
    const uint8_t *w2_packed, *w2_scale;
} k3moe_experts;

/* Bytes of device workspace needed by k3moe_route / k3moe_experts_mxfp4 / k3moe_layer
 * for T tokens (k3moe_layer_host needs k3moe_workspace_size_host).  Returns K3MOE_OK and
 * writes *bytes, or an error for an unsupported configuration. */
int k3moe_workspace_size(const k3moe_cfg *cfg, int32_t T, size_t *bytes);

/* Router for T tokens (README Part II section 9, the k3_router statement).
 *   h:    bf16 [T][hidden]          router input
 *   wr:   bf16 [E][hidden]          router weight
 *   bias: fp32 [E] or NULL          correction bias, added for selection only
 *   idx:  int32 [T][k]  (out)       chosen experts, descending selection score; ties ->
 *                                   lower index
 *   gate: fp32 [T][k]   (out)       combine weights from the unbiased sigmoid scores
 *   gap:  fp32 [T] or NULL (out)    k-th minus (k+1)-th selection score (+inf if k == E)
 * Scores are fp32 sigmoids of fp32-accumulated bf16 dot products. */
int k3moe_route(const k3moe_cfg *cfg, const void *h, const void *wr, const float *bias,
                int32_t T, int32_t *idx, float *gate, float *gap, void *ws, size_t ws_bytes,
                void *stream);

/* The routed-expert sum for T tokens given a routing (README Part II section 9, step 3):
 *   y[t] = sum_j gate[t][j] * W2[e] act(W1[e] x[t], W3[e] x[t]),  e = idx[t][j].
 *   experts: the layer's expert tensors (struct in host memory, pointers to device memory)
 *   x:    bf16 [T][latent]          expert input
 *   idx:  int32 [T][k], gate: fp32 [T][k]
 *   y:    fp32 [T][latent] (out)    fully overwritten (not accumulated into)
 *   status: int32[4] device status block or NULL.  An index outside [0, E) skips that
 *   assignment (its term is zero) and counts it in status[0].
 * Expert weights stay packed in HBM and are never expanded: the tensor-core path feeds the
 * checkpoint's E2M1 bytes and E8M0 scales straight to the block-scaled MMA (kind::mxf4);
 * widths that are not multiples of 512 take a CUDA-core path that decodes nibbles in
 * registers. */
int k3moe_experts_mxfp4(const k3moe_cfg *cfg, const k3moe_experts *experts, const void *x,
                        const int32_t *idx, const float *gate, int32_t T, float *y,
                        int32_t *status, void *ws, size_t ws_bytes, void *stream);

/* The routed-expert sum over one block of experts, for expert parallelism: the E experts
 * are split into contiguous blocks, one per device, and each device sums only the terms of
 * the experts it holds (README Part II section 9's per-token sum, partitioned by expert);
 * the devices' partial y then add up (an all-reduce) to the layer's y.
 *   experts: the block [e0, e1) only, stacked from expert e0 (local expert e - e0), layouts
 *            as in k3moe_experts; cfg->n_experts is the layer's E (0 <= e0 < e1 <= E)
 *   idx, gate: the routing over all E experts (as k3moe_route writes it)
 *   y:    fp32 [T][latent] (out), fully overwritten: sum over the assignments whose expert
 *         is in [e0, e1); a token with none of them gets a zero row
 *   An index in [0, E) outside the block is another device's and is skipped silently; an
 *   index outside [0, E) is skipped and counted in status[0] (on every device).
 *   ws:   at least k3moe_workspace_size(cfg, T) bytes.  Other arguments as k3moe_experts_mxfp4. */
int k3moe_experts_mxfp4_range(const k3moe_cfg *cfg, const k3moe_experts *experts, int32_t e0,
                              int32_t e1, const void *x, const int32_t *idx, const float *gate,
                              int32_t T, float *y, int32_t *status, void *ws, size_t ws_bytes,
                              void *stream);

/* Router + routed-expert sum in one call (the layer).  idx, gate and gap are optional
 * outputs (NULL: kept in the workspace); other arguments as in the two calls above. */
int k3moe_layer(const k3moe_cfg *cfg, const void *h, const void *wr, const float *bias,
                const k3moe_experts *experts, const void *x, int32_t T, float *y,
                int32_t *idx, float *gate, float *gap, int32_t *status, void *ws,
                size_t ws_bytes, void *stream);

/* Bytes of device workspace for k3moe_layer_host with T tokens: the device workspace of
 * k3moe_layer plus staging room for h, x and y. */
int k3moe_workspace_size_host(const k3moe_cfg *cfg, int32_t T, size_t *bytes);

/* k3moe_layer with HOST input and output buffers: copies h (bf16 [T][hidden]) and x
 * (bf16 [T][latent]) from host memory into the workspace, runs the layer, copies y (fp32
 * [T][latent]) back to host memory, and synchronises the stream before returning.  The
 * routing stays in the workspace.  wr, bias, experts and status stay in device memory.
 * When h, x and y are all page-locked host memory mapped into the device's address space
 * (cudaHostAlloc'd or registered pinned buffers), the kernels read h and x and write y in
 * host memory directly (on a Grace-Blackwell node over NVLink-C2C) instead of staging them
 * through the workspace.
 * Host buffers should be page-locked: the library then records the first call with a given
 * set of arguments (configuration, T, every pointer, ws_bytes, stream) as a CUDA graph and
 * replays it for later calls with the same set (one launch instead of three copies and the
 * layer's launches; the buffers' contents are read at each replay).  Up to 16 such graphs are
 * kept per process, least recently used replaced; calls with pageable buffers, or while
 * phase events are set, run without a graph.  Returns K3MOE_ERR_CUDA if a copy, a launch or
 * the synchronisation fails. */
int k3moe_layer_host(const k3moe_cfg *cfg, const void *h_host, const void *wr,
                     const float *bias, const k3moe_experts *experts, const void *x_host,
                     int32_t T, float *y_host, int32_t *status, void *ws, size_t ws_bytes,
                     void *stream);

/* k3moe_layer_host without the final synchronisation, for a serving loop that keeps two calls
 * in flight (double-buffered host buffers): the call enqueues the layer on `stream` and
 * returns; y_host holds the result once the stream reaches that point (synchronise the stream
 * or an event recorded after the call).  The caller must not write h_host or x_host, nor read
 * y_host, until then.  It returns without waiting when h_host, x_host and y_host are all
 * page-locked host memory mapped into the device's address space: the layer's launches are
 * then enqueued as they are (no graph: programmatic dependent launch lets consecutive calls
 * on one stream overlap their first and last kernels), the kernels reading h and x and
 * writing y in host memory.  Otherwise it behaves like k3moe_layer_host (and synchronises).
 * Arguments and errors as k3moe_layer_host. */
int k3moe_layer_host_async(const k3moe_cfg *cfg, const void *h_host, const void *wr,
                           const float *bias, const k3moe_experts *experts, const void *x_host,
                           int32_t T, float *y_host, int32_t *status, void *ws, size_t ws_bytes,
                           void *stream);

/* One MXFP4 mat-vec on the GPU (README Part II section 4, the k3_matmul_mxfp4 statement):
 *   y[r] = sum_c W[r][c] x[c],  W = packed [rows][in/2] + scales [rows][in/32]
 *   x: bf16 [in]; y: fp32 [rows] (out).  in must be a multiple of 32. */
int k3moe_matvec_mxfp4(float *y, const void *x, const uint8_t *packed, const uint8_t *scales,
                       int32_t in, int32_t rows, int32_t group, void *stream);

/* Link between stacked layers: next-layer inputs from a layer output.
 *   y: fp32 [T][L]; x_out: bf16 [T][L] (out); h_out: bf16 [T][2L] or NULL (out).
 *   norm != 0: each token is RMS-normalised with unit weight, eps inside the square root
 *   (README Part II section 5), before rounding to bf16 (nearest even).  h_out is x_out
 *   tiled twice along the feature axis. */
int k3moe_stack_link(const float *y, int32_t T, int32_t L, int32_t norm, float eps,
                     void *x_out, void *h_out, void *stream);

/* The LatentMoE wrapper's dense tensors around the routed experts (README Part II section
 * 9, k3_moe).  Device pointers, bf16 row-major unless noted, each 16-byte aligned; the
 * caller owns them:
 *   down [latent][hidden]      z = down . h, the experts' latent input (rounded to bf16);
 *   up   [hidden][latent]      out = up . a, a = the routed sum after its RMSNorm;
 *   latent_norm_w fp32 [latent], or NULL for unit weight; latent_norm 1 applies the RMSNorm
 *   (sum of squares in fp32 by a fixed reduction tree, eps = rms_eps inside the square root,
 *   README section 5), 0 skips;
 *   sh1, sh3 [n_shared*inter][hidden] and sh2 [hidden][n_shared*inter]: the shared experts,
 *   on the full-width h, with the layer's activation, added unweighted; n_shared 0: none
 *   (the three pointers are then ignored). */
typedef struct k3moe_latent {
  const void *down, *up;
  const float *latent_norm_w;
  int32_t latent_norm;
  float rms_eps;
  int32_t n_shared;
  const void *sh1, *sh3, *sh2;
} k3moe_latent;

/* Device workspace bytes of k3moe_latent_layer for T tokens: k3moe_workspace_size's plus
 * the latent z, the routed sum and its norm, and the shared experts' activations. */
int k3moe_latent_workspace_size(const k3moe_cfg *cfg, const k3moe_latent *lat, int32_t T,
                                size_t *bytes);

/* The LatentMoE layer for T tokens (README Part II section 9, k3_moe), per token:
 *   route on h (idx, gate, gap as k3moe_layer: each may be NULL);
 *   z = bf16(down . h); acc = sum_j gate_j FFN_{idx_j}(z)  (the routed experts, as
 *   k3moe_layer with x = z);
 *   out = up . (latent_norm ? rmsnorm(acc) * latent_norm_w : acc)
 *         + sh2 . act(sh1 . h, sh3 . h).
 *   h: bf16 [T][hidden]; out: fp32 [T][hidden] (out, fully written); other arguments and
 *   errors as k3moe_layer.  T is at most 262140.  One token takes six launches on the
 *   stream (the three of k3moe_layer plus the two dense launches and the norm). */
int k3moe_latent_layer(const k3moe_cfg *cfg, const k3moe_latent *lat, const void *h,
                       const void *wr, const float *bias, const k3moe_experts *experts,
                       int32_t T, float *out, int32_t *idx, float *gate, float *gap,
                       int32_t *status, void *ws, size_t ws_bytes, void *stream);

/* k3moe_layer for callers that cannot allocate device memory.  No counterpart on the
 * pages: this is a deployment variant, not part of the method.
 *
 * Some callers cannot call cudaMalloc (or have no way to hand over a workspace): a host
 * framework whose allocator owns all device memory and forbids raw allocations, a plugin
 * that runs inside someone else's memory budget, or a latency-critical path where an
 * allocation could block or fail.  This entry point takes the same inputs and outputs as
 * k3moe_layer but no workspace: its scratch is one file-scope device array of
 * K3MOE_STATIC_SCRATCH_BYTES (16 MiB), which every GPU that loads the library holds until
 * the process exits.  It allocates nothing, on the device or the host.
 *
 *   - Capacity: a call whose k3moe_workspace_size(cfg, T) exceeds the array returns
 *     K3MOE_ERR_TOO_LARGE and enqueues nothing (Kimi K3 shape: up to 27 tokens).
 *   - Set-up: the first call on a device, with that device current, looks up the array's
 *     device address (cudaGetSymbolAddress) and caches it with the device's current
 *     context; make that first call before any stream capture begins.  A call that finds
 *     another context current (the old one was destroyed, e.g. by cudaDeviceReset) looks
 *     the address up again, so no stale address is used.
 *   - Sharing: all calls on a device share the one array and it keeps the previous call's
 *     contents.  Every scratch value a call reads is written earlier in the same call, so
 *     no clearing is needed between calls; but calls that overlap on the GPU (different streams, no ordering between
 *     them) race on the array and corrupt each other's results.  Order them on one stream.
 * Arguments, layouts and errors are those of k3moe_layer. */
#define K3MOE_STATIC_SCRATCH_BYTES (16u << 20)
int k3moe_layer_static_scratch(const k3moe_cfg *cfg, const void *h, const void *wr,
                               const float *bias, const k3moe_experts *experts, const void *x,
                               int32_t T, float *y, int32_t *idx, float *gate, float *gap,
                               int32_t *status, void *stream);

/* Per-phase timing hook for benchmarks.  events: n (== 6) cudaEvent_t handles (as void*)
 * created by the caller, or NULL to switch the hook off.  While set, every k3moe_layer and
 * k3moe_experts_mxfp4 call records, on its stream: [0] at entry, [1] after the router
 * logits (decode-sized batches run the top-k inside the next phase), [2] after the top-k,
 * bucketing and input preparation, [3] after GEMM1 (w1, w3, activation), [4] after GEMM2
 * (w2, gates), [5] after the combine.  Process-wide, not thread-safe;
 * recording breaks programmatic launch overlap between phases, so time throughput with
 * the hook off.  Returns K3MOE_ERR_INVALID if n != 6 with non-NULL events. */
int k3moe_set_phase_events(void *const *events, int32_t n);

/* Limit of the waits that cross CTAs: how many times a kernel polls a flag or routing word
 * that another CTA writes (the routing words of a one-token layer, the "part written" flags
 * of a tile that several CTAs share) before it gives up.  A wait that gives up counts one
 * timeout in status[1], its CTA stops its work and waits for its own copies and MMAs in
 * flight, and the kernel returns; results of that call are then incomplete, and later calls
 * are unaffected.  polls < 0 restores the default (4,194,304); 0 makes every such wait give
 * up at once (a way to exercise the timeout path without a fault).  Waits inside a CTA's
 * pipeline are not affected.  Process-wide; read when a call enqueues its launches (a
 * captured graph keeps the value it was captured with).  Returns K3MOE_ERR_INVALID if
 * polls > 4,294,967,295. */
int k3moe_set_flag_wait_polls(int64_t polls);

/* ---- Experts beyond HBM: a device cache over an expert store in host memory ------------
 *
 * README Part II section 12 "An LRU cache for the experts": the experts live in a large,
 * slower tier and a fixed number of slots in fast memory hold the recently used ones.  Here
 * the tier is page-locked host memory (on a Grace-Blackwell node the Grace memory, reached
 * over NVLink-C2C) and the slots are device memory laid out as a k3moe_experts of n_slots
 * experts, so that the expert kernels run on the slots unchanged.  A slot holds an expert,
 * is empty, or is in flight (reserved for an expert whose copy has been issued but not yet
 * published).  For one call the cache
 *   1. reserves: experts already resident are marked used; for each missing expert, in
 *      ascending expert order, an empty slot if there is one, else the least recently used
 *      slot that this call does not use and that is not in flight (its expert is evicted);
 *   2. reads: copies each reserved expert host -> device, in ascending expert order (the
 *      store's offset order);
 *   3. publishes: a slot whose copy was issued holds its expert from then on (stream order
 *      makes the data visible to the kernels that follow); a slot whose copy could not be
 *      issued goes back to empty.
 * One cache serves one layer's experts; calls on a cache must not overlap (the state is
 * host memory without locks).  The caller owns every array. */
#define K3MOE_SLOT_EMPTY (-1)
#define K3MOE_SLOT_INFLIGHT (-2)
typedef struct k3moe_expert_cache {
    int32_t n_experts;      /* E: experts in the host store                                 */
    int32_t n_slots;        /* C: device slots, 1 <= C <= E                                 */
    k3moe_experts host;     /* the E experts, page-locked host memory, checkpoint layout    */
    k3moe_experts slots;    /* room for C experts in device memory, the same layout: slot s
                               is expert s of these arrays                                  */
    int32_t *expert_of;     /* host [C]: expert in slot s, K3MOE_SLOT_EMPTY or _INFLIGHT    */
    int32_t *slot_of;       /* host [E]: slot holding expert e, or -1                       */
    uint64_t *used_at;      /* host [C]: the clock at the slot's last use                   */
    uint64_t clock;         /* advanced once per planned call                               */
} k3moe_expert_cache;

/* Empties every slot and resets the clock (host only, no CUDA call). */
int k3moe_cache_reset(k3moe_expert_cache *cache);

/* Step 1 for n expert indices (host memory, any order, repeats allowed): marks the resident
 * ones used, reserves slots for the missing ones (their slots become K3MOE_SLOT_INFLIGHT),
 * and writes slot_idx[i] = the slot of idx[i] (-1 for an index outside [0, E)) and the
 * copies to make, fetch_expert[j] -> fetch_slot[j] for j < *n_fetch, in ascending expert
 * order (both arrays: room for n_slots entries).  Host only, no CUDA call.  Returns
 * K3MOE_ERR_UNSUPPORTED, with the state unchanged, if the indices name more distinct
 * experts than there are slots. */
int k3moe_cache_plan(k3moe_expert_cache *cache, const int32_t *idx, int32_t n, int32_t *slot_idx,
                     int32_t *fetch_expert, int32_t *fetch_slot, int32_t *n_fetch);

/* Step 3: the first n_ok of the planned copies were issued (their slots now hold their
 * experts); the rest were not (their slots become empty). */
int k3moe_cache_publish(k3moe_expert_cache *cache, const int32_t *fetch_expert,
                        const int32_t *fetch_slot, int32_t n_fetch, int32_t n_ok);

/* Device workspace and host scratch of k3moe_layer_cached for T tokens. */
int k3moe_cache_workspace_size(const k3moe_cfg *cfg, int32_t T, size_t *bytes);
int k3moe_cache_host_scratch_size(const k3moe_cfg *cfg, int32_t T, int32_t n_slots, size_t *bytes);

/* The layer with its experts in the cache: routes the T tokens on the device (as
 * k3moe_route), reads the routing back to the host, plans, copies the missing experts from
 * the host store into their slots (by a kernel that reads the store where it is mapped page-
 * locked memory, over NVLink-C2C on a Grace-Blackwell node; otherwise one cudaMemcpyAsync per
 * tensor), publishes, and runs the
 * routed-expert sum on the slots (as k3moe_experts_mxfp4 with the routing mapped to slots);
 * synchronises the stream before returning.  y equals k3moe_layer's for the same inputs
 * bit for bit when the batch takes the large-batch expert kernels (T >= 3 with latent and
 * inter multiples of 512: each assignment's result there does not depend on which others
 * share its tile); otherwise the two agree within rounding (the split of a tile's reduction
 * across CTAs follows the expert numbering, which the slots change).  Needs topk <= n_slots.
 *   cache: cache->n_experts == cfg->n_experts; the store and the slots as described above
 *   h, wr, bias, x, y, status: as in k3moe_layer (device memory)
 *   ws: device, at least k3moe_cache_workspace_size bytes; host_scratch: host memory (page-
 *       locked for the read-back to be asynchronous), at least k3moe_cache_host_scratch_size
 *   n_fetched: optional (out), the experts copied by this call
 * Returns K3MOE_ERR_UNSUPPORTED if the call's routing names more distinct experts than there
 * are slots (nothing is computed; y is left as it was), K3MOE_ERR_CUDA if a copy or launch
 * fails (slots whose copies were not issued are left empty). */
int k3moe_layer_cached(const k3moe_cfg *cfg, k3moe_expert_cache *cache, const void *h,
                       const void *wr, const float *bias, const void *x, int32_t T, float *y,
                       int32_t *status, void *ws, size_t ws_bytes, void *host_scratch,
                       size_t host_scratch_bytes, int32_t *n_fetched, void *stream);

/* Number of kernels the library launched through the entry points above since load
 * (host counter; for launch accounting in benchmarks). */
int64_t k3moe_launch_count(void);

/* The last CUDA failure seen by an entry point on the calling thread: the call that failed
 * and CUDA's description of the error (for example a refused launch), or "" if none.  The
 * string stays valid until the thread's next failing call. */
const char *k3moe_last_error(void);

/* Static string for a status code. */
const char *k3moe_strerror(int status);

/* K3MOE_ABI_VERSION of the loaded library. */
int32_t k3moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* K3MOE_H */
