// abi.cu -- the extern "C" entry points of libk3moe.so (declared in include/k3moe.h):
// argument validation, workspace carving and the launch sequence on the caller's stream.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>

#include "launch.h"
#include "mxq.cuh"

namespace k3 {

std::atomic<int64_t> g_launches{0};
std::atomic<uint32_t> g_flag_polls{kWaitPolls};

uint32_t flag_wait_polls() { return g_flag_polls.load(std::memory_order_relaxed); }

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < 64) cached[dev] = n;
  return n;
}

namespace {

constexpr int32_t kMaxTokens = 1 << 18;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_cfg(const k3moe_cfg* c) {
  if (!c) return K3MOE_ERR_INVALID;
  if (c->hidden <= 0 || c->n_experts <= 0 || c->topk <= 0 || c->latent <= 0 || c->inter <= 0)
    return K3MOE_ERR_INVALID;
  if (c->topk > c->n_experts) return K3MOE_ERR_INVALID;
  if (c->renorm != 0 && c->renorm != 1) return K3MOE_ERR_INVALID;
  if (c->act != K3MOE_ACT_SWIGLU && c->act != K3MOE_ACT_SITU) return K3MOE_ERR_INVALID;
  if (c->act == K3MOE_ACT_SITU && !(c->situ_b1 > 0.f && c->situ_b2 > 0.f)) return K3MOE_ERR_INVALID;
  if (c->group != kGroup) return K3MOE_ERR_UNSUPPORTED;
  if (c->topk > kMaxTopk || c->n_experts > kMaxExperts) return K3MOE_ERR_UNSUPPORTED;
  if (c->hidden % 8 != 0) return K3MOE_ERR_UNSUPPORTED;
  if (c->latent % 32 != 0 || c->inter % 32 != 0) return K3MOE_ERR_UNSUPPORTED;
  if (c->latent > 4096 || c->inter > 4096) return K3MOE_ERR_UNSUPPORTED;
  return K3MOE_OK;
}

// Device workspace layout for T tokens (every region 256-byte aligned).
struct Workspace {
  float* logits;     // [T][E]
  float* rpart;      // [router splits][T][E] partial logits (split-K tensor-core router)
  int32_t* idx;      // [T][k]
  float* gate;       // [T][k]
  float* gap;        // [T]
  BucketOut b;
  bool tc;           // tensor-core expert path (shapes it tiles) or the CUDA-core GEMV
  __half* x16;       // [T][L]                  (GEMV path)
  int32_t* xexp;     // [T]                     (GEMV path)
  float* act;        // [T*k][I]                (GEMV path)
  uint8_t* xq;       // [T*k*kTerms][L/2]       (tensor-core path: x as MXFP4 terms)
  uint8_t* xsf;      // [T*k*kTerms][L/32]
  uint8_t* aq;       // [T*k*kTerms][I/2]       (tensor-core path: act as MXFP4 terms)
  uint8_t* asf;      // [T*k*kTerms][I/32]
  float* part;       // split-tile partial sums (tensor-core path)
  int4* wdesc;       // tile descriptors of the large-batch expert GEMMs
  float* ybuf;       // [T*k][L]
  uint16_t* h_stage; // [T][H]  (host variant only)
  uint16_t* x_stage; // [T][L]
  float* y_stage;    // [T][L]
};

struct Carver {
  uint8_t* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t count) {
    off = (off + 255) & ~size_t(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

size_t carve(const k3moe_cfg* c, int32_t T, void* base, bool host_stage, Workspace* w) {
  Carver cv{static_cast<uint8_t*>(base)};
  const size_t E = c->n_experts, K = c->topk, L = c->latent, I = c->inter, H = c->hidden;
  const size_t Tt = (size_t)std::max(T, 1);
  const size_t P = Tt * K;
  Workspace t{};
  t.logits = cv.take<float>(Tt * E);
  {
    const int ks = router_splits((int)Tt, (int)E, (int)H);
    t.rpart = ks > 1 ? cv.take<float>((size_t)ks * Tt * E) : nullptr;
  }
  t.idx = cv.take<int32_t>(P);
  t.gate = cv.take<float>(P);
  t.gap = cv.take<float>(Tt);
  t.b.counts = cv.take<int32_t>(E);
  t.b.offsets = cv.take<int32_t>(E + 1);
  t.b.perm = cv.take<int32_t>(P);
  t.b.active = cv.take<int32_t>(E);
  t.b.seg_off = cv.take<int32_t>(E);
  t.b.seg_cnt = cv.take<int32_t>(E);
  t.b.meta = cv.take<int32_t>(16);
  t.b.chunk_base = cv.take<int32_t>(E * (size_t)bucket_chunks((int)Tt));
  t.b.nvalid = cv.take<int32_t>(Tt);
  t.b.inv = cv.take<int32_t>(P);
  t.b.ntile_base = cv.take<int32_t>(E + 1);
  t.b.flags = cv.take<int32_t>(kTcFlagWords);
  t.b.tiles = cv.take<int4>((P + kTcTokTile - 1) / kTcTokTile + E + 1);
  t.b.nbase_w = cv.take<int32_t>(E + 1);
  t.b.tiles_w = cv.take<int4>((P + kTcWideTok - 1) / kTcWideTok + E + 1);
  t.b.nbase_r = cv.take<int32_t>(E + 1);
  t.b.tiles_r = cv.take<int4>((P + kTcRowTok - 1) / kTcRowTok + E + 1);
  t.tc = tc_path_supported((int)L, (int)I);
  if (t.tc) {
    t.xq = cv.take<uint8_t>(P * kTerms * (L / 2));
    t.xsf = cv.take<uint8_t>(P * kTerms * (L / 32));
    t.aq = cv.take<uint8_t>(P * kTerms * (I / 2));
    t.asf = cv.take<uint8_t>(P * kTerms * (I / 32));
    t.part = cv.take<float>(tc_part_floats((int)Tt));
    if (T >= kRowsMinTokens && wide_path_supported((int)L, (int)I))
      t.wdesc = cv.take<int4>(wide_desc_count((int)L, (int)I, (int)E, (int)Tt, (int)K));
  } else {
    t.x16 = cv.take<__half>(Tt * L);
    t.xexp = cv.take<int32_t>(Tt);
    t.act = cv.take<float>(P * I);
  }
  t.ybuf = cv.take<float>(P * L);
  if (host_stage) {
    t.h_stage = cv.take<uint16_t>(Tt * H);
    t.x_stage = cv.take<uint16_t>(Tt * L);
    t.y_stage = cv.take<float>(Tt * L);
  }
  if (w) *w = t;
  return (cv.off + 255) & ~size_t(255);
}

int check_ws(const k3moe_cfg* c, int32_t T, void* ws, size_t ws_bytes, bool host_stage,
             Workspace* w) {
  if (!ws || !aligned(ws, 256)) return K3MOE_ERR_WORKSPACE;
  if (ws_bytes < carve(c, T, nullptr, host_stage, nullptr)) return K3MOE_ERR_WORKSPACE;
  carve(c, T, ws, host_stage, w);
  return K3MOE_OK;
}

// The LatentMoE wrapper's regions, after the layer's own workspace.
struct LatentWs {
  uint16_t* z;  // [T][L] bf16: the experts' latent input
  float* y;     // [T][L]: the routed sum
  float* yn;    // [T][L]: after its RMSNorm
  float* act;   // [T][SI]: the shared experts' activations
};

constexpr int32_t kMaxLatentTokens = 4 * 65535;  // grid rows of four tokens

int shared_width(const k3moe_cfg* c, const k3moe_latent* lat) {
  return lat->n_shared > 0 ? lat->n_shared * c->inter : 0;
}

size_t carve_latent(const k3moe_cfg* c, const k3moe_latent* lat, int32_t T, void* base,
                    Workspace* w, LatentWs* lw) {
  Carver cv{static_cast<uint8_t*>(base)};
  cv.off = carve(c, T, base, false, w);
  const size_t Tt = (size_t)std::max(T, 1), L = c->latent;
  LatentWs t{};
  t.z = cv.take<uint16_t>(Tt * L);
  t.y = cv.take<float>(Tt * L);
  t.yn = cv.take<float>(Tt * L);
  t.act = cv.take<float>(Tt * (size_t)std::max(shared_width(c, lat), 1));
  if (lw) *lw = t;
  return (cv.off + 255) & ~size_t(255);
}

int check_latent(const k3moe_cfg* c, const k3moe_latent* lat) {
  if (!lat || !lat->down || !lat->up) return K3MOE_ERR_INVALID;
  if (lat->latent_norm != 0 && lat->latent_norm != 1) return K3MOE_ERR_INVALID;
  if (!(lat->rms_eps >= 0.f) || lat->n_shared < 0) return K3MOE_ERR_INVALID;
  if (!aligned(lat->down, 16) || !aligned(lat->up, 16) ||
      (lat->latent_norm_w && !aligned(lat->latent_norm_w, 4)))
    return K3MOE_ERR_ALIGN;
  if (lat->n_shared > 0) {
    if (!lat->sh1 || !lat->sh3 || !lat->sh2) return K3MOE_ERR_INVALID;
    if (!aligned(lat->sh1, 16) || !aligned(lat->sh3, 16) || !aligned(lat->sh2, 16))
      return K3MOE_ERR_ALIGN;
    if ((int64_t)lat->n_shared * c->inter > (1 << 20)) return K3MOE_ERR_UNSUPPORTED;
  }
  return K3MOE_OK;
}

int check_experts(const k3moe_experts* e) {
  if (!e) return K3MOE_ERR_INVALID;
  const void* p[6] = {e->w1_packed, e->w1_scale, e->w3_packed, e->w3_scale, e->w2_packed,
                      e->w2_scale};
  for (const void* q : p) {
    if (!q) return K3MOE_ERR_INVALID;
    if (!aligned(q, 16)) return K3MOE_ERR_ALIGN;
  }
  return K3MOE_OK;
}

int cuda_fail(const char* what, cudaError_t e);
int cuda_status(cudaError_t e) { return e == cudaSuccess ? K3MOE_OK : cuda_fail("launch", e); }

// Optional phase events (k3moe_set_phase_events).
cudaEvent_t g_phase[6] = {};
bool g_phase_on = false;

// Under stream capture the record is "external", so that it becomes an event-record node of
// the graph (timed on every replay) rather than a capture-internal dependency; outside a
// capture it is a plain record.
cudaError_t phase(int i, cudaStream_t s) {
  if (!g_phase_on) return cudaSuccess;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags(g_phase[i], s, cudaEventRecordExternal)
             : cudaEventRecord(g_phase[i], s);
}

void phase3(cudaStream_t s) { phase(3, s); }

// The last CUDA failure on this thread, for k3moe_last_error: the call that failed and CUDA's
// description of the error.
thread_local char g_last_error[256] = "";

int cuda_fail(const char* what, cudaError_t e) {
  std::snprintf(g_last_error, sizeof g_last_error, "%.120s: %.120s (%d)", what, cudaGetErrorString(e),
                (int)e);
  return K3MOE_ERR_CUDA;
}

#define K3_TRY(expr)                                  \
  do {                                                \
    cudaError_t _e = (expr);                          \
    if (_e != cudaSuccess) return cuda_fail(#expr, _e); \
  } while (0)

// Router launches (logits + top-k) into idx/gate/gap.
int run_route(const k3moe_cfg* c, const void* h, const void* wr, const float* bias, int32_t T,
              int32_t* idx, float* gate, float* gap, const Workspace& w, cudaStream_t s) {
  K3_TRY(launch_router_logits(static_cast<const uint16_t*>(h), static_cast<const uint16_t*>(wr),
                              T, c->n_experts, c->hidden, w.logits, s, false, nullptr, 0,
                              nullptr, nullptr, nullptr, 0, nullptr, w.rpart));
  K3_TRY(launch_topk(w.logits, w.rpart, router_splits(T, c->n_experts, c->hidden), bias, T,
                     c->n_experts, c->topk, c->renorm, c->routed_scale, idx, gate, gap, s, true));
  return K3MOE_OK;
}

// The layer (route = true) or the routed-expert sum alone (route = false):
//   [router logits (+ top-k grid for large T)] -> preparation (top-k for decode-sized T,
//   bucketing, x in f16) -> GEMM1 (w1, w3, activation) -> GEMM2 (w2, gates) -> combine.
//   Decode-sized T takes 5 launches (4 without the router).
int run_pipeline(const k3moe_cfg* c, bool route, const void* h, const void* wr,
                 const float* bias, const k3moe_experts* ex, const void* x, int32_t* idx,
                 float* gate, float* gap, int32_t T, float* y, int32_t* status,
                 const Workspace& w, cudaStream_t s) {
  const int E = c->n_experts, K = c->topk, L = c->latent, I = c->inter;
  ExpertPtrs ep{ex->w1_packed, ex->w1_scale, ex->w3_packed, ex->w3_scale, ex->w2_packed,
                ex->w2_scale};
  const int rsplit = route ? router_splits(T, E, c->hidden) : 1;
  // the preparation takes the top-k itself for small batches whose logits are not split (a
  // split router's partials are summed by the per-token top-k blocks, in parallel)
  const bool fused_topk = route && prep_is_fused(T) && rsplit == 1;
  K3_TRY(phase(0, s));
  // one token with the router's top-k on the tensor-core path: the router launch also
  // writes x's terms and zeroes the GEMMs' flags, and the GEMM CTAs route the token
  // themselves (no preparation launch)
  const bool one = w.tc && fused_topk && T == 1 && (K <= 31 || K == E);
  if (route) {
    K3_TRY(launch_router_logits(static_cast<const uint16_t*>(h), static_cast<const uint16_t*>(wr),
                                T, E, c->hidden, w.logits, s, true,
                                static_cast<const uint16_t*>(x), L, one ? w.xq : nullptr,
                                one ? w.xsf : nullptr, one ? w.b.flags : nullptr,
                                one ? kTcFlagWords : 0, status, w.rpart));
    if (!fused_topk)
      K3_TRY(launch_topk(w.logits, w.rpart, rsplit, bias, T, E, K, c->renorm, c->routed_scale, idx,
                         gate, gap, s, true));
  }
  K3_TRY(phase(1, s));
  // batches: positions of one expert as the MMA's M dimension (moe_wide.cu), the activation
  // terms as MMA rows below kWideMinTokens tokens, folded into the reduction from there; the
  // preparation writes those GEMMs' tile descriptors
  const bool wide = w.tc && T >= kRowsMinTokens && wide_path_supported(L, I);
  const bool rows = T < kWideMinTokens;
  BucketOut b = w.b;
  b.wdesc = nullptr;
  if (wide) wide_desc_setup(b, w.wdesc, L, I, E, T, K, rows);
  PrepArgs p{fused_topk ? w.logits : nullptr, bias, E, K, c->renorm, c->routed_scale, idx, gate,
             gap, T, L, static_cast<const uint16_t*>(x), w.tc ? nullptr : w.x16, w.xexp, b, y,
             status};
  const RouteOne ro{w.logits, bias, c->renorm, c->routed_scale, idx, gate, gap, y};
  if (!one) {
    K3_TRY(launch_prep(p, s, route));
    if (wide)
      K3_TRY(launch_split_x_wide(static_cast<const uint16_t*>(x), T, L, K, E, idx, b, w.xq,
                                 w.xsf, s, true));
    else if (w.tc)
      K3_TRY(launch_split_x(static_cast<const uint16_t*>(x), T, L, K, E, idx, b, w.xq, w.xsf,
                            s, true));
  }
  if (wide) {
    K3_TRY(phase(2, s));
    K3_TRY(launch_wide_experts(ep, L, I, E, T, K, rows, w.xq, w.xsf, b, w.aq, w.asf, c->act,
                               c->situ_b1, c->situ_b2, gate, w.ybuf, status, s, phase3));
    K3_TRY(phase(4, s));
  } else if (w.tc) {
    K3_TRY(phase(2, s));
    K3_TRY(launch_tc_experts(ep, L, I, E, T, K, w.xq, w.xsf, b, w.aq, w.asf, c->act,
                             c->situ_b1, c->situ_b2, gate, w.ybuf, w.part, status, s, true,
                             phase3, one ? &ro : nullptr));
    K3_TRY(phase(4, s));
  } else {
    K3_TRY(phase(2, s));
    K3_TRY(launch_gemm1(ep, L, I, E, T, K, w.x16, w.xexp, b, w.act, c->act, c->situ_b1,
                        c->situ_b2, status, s, true));
    K3_TRY(phase(3, s));
    K3_TRY(launch_gemm2(ep, L, I, E, T, K, w.act, gate, b, w.ybuf, status, s, true));
    K3_TRY(phase(4, s));
  }
  // one routed token: the second GEMM already summed the slots into y
  if (!one) K3_TRY(launch_combine(w.ybuf, idx, T, K, E, L, y, s, true));
  K3_TRY(phase(5, s));
  return K3MOE_OK;
}

// Scratch of k3moe_layer_static_scratch: one array per device that loads the library.  In
// host code g_static_scratch names a host-side stand-in; its device address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
static __device__ __align__(256) unsigned char g_static_scratch[K3MOE_STATIC_SCRATCH_BYTES];

// The address is cached per device together with the context it was looked up in: a
// destroyed and re-created primary context (cudaDeviceReset) holds the array at another
// address, so a change of context triggers a new lookup.
struct ScratchAddr {
  std::mutex m;
  void* ctx = nullptr;
  void* addr = nullptr;
};
ScratchAddr g_static_scratch_addr[64];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetCurrentFn>(nullptr);
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

int static_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return K3MOE_ERR_CUDA;
  CtxGetCurrentFn get = ctx_get_current_fn();
  CUcontext ctx = nullptr;
  if (!get || get(&ctx) != CUDA_SUCCESS) return K3MOE_ERR_CUDA;
  ScratchAddr& c = g_static_scratch_addr[dev];
  std::lock_guard<std::mutex> lk(c.m);
  if (!ctx || c.ctx != static_cast<void*>(ctx) || !c.addr) {
    // (no context yet on this thread: the lookup makes the device's primary context current)
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return K3MOE_ERR_CUDA;
    if (!ctx && (get(&ctx) != CUDA_SUCCESS || !ctx)) return K3MOE_ERR_CUDA;
    c.ctx = ctx;
    c.addr = p;
  }
  *out = c.addr;
  return K3MOE_OK;
}

// ---- k3moe_layer_host: cached CUDA graphs of repeated calls -------------------------------
//
// A call of k3moe_layer_host is two host-to-device copies, the layer's launches and one copy
// back.  Enqueued one by one that is about as much host time as the layer takes on the GPU at
// one token, so repeated calls with the same arguments replay an instantiated graph of the
// whole sequence instead (one launch).  The graph keeps every pointer and size it was recorded
// with, so the key is all of them; the buffers' contents are read at replay time.

struct HostGraphKey {
  k3moe_cfg cfg;
  int32_t T;
  const void *h, *x, *wr;
  const float* bias;
  float* y;
  k3moe_experts ex;
  int32_t* status;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
  uint32_t polls;
  int dev;
  bool operator==(const HostGraphKey& o) const { return std::memcmp(this, &o, sizeof o) == 0; }
};

struct HostGraph {
  HostGraphKey key;
  cudaGraphExec_t exec;  // nullptr: this argument set could not be captured (plain calls)
  uint64_t used;
};

constexpr int kHostGraphs = 16;
std::mutex g_hg_mutex;
HostGraph g_hg[kHostGraphs];
int g_hg_n = 0;
uint64_t g_hg_clock = 0;
cudaStream_t g_capture_stream[64] = {};

// The device's address of a page-locked host buffer that the GPU can reach directly (on a
// Grace-Blackwell node over NVLink-C2C), or nullptr for any other memory.
void* mapped_host(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// The copies and launches of one host-buffer call on stream s.  When all three host buffers
// are page-locked and mapped, the kernels read h and x and write y in host memory themselves
// (no staging copies); otherwise h and x are copied into the workspace and y back.
int enqueue_layer_host(const k3moe_cfg* cfg, const void* h_host, const void* wr, const float* bias,
                       const k3moe_experts* experts, const void* x_host, int32_t T, float* y_host,
                       int32_t* status, const Workspace& w, cudaStream_t s) {
  void* hd = mapped_host(h_host);
  void* xd = mapped_host(x_host);
  void* yd = mapped_host(y_host);
  if (hd && xd && yd && ((uintptr_t)hd | (uintptr_t)xd | (uintptr_t)yd) % 16 == 0)
    return run_pipeline(cfg, true, hd, wr, bias, experts, xd, w.idx, w.gate, w.gap, T,
                        static_cast<float*>(yd), status, w, s);
  const size_t hb = (size_t)T * cfg->hidden * 2, xb = (size_t)T * cfg->latent * 2,
               yb = (size_t)T * cfg->latent * 4;
  K3_TRY(cudaMemcpyAsync(w.h_stage, h_host, hb, cudaMemcpyHostToDevice, s));
  K3_TRY(cudaMemcpyAsync(w.x_stage, x_host, xb, cudaMemcpyHostToDevice, s));
  int rc = run_pipeline(cfg, true, w.h_stage, wr, bias, experts, w.x_stage, w.idx, w.gate, w.gap, T,
                        w.y_stage, status, w, s);
  if (rc) return rc;
  K3_TRY(cudaMemcpyAsync(y_host, w.y_stage, yb, cudaMemcpyDeviceToHost, s));
  return K3MOE_OK;
}

// Records the call as a graph on a private capture stream (the caller's stream may be the
// legacy default stream, which cannot be captured).  Returns nullptr if anything in the
// sequence cannot be captured (for example a copy from pageable host memory).
cudaGraphExec_t record_layer_host(const k3moe_cfg* cfg, const void* h_host, const void* wr,
                                  const float* bias, const k3moe_experts* experts,
                                  const void* x_host, int32_t T, float* y_host, int32_t* status,
                                  const Workspace& w, int dev) {
  if (dev < 0 || dev >= 64) return nullptr;
  if (!g_capture_stream[dev] &&
      cudaStreamCreateWithFlags(&g_capture_stream[dev], cudaStreamNonBlocking) != cudaSuccess)
    return nullptr;
  cudaStream_t cs = g_capture_stream[dev];
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  const int rc = enqueue_layer_host(cfg, h_host, wr, bias, experts, x_host, T, y_host, status, w, cs);
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(cs, &g);
  cudaGraphExec_t exec = nullptr;
  if (rc == K3MOE_OK && e == cudaSuccess && g) {
    if (cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) exec = nullptr;
  }
  if (g) cudaGraphDestroy(g);
  cudaGetLastError();  // a refused capture leaves no error behind
  return exec;
}

// The host-buffer layer: replays a recorded graph when it can, with or without the final
// synchronisation.
int layer_host(const k3moe_cfg* cfg, const void* h_host, const void* wr, const float* bias,
               const k3moe_experts* experts, const void* x_host, int32_t T, float* y_host,
               int32_t* status, void* ws, size_t ws_bytes, void* stream, bool sync) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_experts(experts))) return rc;
  if (T < 0) return K3MOE_ERR_INVALID;
  if (T > kMaxTokens) return K3MOE_ERR_UNSUPPORTED;
  if (T == 0) return K3MOE_OK;
  if (!h_host || !wr || !x_host || !y_host) return K3MOE_ERR_INVALID;
  if (!aligned(wr, 16) || (bias && !aligned(bias, 4)) || (status && !aligned(status, 4)))
    return K3MOE_ERR_ALIGN;
  Workspace w;
  if ((rc = check_ws(cfg, T, ws, ws_bytes, true, &w))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  K3_TRY(cudaGetDevice(&dev));
  if (!sync && mapped_host(h_host) && mapped_host(x_host) && mapped_host(y_host)) {
    // kernels read h and x and write y in host memory: the launches are enqueued as they are
    // (no graph), so that programmatic dependent launch overlaps consecutive calls' edges
    return enqueue_layer_host(cfg, h_host, wr, bias, experts, x_host, T, y_host, status, w, s);
  }
  if (!g_phase_on) {  // (phase events are recorded per call: no graphs while they are on)
    HostGraphKey key;
    std::memset(&key, 0, sizeof key);
    key.cfg = *cfg;
    key.T = T;
    key.h = h_host;
    key.x = x_host;
    key.wr = wr;
    key.bias = bias;
    key.y = y_host;
    key.ex = *experts;
    key.status = status;
    key.ws = ws;
    key.ws_bytes = ws_bytes;
    key.stream = s;
    key.polls = flag_wait_polls();
    key.dev = dev;
    std::unique_lock<std::mutex> lk(g_hg_mutex);
    for (int i = 0; i < g_hg_n; ++i) {
      if (g_hg[i].key == key) {
        g_hg[i].used = ++g_hg_clock;
        if (g_hg[i].exec) {
          K3_TRY(cudaGraphLaunch(g_hg[i].exec, s));
          lk.unlock();
          if (sync) K3_TRY(cudaStreamSynchronize(s));
          return K3MOE_OK;
        }
        lk.unlock();
        goto plain;  // known not to capture
      }
    }
    lk.unlock();
    // first call with these arguments: run it directly, then record it for the next ones
    if ((rc = enqueue_layer_host(cfg, h_host, wr, bias, experts, x_host, T, y_host, status, w, s)))
      return rc;
    K3_TRY(cudaStreamSynchronize(s));
    cudaGraphExec_t exec =
        record_layer_host(cfg, h_host, wr, bias, experts, x_host, T, y_host, status, w, dev);
    lk.lock();
    int slot = g_hg_n < kHostGraphs ? g_hg_n++ : 0;
    if (slot == 0 && g_hg_n == kHostGraphs) {
      for (int i = 1; i < kHostGraphs; ++i)
        if (g_hg[i].used < g_hg[slot].used) slot = i;
      if (g_hg[slot].exec) cudaGraphExecDestroy(g_hg[slot].exec);
    }
    g_hg[slot] = HostGraph{key, exec, ++g_hg_clock};
    return K3MOE_OK;
  }
plain:
  if ((rc = enqueue_layer_host(cfg, h_host, wr, bias, experts, x_host, T, y_host, status, w, s)))
    return rc;
  K3_TRY(cudaStreamSynchronize(s));
  return K3MOE_OK;
}
}  // namespace
}  // namespace k3

using namespace k3;

extern "C" {

int k3moe_workspace_size(const k3moe_cfg* cfg, int32_t T, size_t* bytes) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!bytes || T < 0) return K3MOE_ERR_INVALID;
  if (T > kMaxTokens) return K3MOE_ERR_UNSUPPORTED;
  *bytes = carve(cfg, T, nullptr, false, nullptr);
  return K3MOE_OK;
}

int k3moe_workspace_size_host(const k3moe_cfg* cfg, int32_t T, size_t* bytes) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!bytes || T < 0) return K3MOE_ERR_INVALID;
  if (T > kMaxTokens) return K3MOE_ERR_UNSUPPORTED;
  *bytes = carve(cfg, T, nullptr, true, nullptr);
  return K3MOE_OK;
}

int k3moe_route(const k3moe_cfg* cfg, const void* h, const void* wr, const float* bias, int32_t T,
                int32_t* idx, float* gate, float* gap, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (T < 0) return K3MOE_ERR_INVALID;
  if (T > kMaxTokens) return K3MOE_ERR_UNSUPPORTED;
  if (T == 0) return K3MOE_OK;  // nothing to do; empty tensors may carry null pointers
  if (!h || !wr || !idx || !gate) return K3MOE_ERR_INVALID;
  if (!aligned(h, 16) || !aligned(wr, 16) || !aligned(idx, 4) || !aligned(gate, 4) ||
      (bias && !aligned(bias, 4)) || (gap && !aligned(gap, 4)))
    return K3MOE_ERR_ALIGN;
  Workspace w;
  if ((rc = check_ws(cfg, T, ws, ws_bytes, false, &w))) return rc;
  return run_route(cfg, h, wr, bias, T, idx, gate, gap, w, static_cast<cudaStream_t>(stream));
}

int k3moe_experts_mxfp4(const k3moe_cfg* cfg, const k3moe_experts* experts, const void* x,
                        const int32_t* idx, const float* gate, int32_t T, float* y,
                        int32_t* status, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_experts(experts))) return rc;
  if (T < 0) return K3MOE_ERR_INVALID;
  if (T > kMaxTokens) return K3MOE_ERR_UNSUPPORTED;
  if (T == 0) return K3MOE_OK;
  if (!x || !idx || !gate || !y) return K3MOE_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(idx, 4) || !aligned(gate, 4) ||
      (status && !aligned(status, 4)))
    return K3MOE_ERR_ALIGN;
  Workspace w;
  if ((rc = check_ws(cfg, T, ws, ws_bytes, false, &w))) return rc;
  return run_pipeline(cfg, false, nullptr, nullptr, nullptr, experts, x, const_cast<int32_t*>(idx),
                      const_cast<float*>(gate), nullptr, T, y, status, w,
                      static_cast<cudaStream_t>(stream));
}

int k3moe_experts_mxfp4_range(const k3moe_cfg* cfg, const k3moe_experts* experts, int32_t e0,
                              int32_t e1, const void* x, const int32_t* idx, const float* gate,
                              int32_t T, float* y, int32_t* status, void* ws, size_t ws_bytes,
                              void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_experts(experts))) return rc;
  if (T < 0 || e0 < 0 || e1 <= e0 || e1 > cfg->n_experts) return K3MOE_ERR_INVALID;
  if (T > kMaxTokens) return K3MOE_ERR_UNSUPPORTED;
  if (T == 0) return K3MOE_OK;
  if (!x || !idx || !gate || !y) return K3MOE_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(idx, 4) || !aligned(gate, 4) ||
      (status && !aligned(status, 4)))
    return K3MOE_ERR_ALIGN;
  // the local block as a layer of e1 - e0 experts (k <= E still holds for the routing the
  // caller made over all E; the local count may be smaller than k)
  k3moe_cfg local = *cfg;
  local.n_experts = e1 - e0;
  Workspace w;
  if (!ws || !aligned(ws, 256)) return K3MOE_ERR_WORKSPACE;
  if (ws_bytes < carve(&local, T, nullptr, false, nullptr)) return K3MOE_ERR_WORKSPACE;
  carve(&local, T, ws, false, &w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  K3_TRY(launch_localize_idx(idx, T * cfg->topk, cfg->n_experts, e0, e1, w.idx, s, true));
  return run_pipeline(&local, false, nullptr, nullptr, nullptr, experts, x, w.idx,
                      const_cast<float*>(gate), nullptr, T, y, status, w, s);
}

int k3moe_layer(const k3moe_cfg* cfg, const void* h, const void* wr, const float* bias,
                const k3moe_experts* experts, const void* x, int32_t T, float* y, int32_t* idx,
                float* gate, float* gap, int32_t* status, void* ws, size_t ws_bytes,
                void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_experts(experts))) return rc;
  if (T < 0) return K3MOE_ERR_INVALID;
  if (T > kMaxTokens) return K3MOE_ERR_UNSUPPORTED;
  if (T == 0) return K3MOE_OK;
  if (!h || !wr || !x || !y) return K3MOE_ERR_INVALID;
  if (!aligned(h, 16) || !aligned(wr, 16) || !aligned(x, 16) || !aligned(y, 16) ||
      (bias && !aligned(bias, 4)) || (idx && !aligned(idx, 4)) || (gate && !aligned(gate, 4)) ||
      (gap && !aligned(gap, 4)) || (status && !aligned(status, 4)))
    return K3MOE_ERR_ALIGN;
  Workspace w;
  if ((rc = check_ws(cfg, T, ws, ws_bytes, false, &w))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* idx_use = idx ? idx : w.idx;
  float* gate_use = gate ? gate : w.gate;
  float* gap_use = gap ? gap : w.gap;
  return run_pipeline(cfg, true, h, wr, bias, experts, x, idx_use, gate_use, gap_use, T, y, status,
                      w, s);
}

int k3moe_layer_static_scratch(const k3moe_cfg* cfg, const void* h, const void* wr,
                               const float* bias, const k3moe_experts* experts, const void* x,
                               int32_t T, float* y, int32_t* idx, float* gate, float* gap,
                               int32_t* status, void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_experts(experts))) return rc;
  if (T < 0) return K3MOE_ERR_INVALID;
  if (T > kMaxTokens) return K3MOE_ERR_UNSUPPORTED;
  if (T == 0) return K3MOE_OK;
  if (!h || !wr || !x || !y) return K3MOE_ERR_INVALID;
  if (!aligned(h, 16) || !aligned(wr, 16) || !aligned(x, 16) || !aligned(y, 16) ||
      (bias && !aligned(bias, 4)) || (idx && !aligned(idx, 4)) || (gate && !aligned(gate, 4)) ||
      (gap && !aligned(gap, 4)) || (status && !aligned(status, 4)))
    return K3MOE_ERR_ALIGN;
  const size_t need = carve(cfg, T, nullptr, false, nullptr);
  if (need > K3MOE_STATIC_SCRATCH_BYTES) return K3MOE_ERR_TOO_LARGE;
  void* base = nullptr;
  if ((rc = static_scratch_address(&base))) return rc;
  Workspace w;
  carve(cfg, T, base, false, &w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return run_pipeline(cfg, true, h, wr, bias, experts, x, idx ? idx : w.idx, gate ? gate : w.gate,
                      gap ? gap : w.gap, T, y, status, w, s);
}

int k3moe_layer_host(const k3moe_cfg* cfg, const void* h_host, const void* wr, const float* bias,
                     const k3moe_experts* experts, const void* x_host, int32_t T, float* y_host,
                     int32_t* status, void* ws, size_t ws_bytes, void* stream) {
  return k3::layer_host(cfg, h_host, wr, bias, experts, x_host, T, y_host, status, ws, ws_bytes,
                        stream, true);
}

int k3moe_layer_host_async(const k3moe_cfg* cfg, const void* h_host, const void* wr,
                           const float* bias, const k3moe_experts* experts, const void* x_host,
                           int32_t T, float* y_host, int32_t* status, void* ws, size_t ws_bytes,
                           void* stream) {
  return k3::layer_host(cfg, h_host, wr, bias, experts, x_host, T, y_host, status, ws, ws_bytes,
                        stream, false);
}

int k3moe_latent_workspace_size(const k3moe_cfg* cfg, const k3moe_latent* lat, int32_t T,
                                size_t* bytes) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_latent(cfg, lat))) return rc;
  if (!bytes || T < 0) return K3MOE_ERR_INVALID;
  if (T > kMaxLatentTokens) return K3MOE_ERR_UNSUPPORTED;
  *bytes = carve_latent(cfg, lat, T, nullptr, nullptr, nullptr);
  return K3MOE_OK;
}

int k3moe_latent_layer(const k3moe_cfg* cfg, const k3moe_latent* lat, const void* h,
                       const void* wr, const float* bias, const k3moe_experts* experts,
                       int32_t T, float* out, int32_t* idx, float* gate, float* gap,
                       int32_t* status, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_latent(cfg, lat))) return rc;
  if ((rc = check_experts(experts))) return rc;
  if (T < 0) return K3MOE_ERR_INVALID;
  if (T > kMaxLatentTokens) return K3MOE_ERR_UNSUPPORTED;
  if (T == 0) return K3MOE_OK;
  if (!h || !wr || !out) return K3MOE_ERR_INVALID;
  if (!aligned(h, 16) || !aligned(wr, 16) || !aligned(out, 16) || (bias && !aligned(bias, 4)) ||
      (idx && !aligned(idx, 4)) || (gate && !aligned(gate, 4)) || (gap && !aligned(gap, 4)) ||
      (status && !aligned(status, 4)))
    return K3MOE_ERR_ALIGN;
  if (!ws || !aligned(ws, 256)) return K3MOE_ERR_WORKSPACE;
  if (ws_bytes < carve_latent(cfg, lat, T, nullptr, nullptr, nullptr)) return K3MOE_ERR_WORKSPACE;
  Workspace w;
  LatentWs lw;
  carve_latent(cfg, lat, T, ws, &w, &lw);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int H = cfg->hidden, L = cfg->latent, SI = shared_width(cfg, lat);
  const auto* h16 = static_cast<const uint16_t*>(h);
  K3_TRY(launch_dense_in(h16, T, H, static_cast<const uint16_t*>(lat->down), L, lw.z,
                         static_cast<const uint16_t*>(lat->sh1),
                         static_cast<const uint16_t*>(lat->sh3), SI, lw.act, cfg->act,
                         cfg->situ_b1, cfg->situ_b2, s, true));
  if ((rc = run_pipeline(cfg, true, h, wr, bias, experts, lw.z, idx ? idx : w.idx,
                         gate ? gate : w.gate, gap ? gap : w.gap, T, lw.y, status, w, s)))
    return rc;
  K3_TRY(launch_latent_norm(lw.y, T, L, lat->latent_norm, lat->latent_norm_w, lat->rms_eps,
                            lw.yn, s, true));
  K3_TRY(launch_dense_out(lw.yn, T, L, static_cast<const uint16_t*>(lat->up), H, lw.act,
                          static_cast<const uint16_t*>(lat->sh2), SI, out, s, true));
  return K3MOE_OK;
}

int k3moe_matvec_mxfp4(float* y, const void* x, const uint8_t* packed, const uint8_t* scales,
                       int32_t in, int32_t rows, int32_t group, void* stream) {
  if (!y || !x || !packed || !scales || in <= 0 || rows < 0) return K3MOE_ERR_INVALID;
  if (group != kGroup || in % 32 != 0) return K3MOE_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(packed, 16) || !aligned(y, 4)) return K3MOE_ERR_ALIGN;
  if (rows == 0) return K3MOE_OK;
  return cuda_status(launch_matvec(y, static_cast<const uint16_t*>(x), packed, scales, in, rows,
                                   static_cast<cudaStream_t>(stream)));
}

int k3moe_stack_link(const float* y, int32_t T, int32_t L, int32_t norm, float eps, void* x_out,
                     void* h_out, void* stream) {
  if (T < 0 || L <= 0 || !(eps >= 0.f)) return K3MOE_ERR_INVALID;
  if (T == 0) return K3MOE_OK;
  if (!y || !x_out) return K3MOE_ERR_INVALID;
  if (!aligned(y, 4) || !aligned(x_out, 2) || (h_out && !aligned(h_out, 2))) return K3MOE_ERR_ALIGN;
  return cuda_status(launch_stack_link(y, T, L, norm, eps, static_cast<uint16_t*>(x_out),
                                       static_cast<uint16_t*>(h_out),
                                       static_cast<cudaStream_t>(stream)));
}

int k3moe_set_phase_events(void* const* events, int32_t n) {
  if (!events) {
    g_phase_on = false;
    return K3MOE_OK;
  }
  if (n != 6) return K3MOE_ERR_INVALID;
  for (int i = 0; i < 6; ++i) {
    if (!events[i]) return K3MOE_ERR_INVALID;
    g_phase[i] = static_cast<cudaEvent_t>(events[i]);
  }
  g_phase_on = true;
  return K3MOE_OK;
}

int k3moe_set_flag_wait_polls(int64_t polls) {
  if (polls > (int64_t)UINT32_MAX) return K3MOE_ERR_INVALID;
  g_flag_polls.store(polls < 0 ? kWaitPolls : (uint32_t)polls);
  return K3MOE_OK;
}

int64_t k3moe_launch_count(void) { return g_launches.load(); }

const char* k3moe_last_error(void) { return g_last_error; }

const char* k3moe_strerror(int status) {
  switch (status) {
    case K3MOE_OK: return "ok";
    case K3MOE_ERR_INVALID: return "invalid argument";
    case K3MOE_ERR_UNSUPPORTED: return "unsupported shape or configuration";
    case K3MOE_ERR_ALIGN: return "pointer not aligned";
    case K3MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case K3MOE_ERR_CUDA: return "CUDA launch or copy failed";
    case K3MOE_ERR_TIMEOUT: return "a bounded device wait ran out";
    case K3MOE_ERR_DROPPED: return "expert index out of range (assignment skipped)";
    case K3MOE_ERR_TOO_LARGE: return "request exceeds the static scratch capacity (16 MiB)";
    default: return "unknown status";
  }
}

int32_t k3moe_abi_version(void) { return K3MOE_ABI_VERSION; }

}  // extern "C"
