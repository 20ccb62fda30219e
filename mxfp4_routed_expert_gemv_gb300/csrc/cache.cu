// cache.cu -- experts beyond HBM: a device cache of slots over an expert store in host memory.
//
// README "kimi-k3-in-c", Part II section 12 "An LRU cache for the experts": experts are read
// from a large, slower tier into a fixed set of slots in fast memory; a slot holds an
// expert, is empty, or is in flight; a call reserves its slots first (an empty slot if
// there is one, else the least recently used one that the call itself does not need), then
// reads the reserved experts in the store's offset order, then publishes what arrived.
// Here the tier is page-locked host memory (Grace memory over NVLink-C2C on a Grace-
// Blackwell node), the reads are host-to-device copies on the call's stream, and stream
// order publishes them to the expert kernels that follow.  The planning is host code; the
// slots are an ordinary k3moe_experts of n_slots experts, so the expert kernels run on them
// unchanged with the routing mapped from expert ids to slot ids.
#include <algorithm>
#include <cstring>

#include "k3moe.h"
#include "launch.h"

namespace k3 {
namespace {

constexpr int32_t kWanted = -3;   // planning marker: a missing expert the call needs
constexpr int32_t kListed = -4;   // planning marker: a missing expert already in the list
constexpr int32_t kResBase = -10; // planning marker: a resident expert in slot s is kResBase - s

int check_cache(const k3moe_expert_cache* c) {
  if (!c || !c->expert_of || !c->slot_of || !c->used_at) return K3MOE_ERR_INVALID;
  if (c->n_experts < 1 || c->n_slots < 1 || c->n_slots > c->n_experts) return K3MOE_ERR_INVALID;
  return K3MOE_OK;
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// The device's address of page-locked host memory it can reach directly (over NVLink-C2C on
// a Grace-Blackwell node), or nullptr.
const uint8_t* mapped(const uint8_t* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? static_cast<const uint8_t*>(a.devicePointer) : nullptr;
}

struct CopyArgs {
  const uint8_t* src[6];  // the store's tensors (device addresses of the host memory)
  uint8_t* dst[6];        // the slots' tensors
  size_t per[6];          // bytes of one expert in each tensor (multiples of 16)
  const int32_t* fetch;   // [2][n]: experts, then their slots
  int n;
};

// The planned experts host -> device by the SMs themselves (loads from the mapped host store,
// stores to the slots): block (x, j * 6 + m) copies its stretch of tensor m of fetch j, 16 bytes
// a thread at a time with four loads in flight.
__global__ void __launch_bounds__(256) k_copy_experts(const CopyArgs a) {
  const int j = blockIdx.y / 6, m = blockIdx.y - 6 * (blockIdx.y / 6);
  if (j >= a.n) return;
  const size_t units = a.per[m] >> 4;
  const uint4* src = reinterpret_cast<const uint4*>(a.src[m] + (size_t)a.fetch[j] * a.per[m]);
  uint4* dst = reinterpret_cast<uint4*>(a.dst[m] + (size_t)a.fetch[a.n + j] * a.per[m]);
  const size_t step = (size_t)gridDim.x * blockDim.x;
  size_t u = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; u + 3 * step < units; u += 4 * step) {
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __ldcs(src + u + i * step);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[u + i * step] = v[i];
  }
  for (; u < units; u += step) dst[u] = __ldcs(src + u);
}

}  // namespace
}  // namespace k3

using namespace k3;

extern "C" {

int k3moe_cache_reset(k3moe_expert_cache* c) {
  int rc = check_cache(c);
  if (rc) return rc;
  for (int32_t s = 0; s < c->n_slots; ++s) {
    c->expert_of[s] = K3MOE_SLOT_EMPTY;
    c->used_at[s] = 0;
  }
  for (int32_t e = 0; e < c->n_experts; ++e) c->slot_of[e] = -1;
  c->clock = 0;
  return K3MOE_OK;
}

int k3moe_cache_plan(k3moe_expert_cache* c, const int32_t* idx, int32_t n, int32_t* slot_idx,
                     int32_t* fetch_expert, int32_t* fetch_slot, int32_t* n_fetch) {
  int rc = check_cache(c);
  if (rc) return rc;
  if (n < 0 || !n_fetch || (n > 0 && (!idx || !slot_idx)) || !fetch_expert || !fetch_slot)
    return K3MOE_ERR_INVALID;
  const int32_t E = c->n_experts, C = c->n_slots;
  auto resident = [&](int32_t e) {
    const int32_t s = c->slot_of[e];
    return s >= 0 && s < C && c->expert_of[s] == e;
  };
  // pass 1: mark each distinct expert once (resident: its slot, encoded; missing: wanted)
  int32_t distinct = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t e = idx[i];
    if (e < 0 || e >= E) continue;
    if (resident(e)) {
      c->slot_of[e] = kResBase - c->slot_of[e];
      ++distinct;
    } else if (c->slot_of[e] == -1 || c->slot_of[e] >= 0) {
      c->slot_of[e] = kWanted;
      ++distinct;
    }
  }
  int32_t inflight = 0;
  for (int32_t s = 0; s < C; ++s) inflight += c->expert_of[s] == K3MOE_SLOT_INFLIGHT ? 1 : 0;
  if (distinct + inflight > C) {
    // undo the marks: the state is left as it was
    for (int32_t i = 0; i < n; ++i) {
      const int32_t e = idx[i];
      if (e < 0 || e >= E) continue;
      if (c->slot_of[e] <= kResBase) c->slot_of[e] = kResBase - c->slot_of[e];
      else if (c->slot_of[e] == kWanted) c->slot_of[e] = -1;
    }
    return K3MOE_ERR_UNSUPPORTED;
  }
  const uint64_t now = c->clock + 1;
  // pass 2: the resident ones are used now; the missing ones are listed once each
  int32_t nf = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t e = idx[i];
    if (e < 0 || e >= E) continue;
    if (c->slot_of[e] <= kResBase) {
      const int32_t s = kResBase - c->slot_of[e];
      c->slot_of[e] = s;
      c->used_at[s] = now;
    } else if (c->slot_of[e] == kWanted) {
      c->slot_of[e] = kListed;
      fetch_expert[nf++] = e;
    }
  }
  // reserve in ascending expert order (the store's offset order): an empty slot first,
  // else the least recently used slot that this call does not use and that is not in flight
  std::sort(fetch_expert, fetch_expert + nf);
  for (int32_t j = 0; j < nf; ++j) {
    int32_t v = -1;
    for (int32_t s = 0; s < C && v < 0; ++s)
      if (c->expert_of[s] == K3MOE_SLOT_EMPTY) v = s;
    if (v < 0) {
      for (int32_t s = 0; s < C; ++s) {
        if (c->expert_of[s] < 0 || c->used_at[s] >= now) continue;
        if (v < 0 || c->used_at[s] < c->used_at[v]) v = s;
      }
    }
    // (distinct + in-flight <= C guarantees a slot)
    if (c->expert_of[v] >= 0) c->slot_of[c->expert_of[v]] = -1;  // evicted
    c->expert_of[v] = K3MOE_SLOT_INFLIGHT;
    c->used_at[v] = now;
    c->slot_of[fetch_expert[j]] = v;
    fetch_slot[j] = v;
  }
  for (int32_t i = 0; i < n; ++i) {
    const int32_t e = idx[i];
    slot_idx[i] = (e >= 0 && e < E) ? c->slot_of[e] : -1;
  }
  c->clock = now;
  *n_fetch = nf;
  return K3MOE_OK;
}

int k3moe_cache_publish(k3moe_expert_cache* c, const int32_t* fetch_expert,
                        const int32_t* fetch_slot, int32_t n_fetch, int32_t n_ok) {
  int rc = check_cache(c);
  if (rc) return rc;
  if (n_fetch < 0 || n_ok < 0 || n_ok > n_fetch || (n_fetch > 0 && (!fetch_expert || !fetch_slot)))
    return K3MOE_ERR_INVALID;
  for (int32_t j = 0; j < n_fetch; ++j) {
    const int32_t e = fetch_expert[j], s = fetch_slot[j];
    if (e < 0 || e >= c->n_experts || s < 0 || s >= c->n_slots) return K3MOE_ERR_INVALID;
    if (j < n_ok) {
      c->expert_of[s] = e;
    } else {
      c->expert_of[s] = K3MOE_SLOT_EMPTY;
      if (c->slot_of[e] == s) c->slot_of[e] = -1;
    }
  }
  return K3MOE_OK;
}

int k3moe_cache_workspace_size(const k3moe_cfg* cfg, int32_t T, size_t* bytes) {
  if (!bytes) return K3MOE_ERR_INVALID;
  size_t b = 0;
  int rc = k3moe_workspace_size(cfg, T, &b);
  if (rc) return rc;
  const size_t P = (size_t)T * cfg->topk;
  // idx, gate, then the slot ids followed by room for a fetch list of up to E experts
  *bytes = align256(b) + 2 * align256(P * 4) + align256((P + 2 * (size_t)cfg->n_experts) * 4);
  return K3MOE_OK;
}

int k3moe_cache_host_scratch_size(const k3moe_cfg* cfg, int32_t T, int32_t n_slots,
                                  size_t* bytes) {
  if (!cfg || !bytes || T < 0 || n_slots < 1) return K3MOE_ERR_INVALID;
  *bytes = (2 * (size_t)T * cfg->topk + 2 * (size_t)n_slots) * 4;
  return K3MOE_OK;
}

int k3moe_layer_cached(const k3moe_cfg* cfg, k3moe_expert_cache* c, const void* h,
                       const void* wr, const float* bias, const void* x, int32_t T, float* y,
                       int32_t* status, void* ws, size_t ws_bytes, void* host_scratch,
                       size_t host_scratch_bytes, int32_t* n_fetched, void* stream) {
  int rc = check_cache(c);
  if (rc) return rc;
  if (!cfg) return K3MOE_ERR_INVALID;
  if (c->n_experts != cfg->n_experts) return K3MOE_ERR_INVALID;
  if (cfg->topk > c->n_slots) return K3MOE_ERR_UNSUPPORTED;  // a token's experts need k slots
  if (n_fetched) *n_fetched = 0;
  if (T == 0) return K3MOE_OK;
  size_t need = 0, need_h = 0;
  if ((rc = k3moe_cache_workspace_size(cfg, T, &need))) return rc;
  if ((rc = k3moe_cache_host_scratch_size(cfg, T, c->n_slots, &need_h))) return rc;
  if (!ws || ws_bytes < need) return K3MOE_ERR_WORKSPACE;
  if (!host_scratch || host_scratch_bytes < need_h) return K3MOE_ERR_INVALID;
  const k3moe_experts* hs = &c->host;
  if (!hs->w1_packed || !hs->w1_scale || !hs->w3_packed || !hs->w3_scale || !hs->w2_packed ||
      !hs->w2_scale)
    return K3MOE_ERR_INVALID;
  const int32_t K = cfg->topk, C = c->n_slots;
  const size_t P = (size_t)T * K;
  size_t main_bytes = 0;
  if ((rc = k3moe_workspace_size(cfg, T, &main_bytes))) return rc;
  uint8_t* wp = static_cast<uint8_t*>(ws);
  int32_t* d_idx = reinterpret_cast<int32_t*>(wp + align256(main_bytes));
  float* d_gate = reinterpret_cast<float*>(wp + align256(main_bytes) + align256(P * 4));
  int32_t* d_slot = reinterpret_cast<int32_t*>(wp + align256(main_bytes) + 2 * align256(P * 4));
  int32_t* h_idx = static_cast<int32_t*>(host_scratch);
  int32_t* h_slot = h_idx + P;
  int32_t* f_exp = h_slot + P;
  int32_t* f_slot = f_exp + C;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // route, then read the routing back: it decides what to copy
  if ((rc = k3moe_route(cfg, h, wr, bias, T, d_idx, d_gate, nullptr, ws, main_bytes, stream)))
    return rc;
  if (cudaMemcpyAsync(h_idx, d_idx, P * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return K3MOE_ERR_CUDA;
  int32_t nf = 0;
  if ((rc = k3moe_cache_plan(c, h_idx, (int32_t)P, h_slot, f_exp, f_slot, &nf))) return rc;

  // the reserved experts, host -> device, in ascending expert order: by the SMs from the
  // mapped store when the store is mapped page-locked memory (the slot ids go to the device
  // with the fetch list), else one copy per tensor
  const size_t L = (size_t)cfg->latent, I = (size_t)cfg->inter;
  const size_t b13 = I * L / 2, s13 = I * L / 32, b2 = L * I / 2, s2 = L * I / 32;
  const uint8_t* src[6] = {hs->w1_packed, hs->w1_scale, hs->w3_packed, hs->w3_scale,
                           hs->w2_packed, hs->w2_scale};
  const uint8_t* dst[6] = {c->slots.w1_packed, c->slots.w1_scale, c->slots.w3_packed,
                           c->slots.w3_scale, c->slots.w2_packed, c->slots.w2_scale};
  const size_t per[6] = {b13, s13, b13, s13, b2, s2};
  CopyArgs ca{};
  bool direct = nf > 0;
  for (int m = 0; m < 6 && direct; ++m) {
    ca.src[m] = mapped(src[m]);
    ca.dst[m] = const_cast<uint8_t*>(dst[m]);
    ca.per[m] = per[m];
    direct = ca.src[m] != nullptr && per[m] % 16 == 0 && (reinterpret_cast<uintptr_t>(ca.src[m]) % 16) == 0;
  }
  int32_t ok = 0;
  if (direct) {
    // the slot ids and the fetch list in one copy: h_slot [P], then f_exp [C], f_slot [C]
    int32_t* fs2 = f_exp + nf;  // [experts nf][slots nf], contiguous after h_slot
    std::memmove(fs2, f_slot, (size_t)nf * 4);
    f_slot = fs2;
    if (cudaMemcpyAsync(d_slot, h_slot, (P + 2 * (size_t)nf) * 4, cudaMemcpyHostToDevice, s) !=
        cudaSuccess) {
      k3moe_cache_publish(c, f_exp, f_slot, nf, 0);
      return K3MOE_ERR_CUDA;
    }
    ca.fetch = d_slot + P;
    ca.n = nf;
    const cudaError_t e = launch_kernel(k_copy_experts, dim3(64, 6 * nf), dim3(256), 0, s, false, ca);
    ok = e == cudaSuccess ? nf : 0;
  } else {
    for (; ok < nf; ++ok) {
      bool issued = true;
      for (int m = 0; m < 6 && issued; ++m)
        issued = cudaMemcpyAsync(const_cast<uint8_t*>(dst[m]) + (size_t)f_slot[ok] * per[m],
                                 src[m] + (size_t)f_exp[ok] * per[m], per[m],
                                 cudaMemcpyHostToDevice, s) == cudaSuccess;
      if (!issued) break;
    }
  }
  k3moe_cache_publish(c, f_exp, f_slot, nf, ok);
  if (ok < nf) {
    cudaStreamSynchronize(s);
    return K3MOE_ERR_CUDA;
  }
  if (n_fetched) *n_fetched = nf;

  // the routed-expert sum on the slots
  if (!direct && cudaMemcpyAsync(d_slot, h_slot, P * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return K3MOE_ERR_CUDA;
  k3moe_cfg cs = *cfg;
  cs.n_experts = C;
  rc = k3moe_experts_mxfp4(&cs, &c->slots, x, d_slot, d_gate, T, y, status, ws, main_bytes,
                           stream);
  if (rc) {
    cudaStreamSynchronize(s);
    return rc;
  }
  // the host scratch is read by the copy above: it stays in use until the stream gets here
  if (cudaStreamSynchronize(s) != cudaSuccess) return K3MOE_ERR_CUDA;
  return K3MOE_OK;
}

}  // extern "C"
