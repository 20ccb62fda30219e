// Device twin of the seeded expert-byte generator (see synth/__init__.py).
//
// Input generation only: none of the MoE layer's arithmetic is here.  SplitMix64
// (S. Vigna, public domain) used as a counter-based generator: word i of the stream with
// key K is the SplitMix64 output function applied to K + (i+1)*0x9E3779B97F4A7C15.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kLayerMul = 0xD1B54A32D192ED03ull;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ inline uint64_t stream_key(uint64_t seed, uint64_t layer, uint64_t tensor,
                                               uint64_t expert) {
  uint64_t k0 = mix64(seed + kGamma);
  uint64_t k1 = mix64(k0 ^ (layer * kLayerMul));
  return mix64(k1 ^ ((tensor << 40) ^ expert));
}

// Packed tensors: word w of expert e gives bytes 8w..8w+7 (least significant first).
__global__ void fill_packed(uint8_t* __restrict__ dst, int64_t n_experts, int64_t bpe,
                            uint64_t seed, uint64_t layer, uint64_t tensor) {
  const int64_t wpe = (bpe + 7) / 8;
  const int64_t total = n_experts * wpe;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i / wpe, w = i % wpe;
    const uint64_t key = stream_key(seed, layer, tensor, (uint64_t)e);
    const uint64_t v = mix64(key + (uint64_t)(w + 1) * kGamma);
    uint8_t* p = dst + e * bpe + w * 8;
    const int64_t nb = (bpe - w * 8) < 8 ? (bpe - w * 8) : 8;
    if (nb == 8 && (((uintptr_t)p) & 7) == 0) {
      *reinterpret_cast<uint64_t*>(p) = v;
    } else {
      for (int b = 0; b < nb; ++b) p[b] = (uint8_t)(v >> (8 * b));
    }
  }
}

// Scale tensors: byte i of expert e = lo + (((word_i >> 32) * span) >> 32).
__global__ void fill_scale(uint8_t* __restrict__ dst, int64_t n_experts, int64_t bpe,
                           uint64_t seed, uint64_t layer, uint64_t tensor, uint32_t lo,
                           uint32_t span) {
  const int64_t total = n_experts * bpe;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i / bpe, b = i % bpe;
    const uint64_t key = stream_key(seed, layer, tensor, (uint64_t)e);
    const uint64_t v = mix64(key + (uint64_t)(b + 1) * kGamma);
    dst[i] = (uint8_t)(lo + (uint32_t)(((v >> 32) * span) >> 32));
  }
}

}  // namespace

extern "C" int synth_fill_expert_tensor(void* dst, int64_t n_experts, int64_t bytes_per_expert,
                                        uint64_t seed, int layer, int tensor, int is_scale,
                                        int lo, int span, void* stream) {
  if (!dst || n_experts <= 0 || bytes_per_expert <= 0) return (int)cudaErrorInvalidValue;
  cudaStream_t s = (cudaStream_t)stream;
  const int threads = 256;
  const int blocks = 152 * 8;
  if (is_scale)
    fill_scale<<<blocks, threads, 0, s>>>((uint8_t*)dst, n_experts, bytes_per_expert, seed,
                                          (uint64_t)layer, (uint64_t)tensor, (uint32_t)lo,
                                          (uint32_t)span);
  else
    fill_packed<<<blocks, threads, 0, s>>>((uint8_t*)dst, n_experts, bytes_per_expert, seed,
                                           (uint64_t)layer, (uint64_t)tensor);
  return (int)cudaGetLastError();
}

// Host-side evaluation of the same stream definition (no GPU needed): word i of the stream
// of (seed, layer, tensor, expert).  Lets a CPU test check that the device twin derives
// its keys exactly as the numpy twin does.
extern "C" uint64_t synth_host_word(uint64_t seed, int layer, int tensor, int64_t expert,
                                    int64_t i) {
  const uint64_t key = stream_key(seed, (uint64_t)layer, (uint64_t)tensor, (uint64_t)expert);
  return mix64(key + (uint64_t)(i + 1) * kGamma);
}

// Host fill of one expert's tensor (the same stream definition as the device kernels),
// for the test side, which needs only the experts a routing touches.
extern "C" void synth_host_fill_expert(uint8_t* dst, int64_t expert, int64_t bytes_per_expert,
                                       uint64_t seed, int layer, int tensor, int is_scale, int lo,
                                       int span) {
  const uint64_t key = stream_key(seed, (uint64_t)layer, (uint64_t)tensor, (uint64_t)expert);
  if (is_scale) {
    for (int64_t b = 0; b < bytes_per_expert; ++b) {
      const uint64_t v = mix64(key + (uint64_t)(b + 1) * kGamma);
      dst[b] = (uint8_t)(lo + (uint32_t)(((v >> 32) * (uint64_t)span) >> 32));
    }
  } else {
    for (int64_t w = 0; w * 8 < bytes_per_expert; ++w) {
      const uint64_t v = mix64(key + (uint64_t)(w + 1) * kGamma);
      const int64_t nb = (bytes_per_expert - w * 8) < 8 ? (bytes_per_expert - w * 8) : 8;
      for (int b = 0; b < nb; ++b) dst[w * 8 + b] = (uint8_t)(v >> (8 * b));
    }
  }
}
