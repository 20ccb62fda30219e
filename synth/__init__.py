"""Seeded synthetic inputs for the MXFP4 routed-expert MoE layer.

This module holds only input generation: it contains none of the layer's arithmetic.  Both
the oracle (through the tests and the benchmark) and the CUDA library receive the arrays it
makes.  Nothing here imports the oracle or the CUDA library.

Two kinds of tensors:

* Float tensors (router input h, router weight Wr, correction bias, expert input x) are
  small.  They are drawn on the host with numpy's Philox counter-based generator
  (``numpy.random.Philox``; Salmon et al., "Parallel random numbers: as easy as 1, 2, 3",
  SC'11) and its standard-normal sampler, as float32, then rounded to bf16 (nearest even)
  where the layer takes bf16.  The same arrays go to both sides.
* Expert bytes (packed E2M1 nibbles and E8M0 scales, 17,547,264 B per expert, about 15.7 GB
  per 896-expert layer) are too large to draw on the host.  They come from SplitMix64
  (S. Vigna, public domain; Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA'14) used as a counter-based generator: word i of a stream with key K
  is the SplitMix64 output function applied to K + (i+1)*0x9E3779B97F4A7C15.  The host twin
  below (numpy) and the device twin (``synth_dev.cu``) implement that one definition; a
  test checks that they give the same bytes.

Distributions (the five K3-shaped workloads):

* h ~ N(0, 1) bf16 [T, 7168]; Wr ~ N(0, 1/7168) bf16 [E, 7168]; x ~ N(0, 1) bf16 [T, 3584].
  The second parameter of N(.,.) is read as the variance, the reading under which
  N(0, 1/7168) gives unit-variance router logits.
* bias ~ N(0, 0.3) fp32 [E] (std sqrt(0.3)); the batched-decode workload adds exactly +1.5 to
  32 seeded distinct "hot" experts instead.
* packed bytes uniform over 0..255 (each nibble uniform over the 16 E2M1 codes);
  scale bytes uniform over the 9 integers 118..126.

The LatentMoE wrapper's dense tensors (the pages give them no distribution; these keep
every stage near unit scale): down ~ N(0, 1/H) bf16 [L, H] (so z has unit variance), up ~
N(0, 1/L) bf16 [H, L] (the normed aggregate has unit RMS), the aggregate's norm weight
1 + N(0, 0.01) fp32 [L], shared experts sh1, sh3 ~ N(0, 1/H) bf16 [S, H] and sh2 ~
N(0, 1/S) bf16 [H, S], S = n_shared * I.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_LAYER_MUL = np.uint64(0xD1B54A32D192ED03)

# tensor ids of the streams
W1P, W1S, W3P, W3S, W2P, W2S = 0, 1, 2, 3, 4, 5
T_H, T_WR, T_BIAS, T_X, T_HOT = 10, 11, 12, 13, 14
T_DOWN, T_UP, T_NORM, T_SH1, T_SH3, T_SH2 = 15, 16, 17, 18, 19, 20

SCALE_LO, SCALE_SPAN = 118, 9


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64's output function on uint64 arrays (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64_words(key: int, n: int, start: int = 0) -> np.ndarray:
    """Words start..start+n-1 of the stream with key ``key``."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + i * GAMMA)


def stream_key(seed: int, layer: int, tensor: int, expert: int = 0) -> int:
    """Key of one tensor's stream; the device twin derives it the same way."""
    with np.errstate(over="ignore"):
        k0 = mix64(np.array([seed], dtype=np.uint64) + GAMMA)
        k1 = mix64(k0 ^ (np.array([layer], dtype=np.uint64) * _LAYER_MUL))
        k2 = mix64(k1 ^ ((np.uint64(tensor) << np.uint64(40)) ^ np.uint64(expert)))
    return int(k2[0])


def packed_bytes(key: int, nbytes: int) -> np.ndarray:
    """nbytes uniform bytes: word i supplies bytes 8i..8i+7, least significant first."""
    w = splitmix64_words(key, (nbytes + 7) // 8)
    return w.astype("<u8").view(np.uint8)[:nbytes].copy()


def scale_bytes(key: int, n: int, lo: int = SCALE_LO, span: int = SCALE_SPAN) -> np.ndarray:
    """n bytes uniform over lo..lo+span-1: byte i = lo + (((word_i >> 32) * span) >> 32)."""
    w = splitmix64_words(key, n)
    v = ((w >> np.uint64(32)) * np.uint64(span)) >> np.uint64(32)
    return (np.uint64(lo) + v).astype(np.uint8)


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bit patterns, nearest even (inputs are finite)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_f32(key: int, shape, std: float) -> np.ndarray:
    g = np.random.Generator(np.random.Philox(key=key))
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


# ---- workloads ------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int                 # tokens
    E: int                 # experts
    k: int                 # experts per token
    bias: str              # "none" | "normal" | "hot"
    seed: int
    layers: int = 1
    hidden: int = 7168
    latent: int = 3584
    inter: int = 3072
    group: int = 32
    routed_scale: float = 2.5
    n_hot: int = 32
    hot_bias: float = 1.5
    bias_var: float = 0.3

    def layer_seed(self, layer: int) -> int:
        return self.seed if self.layers == 1 else self.seed * 1000 + layer

    @property
    def expert_bytes(self) -> int:
        L, I, G = self.latent, self.inter, self.group
        return 2 * (I * (L // 2) + I * (L // G)) + (L * (I // 2) + L * (I // G))


WORKLOADS: Dict[int, Workload] = {
    0: Workload("tiny: 4 tokens, 64 experts, top-8, no bias", T=4, E=64, k=8, bias="none", seed=0),
    1: Workload("batch-1 decode: 1 token, 896 experts, top-16", T=1, E=896, k=16, bias="normal", seed=1),
    2: Workload("batched decode: 64 tokens, 896 experts, top-16, 32 hot experts", T=64, E=896, k=16,
                bias="hot", seed=2),
    3: Workload("prefill: 4096 tokens, 896 experts, top-16", T=4096, E=896, k=16, bias="normal", seed=3),
    4: Workload("8-layer stack: 16 tokens, 896 experts, top-16", T=16, E=896, k=16, bias="normal",
                seed=4, layers=8),
}


def small_workload(T=3, E=12, k=4, latent=256, inter=192, hidden=512, bias="normal", seed=7) -> Workload:
    """A shape the oracle finishes in well under a second, still several tiles wide."""
    return Workload(f"small T={T} E={E} k={k} L={latent} I={inter} H={hidden}", T=T, E=E, k=k,
                    bias=bias, seed=seed, hidden=hidden, latent=latent, inter=inter)


@dataclasses.dataclass
class LayerInputs:
    h: np.ndarray                # uint16 bf16 bits [T, H]
    wr: np.ndarray               # uint16 bf16 bits [E, H]
    bias: Optional[np.ndarray]   # float32 [E] or None
    x: np.ndarray                # uint16 bf16 bits [T, L]
    hot: Optional[np.ndarray] = None  # int64 ids of hot experts (batched-decode workload)


def layer_inputs(w: Workload, layer: int = 0, T: Optional[int] = None) -> LayerInputs:
    """Host float inputs of one layer (h and x are those of the first layer of a stack)."""
    T = w.T if T is None else T
    s = w.layer_seed(layer)
    h = f32_to_bf16_bits(normal_f32(stream_key(s, layer, T_H), (T, w.hidden), 1.0))
    wr = f32_to_bf16_bits(normal_f32(stream_key(s, layer, T_WR), (w.E, w.hidden), (1.0 / w.hidden) ** 0.5))
    x = f32_to_bf16_bits(normal_f32(stream_key(s, layer, T_X), (T, w.latent), 1.0))
    bias, hot = None, None
    if w.bias != "none":
        bias = normal_f32(stream_key(s, layer, T_BIAS), (w.E,), w.bias_var ** 0.5)
        if w.bias == "hot":
            g = np.random.Generator(np.random.Philox(key=stream_key(s, layer, T_HOT)))
            hot = np.sort(g.choice(w.E, size=w.n_hot, replace=False))
            bias[hot] = np.float32(w.hot_bias)
    return LayerInputs(h, wr, bias, x, hot)


TENSOR_SHAPES = ("w1p", "w1s", "w3p", "w3s", "w2p", "w2s")


def expert_shapes(w: Workload):
    L, I, G = w.latent, w.inter, w.group
    return {
        "w1p": (I, L // 2), "w1s": (I, L // G),
        "w3p": (I, L // 2), "w3s": (I, L // G),
        "w2p": (L, I // 2), "w2s": (L, I // G),
    }


_TID = {"w1p": W1P, "w1s": W1S, "w3p": W3P, "w3s": W3S, "w2p": W2P, "w2s": W2S}


def expert_tensor_numpy(w: Workload, layer: int, expert: int, name: str) -> np.ndarray:
    """One tensor of one expert from the numpy statement of the generator (slow)."""
    shape = expert_shapes(w)[name]
    n = shape[0] * shape[1]
    key = stream_key(w.layer_seed(layer), layer, _TID[name], expert)
    if name.endswith("s"):
        return scale_bytes(key, n).reshape(shape)
    return packed_bytes(key, n).reshape(shape)


def expert_tensor(w: Workload, layer: int, expert: int, name: str) -> np.ndarray:
    """One tensor of one expert on the host (compiled host loop; same stream definition
    as the numpy statement above and the device kernels)."""
    shape = expert_shapes(w)[name]
    out = np.empty(shape, dtype=np.uint8)
    _dev_lib().synth_host_fill_expert(out.ctypes.data, expert, out.size, w.layer_seed(layer), layer,
                                      _TID[name], 1 if name.endswith("s") else 0, SCALE_LO, SCALE_SPAN)
    return out


def expert_host(w: Workload, layer: int, expert: int) -> Dict[str, np.ndarray]:
    return {n: expert_tensor(w, layer, expert, n) for n in TENSOR_SHAPES}


# ---- device twin ----------------------------------------------------------------------

_dev = None


def _dev_lib():
    global _dev
    if _dev is None:
        from . import build as _b
        path = _b.build()
        L = ctypes.CDLL(path)
        L.synth_fill_expert_tensor.restype = ctypes.c_int
        L.synth_fill_expert_tensor.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        L.synth_host_fill_expert.restype = None
        L.synth_host_fill_expert.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        _dev = L
    return _dev


def fill_expert_tensor_device(dst_ptr: int, n_experts: int, bytes_per_expert: int, w: Workload,
                              layer: int, name: str, stream_ptr: int = 0) -> None:
    """Fill a stacked [n_experts][bytes_per_expert] device buffer with one tensor kind."""
    is_scale = 1 if name.endswith("s") else 0
    rc = _dev_lib().synth_fill_expert_tensor(dst_ptr, n_experts, bytes_per_expert,
                                             w.layer_seed(layer), layer, _TID[name], is_scale,
                                             SCALE_LO, SCALE_SPAN, stream_ptr)
    if rc != 0:
        raise RuntimeError(f"synth_fill_expert_tensor failed: cuda error {rc}")


def experts_device(w: Workload, layer: int, device="cuda"):
    """All E experts of one layer on the device: dict of stacked uint8 torch tensors
    [E, rows, cols] in checkpoint row layout."""
    import torch
    out = {}
    stream = torch.cuda.current_stream(device).cuda_stream
    for name, (r, c) in expert_shapes(w).items():
        t = torch.empty((w.E, r, c), dtype=torch.uint8, device=device)
        fill_expert_tensor_device(t.data_ptr(), w.E, r * c, w, layer, name, stream)
        out[name] = t
    return out


@dataclasses.dataclass
class LatentWeights:
    down: np.ndarray               # uint16 bf16 bits [L, H]
    up: np.ndarray                 # uint16 bf16 bits [H, L]
    norm_w: np.ndarray             # float32 [L]
    n_shared: int
    sh1: Optional[np.ndarray]      # uint16 bf16 bits [S, H]
    sh3: Optional[np.ndarray]
    sh2: Optional[np.ndarray]      # uint16 bf16 bits [H, S]


def latent_weights(w: Workload, layer: int = 0, n_shared: int = 2) -> LatentWeights:
    """Host dense tensors of one layer's LatentMoE wrapper (distributions in the module
    docstring)."""
    s, H, L = w.layer_seed(layer), w.hidden, w.latent
    S = n_shared * w.inter

    def bf(tid, shape, var):
        return f32_to_bf16_bits(normal_f32(stream_key(s, layer, tid), shape, var ** 0.5))

    norm_w = (np.float32(1.0) + normal_f32(stream_key(s, layer, T_NORM), (L,), 0.1)).astype(np.float32)
    return LatentWeights(
        down=bf(T_DOWN, (L, H), 1.0 / H), up=bf(T_UP, (H, L), 1.0 / L), norm_w=norm_w,
        n_shared=n_shared,
        sh1=bf(T_SH1, (S, H), 1.0 / H) if S else None,
        sh3=bf(T_SH3, (S, H), 1.0 / H) if S else None,
        sh2=bf(T_SH2, (H, S), 1.0 / S) if S else None)
