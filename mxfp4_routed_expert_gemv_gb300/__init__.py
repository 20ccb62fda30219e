"""Python binding of libk3moe.so, the MXFP4 routed-expert MoE layer for one GB300.

Argument marshalling only: every step of the layer runs in the library's CUDA kernels
(sm_103a).  The functions carry the C ABI's names (include/k3moe.h) and take torch CUDA
tensors; PyTorch supplies device memory and streams, nothing else.  There is no CPU path:
importing works anywhere, but the first call loads libk3moe.so (building it with nvcc when
it is missing or stale) and raises if that fails.

The layer (README "kimi-k3-in-c", Part II section 9; expert format Part II section 4;
shapes from "K3_ARTIFACT_AUDIT" section 4.3):
  router logits h . Wr  ->  sigmoid scores (+ bias for selection)  ->  top-k, gates
  -> per chosen expert: act(W1 x, W3 x) -> W2  ->  gate-weighted sum y.
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Optional

from . import build as _build

__all__ = [
    "K3moeError", "Cfg", "Experts", "KIMI_K3", "lib", "workspace", "workspace_host",
    "k3moe_workspace_size", "k3moe_workspace_size_host", "k3moe_route", "k3moe_experts_mxfp4",
    "k3moe_layer", "k3moe_layer_host", "k3moe_matvec_mxfp4", "k3moe_stack_link",
    "k3moe_launch_count", "k3moe_strerror", "k3moe_abi_version", "k3moe_set_phase_events",
    "k3moe_layer_static_scratch", "STATIC_SCRATCH_BYTES", "EXPORTED_SYMBOLS",
    "Latent", "k3moe_latent_workspace_size", "latent_workspace", "k3moe_latent_layer",
    "k3moe_set_flag_wait_polls", "k3moe_last_error", "k3moe_experts_mxfp4_range", "expert_block",
    "k3moe_layer_host_async", "ExpertCache", "k3moe_layer_cached", "SLOT_EMPTY", "SLOT_INFLIGHT",
    "k3moe_cache_reset", "k3moe_cache_plan", "k3moe_cache_publish", "k3moe_cache_workspace_size",
    "k3moe_cache_host_scratch_size",
]

EXPORTED_SYMBOLS = (
    "k3moe_workspace_size", "k3moe_workspace_size_host", "k3moe_route", "k3moe_experts_mxfp4",
    "k3moe_layer", "k3moe_layer_host", "k3moe_matvec_mxfp4", "k3moe_stack_link",
    "k3moe_launch_count", "k3moe_strerror", "k3moe_abi_version", "k3moe_set_phase_events",
    "k3moe_layer_static_scratch", "k3moe_latent_workspace_size", "k3moe_latent_layer",
    "k3moe_set_flag_wait_polls", "k3moe_last_error", "k3moe_experts_mxfp4_range",
    "k3moe_layer_host_async", "k3moe_cache_reset", "k3moe_cache_plan", "k3moe_cache_publish",
    "k3moe_cache_workspace_size", "k3moe_cache_host_scratch_size", "k3moe_layer_cached",
)

# Capacity of the library's file-scope scratch array (K3MOE_STATIC_SCRATCH_BYTES).
STATIC_SCRATCH_BYTES = 16 << 20

ACT_SWIGLU, ACT_SITU = 0, 1


class K3moeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        detail = f"; {k3moe_last_error()}" if status == 5 else ""
        super().__init__(f"{fn} failed: {status} ({k3moe_strerror(status)}{detail})")


class _CCfg(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("topk", ctypes.c_int32),
        ("latent", ctypes.c_int32), ("inter", ctypes.c_int32), ("group", ctypes.c_int32),
        ("renorm", ctypes.c_int32), ("routed_scale", ctypes.c_float), ("act", ctypes.c_int32),
        ("situ_b1", ctypes.c_float), ("situ_b2", ctypes.c_float),
    ]


class _CExperts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w1_packed", "w1_scale", "w3_packed", "w3_scale", "w2_packed", "w2_scale")]


class _CExpertCache(ctypes.Structure):
    _fields_ = [("n_experts", ctypes.c_int32), ("n_slots", ctypes.c_int32), ("host", _CExperts),
                ("slots", _CExperts), ("expert_of", ctypes.c_void_p), ("slot_of", ctypes.c_void_p),
                ("used_at", ctypes.c_void_p), ("clock", ctypes.c_uint64)]


SLOT_EMPTY, SLOT_INFLIGHT = -1, -2


@dataclasses.dataclass(frozen=True)
class Cfg:
    """k3moe_cfg.  Defaults are the Kimi K3 layer with the workloads' routed scale 2.5."""

    hidden: int = 7168
    n_experts: int = 896
    topk: int = 16
    latent: int = 3584
    inter: int = 3072
    group: int = 32
    renorm: int = 1
    routed_scale: float = 2.5
    act: int = ACT_SWIGLU
    situ_b1: float = 4.0
    situ_b2: float = 25.0

    def c(self) -> _CCfg:
        return _CCfg(self.hidden, self.n_experts, self.topk, self.latent, self.inter, self.group,
                     self.renorm, self.routed_scale, self.act, self.situ_b1, self.situ_b2)


KIMI_K3 = Cfg()


@dataclasses.dataclass
class Experts:
    """Stacked expert tensors (torch uint8, device), checkpoint row layout:
    w1p/w3p [E, I, L/2], w1s/w3s [E, I, L/32], w2p [E, L, I/2], w2s [E, L, I/32]."""

    w1p: "object"
    w1s: "object"
    w3p: "object"
    w3s: "object"
    w2p: "object"
    w2s: "object"

    def c(self) -> _CExperts:
        return _CExperts(*(t.data_ptr() for t in (self.w1p, self.w1s, self.w3p, self.w3s, self.w2p, self.w2s)))

    @classmethod
    def from_dict(cls, d) -> "Experts":
        return cls(d["w1p"], d["w1s"], d["w3p"], d["w3s"], d["w2p"], d["w2s"])

    def block(self, e0: int, e1: int) -> "Experts":
        """Experts e0 .. e1-1 (views of the stacked tensors, no copy)."""
        return Experts(*(t[e0:e1] for t in (self.w1p, self.w1s, self.w3p, self.w3s, self.w2p, self.w2s)))


def expert_block(n_experts: int, world: int, rank: int):
    """The contiguous block [e0, e1) of experts that rank `rank` of `world` holds under expert
    parallelism: rank r takes experts floor(E r / N) .. floor(E (r+1) / N) - 1 (every expert on
    exactly one rank; block sizes differ by at most one).  Host logic only."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("rank out of range")
    return (n_experts * rank) // world, (n_experts * (rank + 1)) // world


class _CLatent(ctypes.Structure):
    _fields_ = [("down", ctypes.c_void_p), ("up", ctypes.c_void_p),
                ("latent_norm_w", ctypes.c_void_p), ("latent_norm", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("n_shared", ctypes.c_int32),
                ("sh1", ctypes.c_void_p), ("sh3", ctypes.c_void_p), ("sh2", ctypes.c_void_p)]


@dataclasses.dataclass
class Latent:
    """The LatentMoE wrapper's dense tensors (torch, device; bf16 unless noted):
    down [L, H], up [H, L], latent_norm_w fp32 [L] or None, sh1/sh3 [n_shared*I, H],
    sh2 [H, n_shared*I] (None when n_shared == 0)."""

    down: "object"
    up: "object"
    latent_norm_w: "object" = None
    latent_norm: bool = True
    rms_eps: float = 1e-5
    n_shared: int = 0
    sh1: "object" = None
    sh3: "object" = None
    sh2: "object" = None

    def c(self) -> _CLatent:
        return _CLatent(_p(self.down), _p(self.up), _p(self.latent_norm_w), int(bool(self.latent_norm)),
                        float(self.rms_eps), int(self.n_shared), _p(self.sh1), _p(self.sh3), _p(self.sh2))


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libk3moe.so (built from csrc/ with nvcc for sm_103a if needed)."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        pc, pe = ctypes.POINTER(_CCfg), ctypes.POINTER(_CExperts)
        L.k3moe_workspace_size.argtypes = [pc, i32, ctypes.POINTER(sz)]
        L.k3moe_workspace_size_host.argtypes = [pc, i32, ctypes.POINTER(sz)]
        L.k3moe_route.argtypes = [pc, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp]
        L.k3moe_experts_mxfp4.argtypes = [pc, pe, vp, vp, vp, i32, vp, vp, vp, sz, vp]
        L.k3moe_experts_mxfp4_range.argtypes = [pc, pe, i32, i32, vp, vp, vp, i32, vp, vp, vp, sz, vp]
        L.k3moe_layer.argtypes = [pc, vp, vp, vp, pe, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        L.k3moe_layer_host.argtypes = [pc, vp, vp, vp, pe, vp, i32, vp, vp, vp, sz, vp]
        L.k3moe_layer_host_async.argtypes = [pc, vp, vp, vp, pe, vp, i32, vp, vp, vp, sz, vp]
        L.k3moe_layer_static_scratch.argtypes = [pc, vp, vp, vp, pe, vp, i32, vp, vp, vp, vp, vp, vp]
        L.k3moe_matvec_mxfp4.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp]
        pl = ctypes.POINTER(_CLatent)
        L.k3moe_latent_workspace_size.argtypes = [pc, pl, i32, ctypes.POINTER(sz)]
        L.k3moe_latent_layer.argtypes = [pc, pl, vp, vp, vp, pe, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        L.k3moe_stack_link.argtypes = [vp, i32, i32, i32, ctypes.c_float, vp, vp, vp]
        L.k3moe_set_phase_events.restype = ctypes.c_int
        L.k3moe_set_phase_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32]
        L.k3moe_launch_count.restype = ctypes.c_int64
        L.k3moe_set_flag_wait_polls.restype = ctypes.c_int
        L.k3moe_set_flag_wait_polls.argtypes = [ctypes.c_int64]
        L.k3moe_launch_count.argtypes = []
        L.k3moe_last_error.restype = ctypes.c_char_p
        L.k3moe_last_error.argtypes = []
        pcc = ctypes.POINTER(_CExpertCache)
        L.k3moe_cache_reset.argtypes = [pcc]
        L.k3moe_cache_plan.argtypes = [pcc, vp, i32, vp, vp, vp, ctypes.POINTER(i32)]
        L.k3moe_cache_publish.argtypes = [pcc, vp, vp, i32, i32]
        L.k3moe_cache_workspace_size.argtypes = [pc, i32, ctypes.POINTER(sz)]
        L.k3moe_cache_host_scratch_size.argtypes = [pc, i32, i32, ctypes.POINTER(sz)]
        L.k3moe_layer_cached.argtypes = [pc, pcc, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp, sz,
                                         ctypes.POINTER(i32), vp]
        L.k3moe_strerror.restype = ctypes.c_char_p
        L.k3moe_strerror.argtypes = [ctypes.c_int]
        L.k3moe_abi_version.restype = i32
        L.k3moe_abi_version.argtypes = []
        for n in ("k3moe_workspace_size", "k3moe_workspace_size_host", "k3moe_route",
                  "k3moe_experts_mxfp4", "k3moe_experts_mxfp4_range", "k3moe_layer", "k3moe_layer_host", "k3moe_matvec_mxfp4",
                  "k3moe_stack_link", "k3moe_layer_static_scratch", "k3moe_latent_workspace_size",
                  "k3moe_latent_layer"):
            getattr(L, n).restype = ctypes.c_int
        _lib = L
    return _lib


def _p(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _check(fn: str, rc: int):
    if rc != 0:
        raise K3moeError(fn, rc)


def _expect(t, name, dtype, shape, cuda=True):
    import torch
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not cuda and t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    return t


def k3moe_strerror(status: int) -> str:
    return lib().k3moe_strerror(int(status)).decode()


def k3moe_last_error() -> str:
    """The last CUDA failure an entry point saw on this thread ("" if none)."""
    return lib().k3moe_last_error().decode()


def k3moe_abi_version() -> int:
    return int(lib().k3moe_abi_version())


def k3moe_launch_count() -> int:
    return int(lib().k3moe_launch_count())


def k3moe_set_flag_wait_polls(polls: int) -> None:
    """How many polls a wait on another CTA's flag makes before giving up (status[1] counts
    it); negative restores the default, 0 makes such waits give up at once."""
    _check("k3moe_set_flag_wait_polls", lib().k3moe_set_flag_wait_polls(int(polls)))


def k3moe_set_phase_events(events) -> None:
    """events: six torch.cuda.Event (created with enable_timing) or None to switch off."""
    if events is None:
        _check("k3moe_set_phase_events", lib().k3moe_set_phase_events(None, 0))
        return
    handles = [e.cuda_event for e in events]
    if not all(handles):
        raise ValueError("record each event once before passing it (torch creates events lazily)")
    arr = (ctypes.c_void_p * len(events))(*handles)
    _check("k3moe_set_phase_events", lib().k3moe_set_phase_events(arr, len(events)))


def k3moe_workspace_size(cfg: Cfg, T: int) -> int:
    n = ctypes.c_size_t(0)
    c = cfg.c()
    _check("k3moe_workspace_size", lib().k3moe_workspace_size(ctypes.byref(c), int(T), ctypes.byref(n)))
    return int(n.value)


def k3moe_workspace_size_host(cfg: Cfg, T: int) -> int:
    n = ctypes.c_size_t(0)
    c = cfg.c()
    _check("k3moe_workspace_size_host", lib().k3moe_workspace_size_host(ctypes.byref(c), int(T), ctypes.byref(n)))
    return int(n.value)


def workspace(cfg: Cfg, T: int, device="cuda"):
    """A device workspace (uint8 tensor) for T tokens."""
    import torch
    return torch.empty(k3moe_workspace_size(cfg, T), dtype=torch.uint8, device=device)


class ExpertCache:
    """A device cache of `n_slots` experts over a store of all E experts in host memory
    (k3moe_expert_cache): the state arrays live here (numpy), the store and the slots are
    Experts (host: page-locked CPU tensors [E, ...]; slots: device tensors [n_slots, ...]).
    Without store and slots only the host planning (plan, publish) can be used."""

    def __init__(self, n_experts: int, n_slots: int, host: Optional[Experts] = None,
                 slots: Optional[Experts] = None):
        import numpy as np
        self.n_experts, self.n_slots = int(n_experts), int(n_slots)
        self.host, self.slots = host, slots
        self.expert_of = np.full(self.n_slots, SLOT_EMPTY, np.int32)
        self.slot_of = np.full(self.n_experts, -1, np.int32)
        self.used_at = np.zeros(self.n_slots, np.uint64)
        self._c = _CExpertCache(self.n_experts, self.n_slots,
                                host.c() if host is not None else _CExperts(),
                                slots.c() if slots is not None else _CExperts(),
                                self.expert_of.ctypes.data, self.slot_of.ctypes.data,
                                self.used_at.ctypes.data, 0)
        self.reset()

    @classmethod
    def with_slots(cls, host: Experts, n_slots: int, device="cuda") -> "ExpertCache":
        """Device slots shaped like the store's experts, n_slots of them."""
        import torch
        slots = Experts(*(torch.empty((n_slots, *t.shape[1:]), dtype=t.dtype, device=device)
                          for t in (host.w1p, host.w1s, host.w3p, host.w3s, host.w2p, host.w2s)))
        return cls(host.w1p.shape[0], n_slots, host, slots)

    @property
    def clock(self) -> int:
        return int(self._c.clock)

    def reset(self) -> None:
        k3moe_cache_reset(self)

    def plan(self, idx):
        return k3moe_cache_plan(self, idx)

    def publish(self, fetch_expert, fetch_slot, n_ok: Optional[int] = None) -> None:
        k3moe_cache_publish(self, fetch_expert, fetch_slot, n_ok)

    def workspace(self, cfg: Cfg, T: int, device="cuda"):
        import torch
        return torch.empty(k3moe_cache_workspace_size(cfg, T), dtype=torch.uint8, device=device)

    def host_scratch(self, cfg: Cfg, T: int):
        import torch
        n = k3moe_cache_host_scratch_size(cfg, T, self.n_slots)
        return torch.empty((n + 3) // 4, dtype=torch.int32).pin_memory()


def k3moe_cache_reset(cache: ExpertCache) -> None:
    _check("k3moe_cache_reset", lib().k3moe_cache_reset(ctypes.byref(cache._c)))


def k3moe_cache_plan(cache: ExpertCache, idx):
    """Host planning of one call (int32 indices): (slot_idx, fetch_expert, fetch_slot); the
    fetched slots stay in flight until k3moe_cache_publish."""
    import numpy as np
    idx = np.ascontiguousarray(idx, dtype=np.int32).reshape(-1)
    slot_idx = np.empty_like(idx)
    fe = np.empty(cache.n_slots, np.int32)
    fs = np.empty(cache.n_slots, np.int32)
    nf = ctypes.c_int32(0)
    _check("k3moe_cache_plan", lib().k3moe_cache_plan(
        ctypes.byref(cache._c), idx.ctypes.data, idx.size, slot_idx.ctypes.data, fe.ctypes.data,
        fs.ctypes.data, ctypes.byref(nf)))
    return slot_idx, fe[:nf.value].copy(), fs[:nf.value].copy()


def k3moe_cache_publish(cache: ExpertCache, fetch_expert, fetch_slot, n_ok: Optional[int] = None) -> None:
    import numpy as np
    fe = np.ascontiguousarray(fetch_expert, dtype=np.int32)
    fs = np.ascontiguousarray(fetch_slot, dtype=np.int32)
    n_ok = fe.size if n_ok is None else n_ok
    _check("k3moe_cache_publish", lib().k3moe_cache_publish(
        ctypes.byref(cache._c), fe.ctypes.data, fs.ctypes.data, fe.size, int(n_ok)))


def k3moe_cache_workspace_size(cfg: Cfg, T: int) -> int:
    n = ctypes.c_size_t(0)
    _check("k3moe_cache_workspace_size",
           lib().k3moe_cache_workspace_size(ctypes.byref(cfg.c()), T, ctypes.byref(n)))
    return n.value


def k3moe_cache_host_scratch_size(cfg: Cfg, T: int, n_slots: int) -> int:
    n = ctypes.c_size_t(0)
    _check("k3moe_cache_host_scratch_size", lib().k3moe_cache_host_scratch_size(
        ctypes.byref(cfg.c()), T, n_slots, ctypes.byref(n)))
    return n.value


def k3moe_layer_cached(cfg: Cfg, cache: ExpertCache, h, wr, bias, x, y, status, ws, host_scratch,
                       stream=None) -> int:
    """The layer with its experts in the cache (synchronises); returns the experts copied."""
    import torch
    T = h.shape[0]
    _expect(h, "h", torch.bfloat16, (T, cfg.hidden))
    _expect(wr, "wr", torch.bfloat16, (cfg.n_experts, cfg.hidden))
    _expect(x, "x", torch.bfloat16, (T, cfg.latent))
    _expect(y, "y", torch.float32, (T, cfg.latent))
    n = ctypes.c_int32(0)
    c = cfg.c()
    _check("k3moe_layer_cached", lib().k3moe_layer_cached(
        ctypes.byref(c), ctypes.byref(cache._c), _p(h), _p(wr), _p(bias), _p(x), T, _p(y), _p(status),
        _p(ws), ws.numel(), _p(host_scratch), host_scratch.numel() * 4, ctypes.byref(n),
        _stream(stream)))
    return n.value


def workspace_host(cfg: Cfg, T: int, device="cuda"):
    import torch
    return torch.empty(k3moe_workspace_size_host(cfg, T), dtype=torch.uint8, device=device)


def k3moe_route(cfg: Cfg, h, wr, bias, idx, gate, gap, ws, stream=None) -> None:
    import torch
    T = h.shape[0]
    _expect(h, "h", torch.bfloat16, (T, cfg.hidden))
    _expect(wr, "wr", torch.bfloat16, (cfg.n_experts, cfg.hidden))
    if bias is not None:
        _expect(bias, "bias", torch.float32, (cfg.n_experts,))
    _expect(idx, "idx", torch.int32, (T, cfg.topk))
    _expect(gate, "gate", torch.float32, (T, cfg.topk))
    if gap is not None:
        _expect(gap, "gap", torch.float32, (T,))
    c = cfg.c()
    _check("k3moe_route", lib().k3moe_route(ctypes.byref(c), _p(h), _p(wr), _p(bias), T, _p(idx), _p(gate),
                                            _p(gap), _p(ws), ws.numel(), _stream(stream)))


def k3moe_experts_mxfp4(cfg: Cfg, experts: Experts, x, idx, gate, y, status, ws, stream=None) -> None:
    import torch
    T = x.shape[0]
    _expect(x, "x", torch.bfloat16, (T, cfg.latent))
    _expect(idx, "idx", torch.int32, (T, cfg.topk))
    _expect(gate, "gate", torch.float32, (T, cfg.topk))
    _expect(y, "y", torch.float32, (T, cfg.latent))
    if status is not None:
        _expect(status, "status", torch.int32, (4,))
    c, e = cfg.c(), experts.c()
    _check("k3moe_experts_mxfp4", lib().k3moe_experts_mxfp4(
        ctypes.byref(c), ctypes.byref(e), _p(x), _p(idx), _p(gate), T, _p(y), _p(status), _p(ws),
        ws.numel(), _stream(stream)))


def k3moe_experts_mxfp4_range(cfg: Cfg, experts: Experts, e0: int, e1: int, x, idx, gate, y, status,
                              ws, stream=None) -> None:
    """The routed sum over experts [e0, e1) only; `experts` holds that block (Experts.block)."""
    import torch
    T = x.shape[0]
    _expect(x, "x", torch.bfloat16, (T, cfg.latent))
    _expect(idx, "idx", torch.int32, (T, cfg.topk))
    _expect(gate, "gate", torch.float32, (T, cfg.topk))
    _expect(y, "y", torch.float32, (T, cfg.latent))
    if status is not None:
        _expect(status, "status", torch.int32, (4,))
    c, e = cfg.c(), experts.c()
    _check("k3moe_experts_mxfp4_range", lib().k3moe_experts_mxfp4_range(
        ctypes.byref(c), ctypes.byref(e), int(e0), int(e1), _p(x), _p(idx), _p(gate), T, _p(y),
        _p(status), _p(ws), ws.numel(), _stream(stream)))


def k3moe_layer(cfg: Cfg, h, wr, bias, experts: Experts, x, y, idx=None, gate=None, gap=None,
                status=None, ws=None, stream=None) -> None:
    import torch
    T = h.shape[0]
    _expect(h, "h", torch.bfloat16, (T, cfg.hidden))
    _expect(wr, "wr", torch.bfloat16, (cfg.n_experts, cfg.hidden))
    if bias is not None:
        _expect(bias, "bias", torch.float32, (cfg.n_experts,))
    _expect(x, "x", torch.bfloat16, (T, cfg.latent))
    _expect(y, "y", torch.float32, (T, cfg.latent))
    if idx is not None:
        _expect(idx, "idx", torch.int32, (T, cfg.topk))
    if gate is not None:
        _expect(gate, "gate", torch.float32, (T, cfg.topk))
    if gap is not None:
        _expect(gap, "gap", torch.float32, (T,))
    if status is not None:
        _expect(status, "status", torch.int32, (4,))
    if ws is None:
        raise ValueError("ws (workspace) is required")
    c, e = cfg.c(), experts.c()
    _check("k3moe_layer", lib().k3moe_layer(
        ctypes.byref(c), _p(h), _p(wr), _p(bias), ctypes.byref(e), _p(x), T, _p(y), _p(idx), _p(gate),
        _p(gap), _p(status), _p(ws), ws.numel(), _stream(stream)))


def k3moe_layer_static_scratch(cfg: Cfg, h, wr, bias, experts: Experts, x, y, idx=None, gate=None,
                               gap=None, status=None, stream=None) -> None:
    """k3moe_layer without a workspace, for callers that cannot allocate device memory
    (for example a host framework whose allocator owns all of it).  The library's own
    16 MiB device array serves as scratch; it is shared by every call on the device, so
    calls must be ordered on one stream.  Raises K3moeError (status 8) when the batch needs
    more scratch than the array holds."""
    import torch
    T = h.shape[0]
    _expect(h, "h", torch.bfloat16, (T, cfg.hidden))
    _expect(wr, "wr", torch.bfloat16, (cfg.n_experts, cfg.hidden))
    if bias is not None:
        _expect(bias, "bias", torch.float32, (cfg.n_experts,))
    _expect(x, "x", torch.bfloat16, (T, cfg.latent))
    _expect(y, "y", torch.float32, (T, cfg.latent))
    if idx is not None:
        _expect(idx, "idx", torch.int32, (T, cfg.topk))
    if gate is not None:
        _expect(gate, "gate", torch.float32, (T, cfg.topk))
    if gap is not None:
        _expect(gap, "gap", torch.float32, (T,))
    if status is not None:
        _expect(status, "status", torch.int32, (4,))
    c, e = cfg.c(), experts.c()
    _check("k3moe_layer_static_scratch", lib().k3moe_layer_static_scratch(
        ctypes.byref(c), _p(h), _p(wr), _p(bias), ctypes.byref(e), _p(x), T, _p(y), _p(idx), _p(gate),
        _p(gap), _p(status), _stream(stream)))


def _layer_host(fn, cfg: Cfg, h_host, wr, bias, experts: Experts, x_host, y_host, status, ws, stream):
    import torch
    T = h_host.shape[0]
    _expect(h_host, "h_host", torch.bfloat16, (T, cfg.hidden), cuda=False)
    _expect(x_host, "x_host", torch.bfloat16, (T, cfg.latent), cuda=False)
    _expect(y_host, "y_host", torch.float32, (T, cfg.latent), cuda=False)
    _expect(wr, "wr", torch.bfloat16, (cfg.n_experts, cfg.hidden))
    c, e = cfg.c(), experts.c()
    _check(fn, getattr(lib(), fn)(
        ctypes.byref(c), _p(h_host), _p(wr), _p(bias), ctypes.byref(e), _p(x_host), T, _p(y_host),
        _p(status), _p(ws), ws.numel(), _stream(stream)))


def k3moe_layer_host(cfg: Cfg, h_host, wr, bias, experts: Experts, x_host, y_host, status, ws,
                     stream=None) -> None:
    """The layer with host (ideally pinned) h, x and y; synchronises the stream."""
    _layer_host("k3moe_layer_host", cfg, h_host, wr, bias, experts, x_host, y_host, status, ws, stream)


def k3moe_layer_host_async(cfg: Cfg, h_host, wr, bias, experts: Experts, x_host, y_host, status,
                           ws, stream=None) -> None:
    """k3moe_layer_host that returns once the layer is enqueued (when h, x and y are mapped
    page-locked host buffers); y_host is ready when the stream reaches this point."""
    _layer_host("k3moe_layer_host_async", cfg, h_host, wr, bias, experts, x_host, y_host, status, ws,
                stream)


def k3moe_matvec_mxfp4(y, x, packed, scales, stream=None) -> None:
    """y[rows] = W x for one MXFP4 matrix W (packed [rows, in/2], scales [rows, in/32])."""
    import torch
    n_in = x.shape[0]
    rows = packed.shape[0]
    _expect(x, "x", torch.bfloat16, (n_in,))
    _expect(packed, "packed", torch.uint8, (rows, n_in // 2))
    _expect(scales, "scales", torch.uint8, (rows, n_in // 32))
    _expect(y, "y", torch.float32, (rows,))
    _check("k3moe_matvec_mxfp4", lib().k3moe_matvec_mxfp4(_p(y), _p(x), _p(packed), _p(scales), n_in,
                                                          rows, 32, _stream(stream)))


def k3moe_stack_link(y, x_out, h_out=None, norm: bool = True, eps: float = 1e-5, stream=None) -> None:
    import torch
    T, L = y.shape
    _expect(y, "y", torch.float32, (T, L))
    _expect(x_out, "x_out", torch.bfloat16, (T, L))
    if h_out is not None:
        _expect(h_out, "h_out", torch.bfloat16, (T, 2 * L))
    _check("k3moe_stack_link", lib().k3moe_stack_link(_p(y), T, L, 1 if norm else 0, float(eps), _p(x_out),
                                                      _p(h_out), _stream(stream)))


def k3moe_latent_workspace_size(cfg: Cfg, lat: Latent, T: int) -> int:
    n = ctypes.c_size_t(0)
    c, la = cfg.c(), lat.c()
    _check("k3moe_latent_workspace_size",
           lib().k3moe_latent_workspace_size(ctypes.byref(c), ctypes.byref(la), int(T), ctypes.byref(n)))
    return int(n.value)


def latent_workspace(cfg: Cfg, lat: Latent, T: int, device="cuda"):
    """A device workspace (uint8 tensor) of k3moe_latent_layer for T tokens."""
    import torch
    return torch.empty(k3moe_latent_workspace_size(cfg, lat, T), dtype=torch.uint8, device=device)


def k3moe_latent_layer(cfg: Cfg, lat: Latent, h, wr, bias, experts: Experts, out, idx=None,
                       gate=None, gap=None, status=None, ws=None, stream=None) -> None:
    """The LatentMoE layer (README Part II section 9, k3_moe): route on h, the routed experts
    on z = bf16(down . h), RMSNorm of their sum, up-projection, plus the shared experts on h."""
    import torch
    T = h.shape[0]
    H, L = cfg.hidden, cfg.latent
    SI = cfg.inter * lat.n_shared
    _expect(h, "h", torch.bfloat16, (T, H))
    _expect(wr, "wr", torch.bfloat16, (cfg.n_experts, H))
    if bias is not None:
        _expect(bias, "bias", torch.float32, (cfg.n_experts,))
    _expect(lat.down, "down", torch.bfloat16, (L, H))
    _expect(lat.up, "up", torch.bfloat16, (H, L))
    if lat.latent_norm_w is not None:
        _expect(lat.latent_norm_w, "latent_norm_w", torch.float32, (L,))
    if lat.n_shared > 0:
        _expect(lat.sh1, "sh1", torch.bfloat16, (SI, H))
        _expect(lat.sh3, "sh3", torch.bfloat16, (SI, H))
        _expect(lat.sh2, "sh2", torch.bfloat16, (H, SI))
    _expect(out, "out", torch.float32, (T, H))
    if idx is not None:
        _expect(idx, "idx", torch.int32, (T, cfg.topk))
    if gate is not None:
        _expect(gate, "gate", torch.float32, (T, cfg.topk))
    if gap is not None:
        _expect(gap, "gap", torch.float32, (T,))
    if status is not None:
        _expect(status, "status", torch.int32, (4,))
    if ws is None:
        raise ValueError("ws (workspace) is required")
    c, la, e = cfg.c(), lat.c(), experts.c()
    _check("k3moe_latent_layer", lib().k3moe_latent_layer(
        ctypes.byref(c), ctypes.byref(la), _p(h), _p(wr), _p(bias), ctypes.byref(e), T, _p(out),
        _p(idx), _p(gate), _p(gap), _p(status), _p(ws), ws.numel(), _stream(stream)))
