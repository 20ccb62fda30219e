"""The ORACLE of the MXFP4 routed-expert MoE layer -- TEST INFRASTRUCTURE ONLY.

A numpy-facing ctypes wrapper over ``k3o.c``: plain scalar fp64 C that states what the
layer computes (router, MXFP4 mat-vec, expert FFN, routed sum, RMSNorm).  Only the test
suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference legs may
import this package.  It imports nothing from the CUDA library and the CUDA library imports
nothing from it.

Sources (cited by page title and section):
  * "kimi-k3-in-c" README, Part II section 4 (MXFP4 format and mat-vec), section 5
    (RMSNorm), section 9 (router and the per-token MoE).
  * "K3_ARTIFACT_AUDIT" (llm-atlas), section 4.3 (expert tensor shapes, group 32).

Every function here checks its arguments and raises ``ValueError`` on anything the C code
would refuse.  All floating outputs are float64.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Mapping, Optional

import numpy as np

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int),
        ("n_experts", ctypes.c_int),
        ("topk", ctypes.c_int),
        ("latent", ctypes.c_int),
        ("inter", ctypes.c_int),
        ("group", ctypes.c_int),
        ("renorm", ctypes.c_int),
        ("routed_scale", ctypes.c_double),
        ("act", ctypes.c_int),
        ("situ_b1", ctypes.c_double),
        ("situ_b2", ctypes.c_double),
    ]


class _Expert(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w1p", "w1s", "w3p", "w3s", "w2p", "w2s")]


@dataclasses.dataclass(frozen=True)
class Cfg:
    """Layer configuration (the README's config struct plus the audit's expert shapes)."""

    hidden: int = 7168
    n_experts: int = 896
    topk: int = 16
    latent: int = 3584
    inter: int = 3072
    group: int = 32
    renorm: int = 1
    routed_scale: float = 2.5
    act: int = 0  # 0 SwiGLU, 1 SiTU-GLU
    situ_b1: float = 4.0
    situ_b2: float = 25.0

    def c(self) -> _Cfg:
        return _Cfg(self.hidden, self.n_experts, self.topk, self.latent, self.inter,
                    self.group, self.renorm, float(self.routed_scale), self.act,
                    float(self.situ_b1), float(self.situ_b2))


_lib = None


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    if _lib is None:
        # K3O_LIB points the wrapper at another build of k3o.c; the mutation tests use it to
        # load deliberately broken copies and check that the pins reject them.
        path = os.environ.get("K3O_LIB") or _build.build()
        L = ctypes.CDLL(path)
        d, i, vp = ctypes.c_double, ctypes.c_int, ctypes.c_void_p
        L.k3o_e2m1.restype, L.k3o_e2m1.argtypes = d, [i]
        L.k3o_e8m0.restype, L.k3o_e8m0.argtypes = d, [i]
        L.k3o_bf16_value.restype, L.k3o_bf16_value.argtypes = d, [ctypes.c_uint16]
        L.k3o_bf16_from_f32.restype, L.k3o_bf16_from_f32.argtypes = ctypes.c_uint16, [ctypes.c_float]
        L.k3o_matvec_mxfp4.restype = None
        L.k3o_matvec_mxfp4.argtypes = [vp, vp, vp, vp, i, i, i]
        L.k3o_dequant_mxfp4.restype = None
        L.k3o_dequant_mxfp4.argtypes = [vp, vp, vp, i, i, i]
        L.k3o_route.restype = i
        L.k3o_route.argtypes = [ctypes.POINTER(_Cfg), vp, vp, vp, i, vp, vp, vp, vp, vp]
        L.k3o_gates_for.restype = None
        L.k3o_gates_for.argtypes = [ctypes.POINTER(_Cfg), vp, vp, vp]
        L.k3o_activation.restype = None
        L.k3o_activation.argtypes = [ctypes.POINTER(_Cfg), vp, vp, vp, i]
        L.k3o_expert_ffn.restype = i
        L.k3o_expert_ffn.argtypes = [ctypes.POINTER(_Cfg), ctypes.POINTER(_Expert), vp, vp]
        L.k3o_experts.restype = i
        L.k3o_experts.argtypes = [ctypes.POINTER(_Cfg), ctypes.POINTER(_Expert), i, vp, vp, vp, i, vp]
        L.k3o_rmsnorm.restype = None
        L.k3o_rmsnorm.argtypes = [vp, vp, i, ctypes.c_double]
        L.k3o_rmsnorm_w.restype = None
        L.k3o_rmsnorm_w.argtypes = [vp, vp, vp, i, ctypes.c_double]
        L.k3o_matvec_bf16.restype = None
        L.k3o_matvec_bf16.argtypes = [vp, vp, vp, i, i]
        L.k3o_latent_moe.restype = i
        L.k3o_latent_moe.argtypes = [ctypes.POINTER(_Cfg), ctypes.POINTER(_Latent), vp, vp, vp,
                                     ctypes.POINTER(_Expert), i, i, vp, vp, vp]
        L.k3o_threads.restype, L.k3o_threads.argtypes = i, []
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype, shape=None, name="array"):
    a = np.ascontiguousarray(a, dtype=dtype)
    if shape is not None and tuple(a.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(a.shape)}")
    return a


# ---- number formats -------------------------------------------------------------------

def e2m1(code: int) -> float:
    return lib().k3o_e2m1(int(code))


def e8m0(byte: int) -> float:
    return lib().k3o_e8m0(int(byte))


def bf16_value(bits: int) -> float:
    return lib().k3o_bf16_value(int(bits) & 0xFFFF)


def bf16_from_f32(v: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (round to nearest even), element by element."""
    f = lib().k3o_bf16_from_f32
    v = np.asarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    flat_in, flat_out = v.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = f(float(flat_in[i]))
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact float64 values (a 16-bit shift into fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ---- MXFP4 mat-vec --------------------------------------------------------------------

def matvec_mxfp4(x: np.ndarray, packed: np.ndarray, scales: np.ndarray, group: int = 32) -> np.ndarray:
    """y = W x for W[rows][in] in MXFP4 (packed [rows][ceil(in/2)], scales [rows][ceil(in/group)])."""
    x = _c(x, np.float64, name="x")
    n_in = x.shape[0]
    rows = packed.shape[0]
    packed = _c(packed, np.uint8, (rows, (n_in + 1) // 2), "packed")
    scales = _c(scales, np.uint8, (rows, (n_in + group - 1) // group), "scales")
    y = np.empty(rows, dtype=np.float64)
    lib().k3o_matvec_mxfp4(_ptr(y), _ptr(x), _ptr(packed), _ptr(scales), n_in, rows, group)
    return y


def dequant_mxfp4(packed: np.ndarray, scales: np.ndarray, n_in: int, group: int = 32) -> np.ndarray:
    """The dense fp64 matrix W [rows, n_in] of an MXFP4 matrix: W = E2M1[nibble] * 2^(s-127),
    a scale byte of 255 zeroing its group (README Part II section 4)."""
    rows = packed.shape[0]
    packed = _c(packed, np.uint8, (rows, (n_in + 1) // 2), "packed")
    scales = _c(scales, np.uint8, (rows, (n_in + group - 1) // group), "scales")
    w = np.empty((rows, n_in), dtype=np.float64)
    lib().k3o_dequant_mxfp4(_ptr(w), _ptr(packed), _ptr(scales), n_in, rows, group)
    return w


# ---- router ---------------------------------------------------------------------------

@dataclasses.dataclass
class Routing:
    idx: np.ndarray   # int32 [T, k], descending selection score, lower index wins a tie
    gate: np.ndarray  # float64 [T, k]
    gap: np.ndarray   # float64 [T]: k-th minus (k+1)-th selection score
    sc: np.ndarray    # float64 [T, E]: unbiased sigmoid scores
    ch: np.ndarray    # float64 [T, E]: selection scores (sc + bias)


def route(cfg: Cfg, h: np.ndarray, wr: np.ndarray, bias: Optional[np.ndarray]) -> Routing:
    """Router for T tokens.  h: bf16 bits [T, H]; wr: bf16 bits [E, H]; bias fp32 [E] or None."""
    T = h.shape[0]
    h = _c(h, np.uint16, (T, cfg.hidden), "h")
    wr = _c(wr, np.uint16, (cfg.n_experts, cfg.hidden), "wr")
    if bias is not None:
        bias = _c(bias, np.float32, (cfg.n_experts,), "bias")
    idx = np.empty((T, cfg.topk), dtype=np.int32)
    gate = np.empty((T, cfg.topk), dtype=np.float64)
    gap = np.empty(T, dtype=np.float64)
    sc = np.empty((T, cfg.n_experts), dtype=np.float64)
    ch = np.empty((T, cfg.n_experts), dtype=np.float64)
    c = cfg.c()
    rc = lib().k3o_route(ctypes.byref(c), _ptr(h), _ptr(wr), _ptr(bias), T, _ptr(idx), _ptr(gate),
                         _ptr(gap), _ptr(sc), _ptr(ch))
    if rc != 0:
        raise ValueError(f"k3o_route failed with code {rc}")
    return Routing(idx, gate, gap, sc, ch)


def gates_for(cfg: Cfg, sc_row: np.ndarray, idx_row: np.ndarray) -> np.ndarray:
    """Gates of a given index list from one token's unbiased scores."""
    sc_row = _c(sc_row, np.float64, (cfg.n_experts,), "sc")
    idx_row = _c(idx_row, np.int32, (cfg.topk,), "idx")
    if idx_row.min() < 0 or idx_row.max() >= cfg.n_experts:
        raise ValueError("index out of range")
    gate = np.empty(cfg.topk, dtype=np.float64)
    c = cfg.c()
    lib().k3o_gates_for(ctypes.byref(c), _ptr(sc_row), _ptr(idx_row), _ptr(gate))
    return gate


# ---- experts --------------------------------------------------------------------------

@dataclasses.dataclass
class ExpertBytes:
    """One expert's six tensors in checkpoint row layout (uint8 numpy arrays)."""

    w1p: np.ndarray  # [I, L/2]
    w1s: np.ndarray  # [I, L/group]
    w3p: np.ndarray  # [I, L/2]
    w3s: np.ndarray  # [I, L/group]
    w2p: np.ndarray  # [L, I/2]
    w2s: np.ndarray  # [L, I/group]

    def checked(self, cfg: Cfg) -> "ExpertBytes":
        L, I, G = cfg.latent, cfg.inter, cfg.group
        return ExpertBytes(
            _c(self.w1p, np.uint8, (I, (L + 1) // 2), "w1p"),
            _c(self.w1s, np.uint8, (I, (L + G - 1) // G), "w1s"),
            _c(self.w3p, np.uint8, (I, (L + 1) // 2), "w3p"),
            _c(self.w3s, np.uint8, (I, (L + G - 1) // G), "w3s"),
            _c(self.w2p, np.uint8, (L, (I + 1) // 2), "w2p"),
            _c(self.w2s, np.uint8, (L, (I + G - 1) // G), "w2s"),
        )


def _expert_struct(ex: Optional[ExpertBytes]) -> _Expert:
    if ex is None:
        return _Expert()
    return _Expert(*(a.ctypes.data for a in (ex.w1p, ex.w1s, ex.w3p, ex.w3s, ex.w2p, ex.w2s)))


def activation(cfg: Cfg, g: np.ndarray, u: np.ndarray) -> np.ndarray:
    g = _c(g, np.float64, name="g")
    u = _c(u, np.float64, g.shape, "u")
    out = np.empty_like(g)
    c = cfg.c()
    lib().k3o_activation(ctypes.byref(c), _ptr(g), _ptr(u), _ptr(out), g.size)
    return out


def expert_ffn(cfg: Cfg, ex: ExpertBytes, x: np.ndarray) -> np.ndarray:
    """o = W2 act(W1 x, W3 x) for one fp64 latent vector x [L]."""
    ex = ex.checked(cfg)
    x = _c(x, np.float64, (cfg.latent,), "x")
    o = np.empty(cfg.latent, dtype=np.float64)
    c = cfg.c()
    st = _expert_struct(ex)
    rc = lib().k3o_expert_ffn(ctypes.byref(c), ctypes.byref(st), _ptr(x), _ptr(o))
    if rc != 0:
        raise ValueError(f"k3o_expert_ffn failed with code {rc}")
    return o


def experts(cfg: Cfg, table: Mapping[int, ExpertBytes], x: np.ndarray, idx: np.ndarray,
            gate: np.ndarray) -> np.ndarray:
    """y[t] = sum_j gate[t,j] * FFN_{idx[t,j]}(x[t]) in fp64.  x: bf16 bits [T, L]."""
    T = x.shape[0]
    x = _c(x, np.uint16, (T, cfg.latent), "x")
    idx = _c(idx, np.int32, (T, cfg.topk), "idx")
    gate = _c(gate, np.float64, (T, cfg.topk), "gate")
    checked = {int(e): ex.checked(cfg) for e, ex in table.items()}  # keeps arrays alive
    arr = (_Expert * cfg.n_experts)()
    for e, ex in checked.items():
        if not 0 <= e < cfg.n_experts:
            raise ValueError(f"expert id {e} out of range")
        arr[e] = _expert_struct(ex)
    y = np.empty((T, cfg.latent), dtype=np.float64)
    c = cfg.c()
    rc = lib().k3o_experts(ctypes.byref(c), arr, cfg.n_experts, _ptr(x), _ptr(idx), _ptr(gate), T, _ptr(y))
    if rc != 0:
        raise ValueError(f"k3o_experts failed with code {rc} (missing expert or bad index)")
    return y


def experts_dense(cfg: Cfg, table: Mapping[int, ExpertBytes], x: np.ndarray, idx: np.ndarray,
                  gate: np.ndarray) -> np.ndarray:
    """The routed sum of ``experts`` for large batches, fp64, in another arrangement of the
    same definition: each chosen expert's three matrices are expanded to dense fp64
    (``dequant_mxfp4``) and all of its tokens go through them at once with a library matmul
    (g = X W1^T, u = X W3^T, act, o = act W2^T); y[t] then sums gate[t, j] * o in slot order
    j = 0..k-1.  Only the order of the fp64 additions differs from ``experts`` (rounding
    order, about 1e-15 relative).  An index outside [0, E) raises, as in ``experts``."""
    T = x.shape[0]
    L, I, G = cfg.latent, cfg.inter, cfg.group
    x = _c(x, np.uint16, (T, L), "x")
    idx = _c(idx, np.int32, (T, cfg.topk), "idx")
    gate = _c(gate, np.float64, (T, cfg.topk), "gate")
    if T and (idx.min() < 0 or idx.max() >= cfg.n_experts):
        raise ValueError("expert index out of range")
    xd = bf16_to_f64(x)
    o = np.zeros((T, cfg.topk, L), dtype=np.float64)
    for e in np.unique(idx):
        e = int(e)
        if e not in table:
            raise ValueError(f"expert {e} missing from the table")
        ex = table[e].checked(cfg)
        tok, slot = np.nonzero(idx == e)
        xe = xd[tok]
        g = xe @ dequant_mxfp4(ex.w1p, ex.w1s, L, G).T
        u = xe @ dequant_mxfp4(ex.w3p, ex.w3s, L, G).T
        a = activation(cfg, g, u)
        o[tok, slot] = a @ dequant_mxfp4(ex.w2p, ex.w2s, I, G).T
    y = np.zeros((T, L), dtype=np.float64)
    for j in range(cfg.topk):
        y += gate[:, j:j + 1] * o[:, j]
    return y


def rmsnorm(x: np.ndarray, eps: float) -> np.ndarray:
    x = _c(x, np.float64, name="x")
    out = np.empty_like(x)
    lib().k3o_rmsnorm(_ptr(out), _ptr(x), x.size, float(eps))
    return out


def stack_link(y: np.ndarray, norm: bool, eps: float = 1e-5):
    """Next-layer inputs of the 8-layer stack from a layer output y [T, L] (fp64).

    y is first rounded to fp32 (the layer's output type).  With ``norm`` each token is
    RMS-normalised with unit weight (eps inside the square root), in fp64, then rounded to
    fp32.  The result is rounded to bf16 (nearest even) and becomes x; h is x tiled twice
    along the feature axis.  Returns (x_bits [T, L], h_bits [T, 2L]) as uint16.
    """
    y32 = np.asarray(y, dtype=np.float64).astype(np.float32)
    T, L = y32.shape
    v = np.empty((T, L), dtype=np.float32)
    for t in range(T):
        row = y32[t].astype(np.float64)
        v[t] = (rmsnorm(row, eps) if norm else row).astype(np.float32)
    xb = bf16_from_f32(v)
    hb = np.concatenate([xb, xb], axis=1)
    return xb, hb


def rmsnorm_w(x: np.ndarray, w: Optional[np.ndarray], eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w (w fp32, or None for unit weight), fp64."""
    x = _c(x, np.float64, name="x")
    wv = None if w is None else _c(w, np.float32, (x.size,), "w")
    out = np.empty_like(x)
    lib().k3o_rmsnorm_w(_ptr(out), _ptr(x), _ptr(wv), x.size, float(eps))
    return out


def matvec_bf16(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """y[r] = sum_c W[r, c] x[c] in fp64; W: bf16 bits [rows, in]."""
    W = _c(W, np.uint16, name="W")
    rows, n = W.shape
    x = _c(x, np.float64, (n,), "x")
    y = np.empty(rows, dtype=np.float64)
    lib().k3o_matvec_bf16(_ptr(y), _ptr(x), _ptr(W), n, rows)
    return y


@dataclasses.dataclass
class LatentWeights:
    """The LatentMoE wrapper's dense tensors (bf16 bits unless noted): down [L, H], up [H, L],
    norm_w fp32 [L] or None, sh1/sh3 [n_shared*I, H], sh2 [H, n_shared*I]."""
    down: np.ndarray
    up: np.ndarray
    norm_w: Optional[np.ndarray] = None
    latent_norm: bool = True
    rms_eps: float = 1e-5
    n_shared: int = 0
    sh1: Optional[np.ndarray] = None
    sh3: Optional[np.ndarray] = None
    sh2: Optional[np.ndarray] = None


class _Latent(ctypes.Structure):
    _fields_ = [("down", ctypes.c_void_p), ("up", ctypes.c_void_p), ("norm_w", ctypes.c_void_p),
                ("latent_norm", ctypes.c_int), ("rms_eps", ctypes.c_double),
                ("n_shared", ctypes.c_int), ("sh1", ctypes.c_void_p), ("sh3", ctypes.c_void_p),
                ("sh2", ctypes.c_void_p)]


def latent_moe(cfg: Cfg, lw: LatentWeights, h: np.ndarray, wr: np.ndarray,
               bias: Optional[np.ndarray], table: Mapping[int, ExpertBytes]):
    """The LatentMoE layer (README Part II section 9, k3_moe) for T tokens, fp64.

    h: bf16 bits [T, H].  Returns (out fp64 [T, H], idx [T, k], gate [T, k])."""
    T = h.shape[0]
    H, L, SI = cfg.hidden, cfg.latent, cfg.inter * lw.n_shared
    h = _c(h, np.uint16, (T, H), "h")
    wr = _c(wr, np.uint16, (cfg.n_experts, H), "wr")
    bias = None if bias is None else _c(bias, np.float32, (cfg.n_experts,), "bias")
    keep = [_c(lw.down, np.uint16, (L, H), "down"), _c(lw.up, np.uint16, (H, L), "up"),
            None if lw.norm_w is None else _c(lw.norm_w, np.float32, (L,), "norm_w")]
    if lw.n_shared > 0:
        keep += [_c(lw.sh1, np.uint16, (SI, H), "sh1"), _c(lw.sh3, np.uint16, (SI, H), "sh3"),
                 _c(lw.sh2, np.uint16, (H, SI), "sh2")]
    else:
        keep += [None, None, None]
    st = _Latent(_ptr(keep[0]), _ptr(keep[1]), _ptr(keep[2]), int(bool(lw.latent_norm)),
                 float(lw.rms_eps), int(lw.n_shared), _ptr(keep[3]), _ptr(keep[4]), _ptr(keep[5]))
    checked = {int(e): ex.checked(cfg) for e, ex in table.items()}
    arr = (_Expert * cfg.n_experts)()
    for e, ex in checked.items():
        arr[e] = _expert_struct(ex)
    out = np.empty((T, H), dtype=np.float64)
    idx = np.empty((T, cfg.topk), dtype=np.int32)
    gate = np.empty((T, cfg.topk), dtype=np.float64)
    c = cfg.c()
    rc = lib().k3o_latent_moe(ctypes.byref(c), ctypes.byref(st), _ptr(h), _ptr(wr), _ptr(bias),
                              arr, cfg.n_experts, T, _ptr(idx), _ptr(gate), _ptr(out))
    if rc != 0:
        raise ValueError(f"k3o_latent_moe failed with code {rc}")
    return out, idx, gate


def threads() -> int:
    return int(lib().k3o_threads())
