"""The C-ABI library without a GPU: it builds, loads, exports every entry point that
include/k3moe.h declares (and the Python binding has each name), and its host-side checks
refuse bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "k3moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(k3moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("k3moe_route", "k3moe_experts_mxfp4", "k3moe_layer", "k3moe_workspace_size",
              "k3moe_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import mxfp4_routed_expert_gemv_gb300 as k3
    lib = k3.lib()
    for n in _declared():
        assert hasattr(lib, n), n
        assert hasattr(k3, n), f"binding lacks {n}"
    assert set(_declared()) == set(k3.EXPORTED_SYMBOLS)
    assert k3.k3moe_abi_version() == 1
    assert k3.k3moe_strerror(4).startswith("workspace")


def test_library_has_no_oracle_dependency():
    """The CUDA path never links, loads or names the oracle."""
    import mxfp4_routed_expert_gemv_gb300 as k3
    pkg = os.path.dirname(k3.__file__)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "k3o_" not in text and "k3o.h" not in text, f


def test_workspace_sizes_and_config_checks():
    import mxfp4_routed_expert_gemv_gb300 as k3
    cfg = k3.KIMI_K3
    n1 = k3.k3moe_workspace_size(cfg, 1)
    n64 = k3.k3moe_workspace_size(cfg, 64)
    assert 0 < n1 < n64
    assert k3.k3moe_workspace_size_host(cfg, 64) > n64
    # act [T*k, I] + ybuf [T*k, L] dominate
    assert n64 >= 64 * 16 * (3072 + 3584) * 4
    for bad, code in ((dict(group=16), 2), (dict(topk=0), 1), (dict(topk=40, n_experts=896), 2),
                      (dict(n_experts=2000), 2), (dict(latent=3583), 2), (dict(inter=8192), 2),
                      (dict(hidden=7170), 2), (dict(renorm=2), 1), (dict(act=5), 1),
                      (dict(topk=20, n_experts=16), 1)):
        c = k3.Cfg(**{**k3.KIMI_K3.__dict__, **bad})
        with pytest.raises(k3.K3moeError) as ei:
            k3.k3moe_workspace_size(c, 4)
        assert ei.value.status == code, bad
    with pytest.raises(k3.K3moeError):
        k3.k3moe_workspace_size(cfg, -1)


def test_host_checks_refuse_null_pointers_without_cuda():
    import mxfp4_routed_expert_gemv_gb300 as k3
    lib = k3.lib()
    c = k3.KIMI_K3.c()
    # null inputs: refused before any CUDA call
    rc = lib.k3moe_route(ctypes.byref(c), None, None, None, 1, None, None, None, None, 0, None)
    assert rc == 1
    e = k3._CExperts()
    rc = lib.k3moe_experts_mxfp4(ctypes.byref(c), ctypes.byref(e), None, None, None, 1, None, None, None, 0, None)
    assert rc == 1
    rc = lib.k3moe_matvec_mxfp4(None, None, None, None, 64, 1, 32, None)
    assert rc == 1
    rc = lib.k3moe_matvec_mxfp4(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                48, 1, 32, None)
    assert rc == 2
    # misaligned expert pointer
    e = k3._CExperts(*([256] * 5 + [257]))
    rc = lib.k3moe_layer(ctypes.byref(c), ctypes.c_void_p(256), ctypes.c_void_p(256), None, ctypes.byref(e),
                         ctypes.c_void_p(256), 1, ctypes.c_void_p(256), None, None, None, None,
                         ctypes.c_void_p(256), 1 << 40, None)
    assert rc == 3
    # workspace too small / misaligned
    e = k3._CExperts(*([256] * 6))
    rc = lib.k3moe_layer(ctypes.byref(c), ctypes.c_void_p(256), ctypes.c_void_p(256), None, ctypes.byref(e),
                         ctypes.c_void_p(256), 1, ctypes.c_void_p(256), None, None, None, None,
                         ctypes.c_void_p(256), 16, None)
    assert rc == 4
    rc = lib.k3moe_layer(ctypes.byref(c), ctypes.c_void_p(256), ctypes.c_void_p(256), None, ctypes.byref(e),
                         ctypes.c_void_p(256), 1, ctypes.c_void_p(256), None, None, None, None,
                         ctypes.c_void_p(258), 1 << 40, None)
    assert rc == 4


def test_latent_workspace_and_checks_without_cuda():
    """The LatentMoE entry points' host-side checks (no device memory is touched: the size
    query only reads the pointers' values)."""
    import mxfp4_routed_expert_gemv_gb300 as k3
    cfg = k3.KIMI_K3
    L, H, I = cfg.latent, cfg.hidden, cfg.inter
    buf = torch.zeros(64, dtype=torch.uint8)  # any aligned non-null address
    lat = k3.Latent(down=buf, up=buf, n_shared=2, sh1=buf, sh3=buf, sh2=buf)
    n1 = k3.k3moe_latent_workspace_size(cfg, lat, 1)
    n4 = k3.k3moe_latent_workspace_size(cfg, lat, 4)
    # the layer's workspace plus z (bf16), the routed sum and its norm (fp32), act (fp32)
    assert n1 >= k3.k3moe_workspace_size(cfg, 1) + L * 2 + 2 * L * 4 + 2 * I * 4
    assert n4 > n1
    lat0 = k3.Latent(down=buf, up=buf, n_shared=0)
    assert k3.k3moe_latent_workspace_size(cfg, lat0, 1) < n1
    for bad, code in ((dict(down=None), 1), (dict(n_shared=-1), 1), (dict(sh2=None), 1),
                      (dict(rms_eps=-1.0), 1), (dict(n_shared=1000), 2)):
        b = k3.Latent(**{**lat.__dict__, **bad})
        with pytest.raises(k3.K3moeError) as ei:
            k3.k3moe_latent_workspace_size(cfg, b, 1)
        assert ei.value.status == code, bad
    raw = lat.c()
    raw.latent_norm = 2  # the C check itself (the binding passes a bool)
    n = ctypes.c_size_t(0)
    assert k3.lib().k3moe_latent_workspace_size(ctypes.byref(cfg.c()), ctypes.byref(raw), 1, ctypes.byref(n)) == 1
    # a null output is refused before any CUDA call
    lib = k3.lib()
    c, la, e = cfg.c(), lat.c(), k3._CExperts(*([buf.data_ptr()] * 6))
    rc = lib.k3moe_latent_layer(ctypes.byref(c), ctypes.byref(la), buf.data_ptr(), buf.data_ptr(), None,
                                ctypes.byref(e), 1, None, None, None, None, None, None, 0, None)
    assert rc == 1
    # T = 0: nothing to do
    rc = lib.k3moe_latent_layer(ctypes.byref(c), ctypes.byref(la), None, None, None, ctypes.byref(e), 0,
                                None, None, None, None, None, None, 0, None)
    assert rc == 0


def test_header_is_plain_c_and_cxx(tmp_path):
    """include/k3moe.h compiles as C99 and as C++17 with no CUDA header: the boundary uses
    plain pointers and sizes only."""
    import subprocess
    src = tmp_path / "use.c"
    src.write_text('#include "k3moe.h"\n'
                   'int main(void) { k3moe_cfg c; (void)c; k3moe_latent l; (void)l;\n'
                   '  return (int)(sizeof(k3moe_experts) > 0) - 1; }\n')
    inc = os.path.join(ROOT, "include")
    for cmd in (["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", inc, str(src)],
                ["g++", "-std=c++17", "-x", "c++", "-Wall", "-Werror", "-fsyntax-only", "-I", inc, str(src)]):
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
