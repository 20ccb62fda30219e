"""GPU unit tests of the decode building blocks, through the C ABI: the standalone MXFP4
mat-vec (exact one-hot nibble and scale cases, random rows against the oracle), the stack
link, and the device twin of the input generator."""
import numpy as np
import pytest

import oracle
import synth
from _parity import from_dev_bf16, to_dev_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _k3():
    import mxfp4_routed_expert_gemv_gb300 as k3
    return k3


def _matvec(x_bits, packed, scales):
    k3 = _k3()
    y = torch.empty(packed.shape[0], dtype=torch.float32, device="cuda")
    k3.k3moe_matvec_mxfp4(y, to_dev_bf16(x_bits), torch.from_numpy(packed).cuda(), torch.from_numpy(scales).cuda())
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _bf16(v):
    return synth.f32_to_bf16_bits(np.asarray(v, dtype=np.float32))


def test_one_hot_nibble_positions_exact():
    """Every code at every position of a 64-wide row: catches a swapped nibble order or a
    misplaced half in the hardware pair conversion."""
    cols = 64
    x = np.zeros(cols, dtype=np.float32)
    x[:] = np.arange(1, cols + 1, dtype=np.float32)  # distinct, exact in bf16 and f16
    xb = _bf16(x)
    rows = []
    expect = []
    for col in range(cols):
        for code in range(16):
            row = np.zeros(cols // 2, dtype=np.uint8)
            row[col // 2] = code if col % 2 == 0 else code << 4
            rows.append(row)
            expect.append(oracle.e2m1(code) * float(x[col]))
    packed = np.stack(rows)
    scales = np.full((packed.shape[0], cols // 32), 127, dtype=np.uint8)
    y = _matvec(xb, packed, scales)
    assert np.array_equal(y, np.array(expect, dtype=np.float32))


def test_scale_bytes_exact():
    cols = 64
    xb = _bf16(np.ones(cols))
    packed = np.full((6, cols // 2), 0x22, dtype=np.uint8)  # every weight 1.0
    scales = np.array([[127, 127], [128, 126], [0, 127], [255, 127], [1, 200], [118, 126]], dtype=np.uint8)
    y = _matvec(xb, packed, scales)
    ref = [sum(32 * oracle.e8m0(int(s)) for s in row) for row in scales]
    assert np.array_equal(y, np.array(ref, dtype=np.float32))


@pytest.mark.parametrize("cols,rows", [(32, 3), (3584, 257), (3072, 100), (96, 7)])
def test_matvec_random_against_oracle(cols, rows):
    rng = np.random.default_rng(cols + rows)
    packed = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    scales = rng.integers(118, 127, size=(rows, cols // 32), dtype=np.uint8)
    scales[0, 0] = 255
    xb = _bf16(rng.standard_normal(cols) * 3)
    y = _matvec(xb, packed, scales)
    ref = oracle.matvec_mxfp4(oracle.bf16_to_f64(xb), packed, scales)
    np.testing.assert_allclose(y, ref, rtol=1e-5, atol=1e-6 * np.max(np.abs(ref)))


def test_matvec_large_dynamic_range_x():
    """x spanning 2^-20..2^20: the per-vector power-of-two scaling keeps every element whose
    magnitude is within 2^28 of the largest exact."""
    rng = np.random.default_rng(1)
    cols, rows = 256, 33
    x = rng.standard_normal(cols) * np.exp2(rng.integers(-20, 21, size=cols))
    xb = _bf16(x)
    packed = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    scales = rng.integers(110, 140, size=(rows, cols // 32), dtype=np.uint8)
    y = _matvec(xb, packed, scales)
    ref = oracle.matvec_mxfp4(oracle.bf16_to_f64(xb), packed, scales)
    scale = np.max(np.abs(ref))
    np.testing.assert_allclose(y, ref, rtol=1e-5, atol=1e-6 * scale)


@pytest.mark.parametrize("norm", [True, False])
def test_stack_link_against_oracle(norm):
    k3 = _k3()
    rng = np.random.default_rng(5)
    y = (rng.standard_normal((5, 3584)) * 1.6e4).astype(np.float32)
    yd = torch.from_numpy(y).cuda()
    xo = torch.empty((5, 3584), dtype=torch.bfloat16, device="cuda")
    ho = torch.empty((5, 7168), dtype=torch.bfloat16, device="cuda")
    k3.k3moe_stack_link(yd, xo, ho, norm=norm)
    torch.cuda.synchronize()
    xb_ref, hb_ref = oracle.stack_link(y.astype(np.float64), norm=norm)
    xg, hg = from_dev_bf16(xo), from_dev_bf16(ho)
    assert np.array_equal(hg[:, :3584], xg) and np.array_equal(hg[:, 3584:], xg)
    diff = np.abs(xg.astype(np.int32) - xb_ref.astype(np.int32))  # ulps of the same sign
    assert diff.max() <= 1 and np.mean(diff == 0) > 0.999


def test_device_generator_matches_host_twin():
    w = synth.WORKLOADS[1]
    small = synth.Workload("gen", T=1, E=5, k=2, bias="none", seed=w.seed)
    d = synth.experts_device(small, 0)
    for e in (0, 3, 4):
        host = synth.expert_host(small, 0, e)
        for name, arr in host.items():
            assert np.array_equal(d[name][e].cpu().numpy(), arr), (e, name)
    assert np.array_equal(d["w2s"][1].cpu().numpy(), synth.expert_tensor_numpy(small, 0, 1, "w2s"))
