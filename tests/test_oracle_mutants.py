"""Plant plausible mistakes in copies of the oracle and check that the pins catch each one.

Every mutant is a one-line change to a temporary copy of ``oracle/k3o.c``: a swapped
nibble order, an off-by-one exponent bias, a flipped tie rule, gates taken from the biased
score, a dropped renormalisation, a dropped group, a shifted scale or a neighbour's nibble in the dense expansion, gate and
up swapped in SwiGLU, w1 and w3
swapped, a transposed activation operand, and in the LatentMoE wrapper a dropped norm
weight, a transposed dense mat-vec, a mis-rounded latent, a skipped aggregate norm, weighted
or swapped shared experts.  ``tests/test_oracle_pins.py`` and ``tests/test_oracle_latent.py``
run against each mutant in a subprocess and must fail.  The oracle itself is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "k3o.c")

MUTANTS = {
    "nibble_swap": ("(col % 2 == 0) ? (byte & 15) : (byte >> 4)", "(col % 2 == 0) ? (byte >> 4) : (byte & 15)"),
    "scale_bias_off_by_one": ("ldexp(1.0, byte - 127)", "ldexp(1.0, byte - 126)"),
    "nan_scale_not_zero": ("if (byte == 255) return 0.0;", "if (byte == 256) return 0.0;"),
    "tie_to_higher_index": ("(best < 0 || cht[e] > cht[best])", "(best < 0 || cht[e] >= cht[best])"),
    "gates_from_selection_score": ("k3o_gates_for(c, sc + (size_t)t * E, it", "k3o_gates_for(c, ch + (size_t)t * E, it"),
    "no_renorm": ("if (c->renorm && sum > 0.0)", "if (0)"),
    "dropped_last_group": ("for (int g = 0; g < ngroup; g++) {", "for (int g = 0; g < ngroup - (ngroup > 1); g++) {"),
    "swiglu_gate_up_swapped": ("act[i] = g[i] * sigmoid(g[i]) * u[i];", "act[i] = u[i] * sigmoid(u[i]) * g[i];"),
    "w1_w3_swapped": ("k3o_matvec_mxfp4(g, x, ex->w1p, ex->w1s, L, I, G);", "k3o_matvec_mxfp4(g, x, ex->w3p, ex->w3s, L, I, G);"),
    "gap_wrong_sign": ("cht[it[K - 1]] - cht[rest]", "cht[rest] - cht[it[K - 1]]"),
    "bias_ignored": ("ch[te] = sc[te] + (bias ? (double)bias[e] : 0.0);", "ch[te] = sc[te];"),
    "situ_capped_sigmoid": ("tanh(g[i] / c->situ_b1) * sigmoid(g[i])", "tanh(g[i] / c->situ_b1) * sigmoid(tanh(g[i]))"),
    "rmsnorm_eps_outside": ("1.0 / sqrt(ss / (double)n + eps)", "1.0 / (sqrt(ss / (double)n) + eps)"),
    "rmsnorm_weight_dropped": ("x[i] * inv * (w ? (double)w[i] : 1.0)", "x[i] * inv"),
    "matvec_bf16_transposed": ("k3o_bf16_value(wr[c]) * x[c]", "k3o_bf16_value(W[(size_t)c * rows + r]) * x[c]"),
    "latent_z_misrounded": ("k3o_bf16_from_f32((float)zd[i])", "k3o_bf16_from_f32((float)(zd[i] * 1.0078125))"),
    "latent_norm_skipped": ("if (lw->latent_norm) k3o_rmsnorm_w", "if (0) k3o_rmsnorm_w"),
    "latent_shared_weighted": ("for (int i = 0; i < H; i++) ot[i] += o[i];", "for (int i = 0; i < H; i++) ot[i] += 0.5 * o[i];"),
    "dequant_scale_off_by_one": ("* k3o_e8m0(srow[col / group]);", "* k3o_e8m0(srow[col / group] + 1);"),
    "dequant_neighbour_column": ("wr[col] = k3o_e2m1(nibble_at(prow, col))", "wr[col] = k3o_e2m1(nibble_at(prow, col ^ 1))"),
    "latent_shared_gate_is_up": ("k3o_matvec_bf16(g, hd, lw->sh1, H, SI);", "k3o_matvec_bf16(g, hd, lw->sh3, H, SI);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    d = tmp_path / "mut"
    d.mkdir()
    shutil.copy(os.path.join(ROOT, "oracle", "k3o.h"), d / "k3o.h")
    (d / "k3o.c").write_text(src.replace(old, new))
    lib = str(d / "libk3o_mut.so")
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                    str(d / "k3o.c"), "-o", lib, "-lm"], check=True)
    env = dict(os.environ, K3O_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_latent.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
