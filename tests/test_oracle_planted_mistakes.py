"""Each plausible mistake planted in a copy of the oracle must make at least
one pin in test_oracle_pins.py fail.  The mistakes are planted in a temporary
copy of oracle/moe_oracle.c (the arithmetic) or of oracle/__init__.py (how
the layer strings the steps together) on the CPU; the committed oracle is
untouched."""
import os
import shutil
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MISTAKES = {
    "sign_dropped": ("double sgn = (c >> 7) ? -1.0 : 1.0;", "double sgn = 1.0;"),
    "scale_block_index": ("scales[(size_t)r * KB + (4 * q) / 128]",
                          "scales[(size_t)r * KB + ((4 * q) / 64) % KB]"),
    "codebook_component_order": ("fp16_value(cb[idx * 4 + i])", "fp16_value(cb[idx * 4 + (3 - i)])"),
    "silu_on_up": ("g[r] = g[r] / (1.0 + exp(-g[r])) * u[r];",
                   "g[r] = u[r] / (1.0 + exp(-u[r])) * g[r];"),
    "tie_to_higher_id": ("l[e] > l[best]", "l[e] >= l[best]"),
    "offsets_off_by_one": ("cursor[ids[p] + 1] += 1;", "cursor[ids[p]] += 1;"),
    "router_lane_mapping": ("int l = (h / 8) % 32;", "int l = h % 32;"),
    "softmax_denominator": ("den += exp((double)l[ids[(size_t)t * k + j]] - top);",
                            "den += exp((double)l[ids[(size_t)t * k]] - top);"),
    "e2m1_exponent_bias": ("ldexp(1.0 + 0.5 * m, ex - 1)", "ldexp(1.0 + 0.5 * m, ex)"),
    "combine_weight_index": ("o[h] += weights[p] * y[h];", "o[h] += weights[(size_t)t * k] * y[h];"),
    "fp4_nibble_order": ("unsigned nib = h ? (v >> 4) : (v & 15);",
                         "unsigned nib = h ? (v & 15) : (v >> 4);"),
    "bias_dropped": ("if (bias) s = s + bias[e];", "(void)bias;"),
    "permute_not_stable": ("    for (int p = 0; p < P; ++p) {\n        int s = cursor[ids[p]]++;",
                           "    for (int p = P - 1; p >= 0; --p) {\n        int s = cursor[ids[p]]++;"),
    "down_scales_from_up": ("decode_matrix(fmt, c_down, s_down, cb, H, I, Wd)",
                            "decode_matrix(fmt, c_down, s_up, cb, H, I, Wd)"),
    "fp4_scale_block_64": ("e8m0_value(scales[(size_t)r * KB + col / 32])",
                           "e8m0_value(scales[(size_t)r * KB + col / 64])"),
    "renormalize_ignored": ("if (renormalize)", "if (0)"),
    "fp16_subnormal_exponent": ("ldexp((double)fr, -24)", "ldexp((double)fr, -25)"),
    "butterfly_order_reversed": ("for (int off = 16; off >= 1; off /= 2)", "for (int off = 1; off <= 16; off *= 2)"),
    "up_uses_gate_codes": ("decode_matrix(fmt, c_up, s_up, cb, I, H, Wu)",
                           "decode_matrix(fmt, c_gate, s_up, cb, I, H, Wu)"),
    "ue8m0_bias_126": ("ldexp(1.0, (int)e - 127)", "ldexp(1.0, (int)e - 126)"),
    "vq2_index_six_bits": ("int idx = c & 127;", "int idx = c & 63;"),
    "e2m1_mantissa_quarter": ("ldexp(1.0 + 0.5 * m, ex - 1)", "ldexp(1.0 + 0.25 * m, ex - 1)"),
    "fp16_normal_exponent": ("ldexp((double)(1024 + fr), ex - 25)", "ldexp((double)(1024 + fr), ex - 24)"),
    "matvec_drops_last_input": ("for (int c = 0; c < K; ++c) s += w[c] * x[c];",
                                "for (int c = 0; c < K - 1; ++c) s += w[c] * x[c];"),
    "silu_sign": ("g[r] = g[r] / (1.0 + exp(-g[r])) * u[r];", "g[r] = g[r] / (1.0 + exp(g[r])) * u[r];"),
    "topk_excludes_nothing": ("taken[best] = 1;", "(void)taken;"),
}


@pytest.mark.parametrize("name", sorted(MISTAKES))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MISTAKES[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"pattern for {name} not found exactly once"
    mutated = tmp_path / "moe_oracle.c"
    mutated.write_text(src.replace(old, new))
    so = oracle.build(out=str(tmp_path / "libmutant.so"), src=str(mutated))
    env = dict(os.environ, MOE_ORACLE_LIB=so, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake {name} passed every pin:\n{r.stdout[-2000:]}"


# Mistakes in the layer's composition (oracle/__init__.py).
MISTAKES_PY = {
    "token_row_of_pair": ("X = xf[[p // k for p in pairs]]", "X = xf[[p % k for p in pairs]]"),
    "ypair_by_sorted_position": ("pairs = [int(sp[s]) for s in pairs]", "pairs = [int(s) for s in pairs]"),
    "remainder_is_partial": ("remainder = self.combine(wsel, ysel, 1 - inc_res[sel])",
                             "remainder = self.combine(wsel, ysel, inc_res[sel])"),
    "weights_not_selected": ("wsel = w[sel]", "wsel = w[:len(sel)]"),
}


@pytest.mark.parametrize("name", sorted(MISTAKES_PY))
def test_planted_composition_mistake_is_caught(name, tmp_path):
    old, new = MISTAKES_PY[name]
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    shutil.copy(SRC, pkg / "moe_oracle.c")
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert src.count(old) == 1, f"pattern for {name} not found exactly once"
    (pkg / "__init__.py").write_text(src.replace(old, new))
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([str(tmp_path), ROOT]))
    env.pop("MOE_ORACLE_LIB", None)
    # the pins must import the mutant package, not the committed one
    probe = subprocess.run([sys.executable, "-c", "import oracle; print(oracle.__file__)"], cwd=str(tmp_path),
                           env=env, capture_output=True, text=True, timeout=120)
    assert probe.stdout.strip().startswith(str(tmp_path)), probe.stdout + probe.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "--rootdir", str(tmp_path), os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=str(tmp_path), env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake {name} passed every pin:\n{r.stdout[-2000:]}"
