"""Each plausible mistake planted in a copy of the oracle must make at least
one pin in test_oracle_pins.py fail.  The mistakes are planted in a temporary
copy of oracle/moe_oracle.c on the CPU; the committed oracle is untouched."""
import os
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
