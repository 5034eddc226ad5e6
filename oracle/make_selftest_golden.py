"""Writes the expected values of the library's boot self-check.

TEST INFRASTRUCTURE (part of the oracle).  The self-check (Tandem-vLLM page,
"New in 0.2.0": each kernel is checked against a reference at boot) runs the
tiny layer (hidden 256, intermediate 128, 8 experts, top-2, 4 tokens) on the
GPU from inputs it draws itself with SplitMix64, and compares what it gets
with the numbers this script stores in
``bit_vq_routed_gb300/csrc/selftest_expected.h``.  Those numbers come from
the CPU oracle alone, fed the same draws (``moe_synth.SelftestLayer``,
``moe_synth.selftest_tokens``); nothing here reads a GPU result.

    python -m oracle.make_selftest_golden          # rewrite the header
    python -m oracle.make_selftest_golden --check  # exit 1 if it is stale

Stored:
  * routing of the four tokens (the same router in both layers): logits as
    fp32 bit patterns, ids, softmax weights, expert_offsets, sorted_pair,
    pair_to_sorted;
  * out of the all-VQ2 layer, of the mixed layer (FP4 experts 1, 3, 5, 7),
    and the partial output of the all-VQ2 layer when experts 2 and 7 are not
    resident (the pairs of the resident experts only; Tandem-vLLM page, "How
    it works": nothing is skipped or substituted).
"""
from __future__ import annotations

import os
import sys

import numpy as np

import moe_synth as ms

from . import default as oracle

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(_ROOT, "bit_vq_routed_gb300", "csrc", "selftest_expected.h")
NOT_RESIDENT = (2, 7)


def compute():
    x = ms.selftest_tokens()
    vq2 = ms.SelftestLayer(mixed=False)
    mixed = ms.SelftestLayer(mixed=True)
    resident = np.ones(ms.SELFTEST_E, bool)
    resident[list(NOT_RESIDENT)] = False
    a = oracle.moe_layer(vq2, x, resident=resident)
    b = oracle.moe_layer(mixed, x)
    for key in ("logits", "ids", "offsets", "sorted_pair", "pair_to_sorted"):
        assert np.array_equal(a[key], b[key]), key
    ids = a["ids"]
    counts = np.bincount(ids.ravel(), minlength=ms.SELFTEST_E)
    routed = counts > 0
    fp4 = np.zeros(ms.SELFTEST_E, bool)
    fp4[list(ms.SELFTEST_FP4_EXPERTS)] = True
    # the draws must reach every branch the check is meant to cover
    assert (routed & fp4).any() and (routed & ~fp4).any(), "mixed layer routes one format only"
    assert (counts[~fp4] == 1).any() and (counts[~fp4] >= 2).any(), "no 1-token and multi-token VQ2 expert"
    assert (routed & ~resident).any() and (routed & resident).any(), "residency split is empty"
    return dict(logits=a["logits"], ids=ids, weights=a["weights"], offsets=a["offsets"],
                sorted_pair=a["sorted_pair"], pair_to_sorted=a["pair_to_sorted"],
                out_vq2=a["out"], partial_vq2=a["partial"], out_mixed=b["out"],
                resident=resident.astype(np.uint8))


def _ints(a) -> str:
    return ", ".join(str(int(v)) for v in np.asarray(a).ravel())


def _doubles(a, per_line=4) -> str:
    v = [format(float(x), ".17g") for x in np.asarray(a, np.float64).ravel()]
    lines = [", ".join(v[i:i + per_line]) for i in range(0, len(v), per_line)]
    return ",\n    ".join(lines)


def render() -> str:
    r = compute()
    T, E, k, H = ms.SELFTEST_T, ms.SELFTEST_E, ms.SELFTEST_K, ms.SELFTEST_H
    logit_bits = np.ascontiguousarray(r["logits"], np.float32).view(np.uint32)
    parts = [
        "/* Expected results of moe_selftest: the tiny routed-expert layer (hidden 256,",
        " * intermediate 128, 8 experts, top-2, 4 tokens) computed by the CPU oracle from",
        " * the SplitMix64 draws that the self-check makes on the GPU.",
        " * Written by oracle/make_selftest_golden.py; do not edit by hand. */",
        "#pragma once",
        "#include <stdint.h>",
        "",
        "namespace moe {",
        "namespace selftest_expected {",
        f"constexpr int T = {T}, H = {H}, I = {ms.SELFTEST_I}, E = {E}, K = {k};",
        f"static const uint32_t logits_bits[{T * E}] = {{{', '.join(hex(int(v)) for v in logit_bits.ravel())}}};",
        f"static const int32_t ids[{T * k}] = {{{_ints(r['ids'])}}};",
        f"static const double weights[{T * k}] = {{{_doubles(r['weights'], 8)}}};",
        f"static const int32_t expert_offsets[{E + 1}] = {{{_ints(r['offsets'])}}};",
        f"static const int32_t sorted_pair[{T * k}] = {{{_ints(r['sorted_pair'])}}};",
        f"static const int32_t pair_to_sorted[{T * k}] = {{{_ints(r['pair_to_sorted'])}}};",
        f"static const uint8_t resident[{E}] = {{{_ints(r['resident'])}}};",
        f"static const double out_vq2[{T * H}] = {{\n    {_doubles(r['out_vq2'])}}};",
        f"static const double partial_vq2[{T * H}] = {{\n    {_doubles(r['partial_vq2'])}}};",
        f"static const double out_mixed[{T * H}] = {{\n    {_doubles(r['out_mixed'])}}};",
        "}  // namespace selftest_expected",
        "}  // namespace moe",
        "",
    ]
    return "\n".join(parts)


def main(argv) -> int:
    text = render()
    if "--check" in argv:
        with open(HEADER) as f:
            same = f.read() == text
        print("up to date" if same else "stale: rerun python -m oracle.make_selftest_golden")
        return 0 if same else 1
    with open(HEADER, "w") as f:
        f.write(text)
    print(HEADER)
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
