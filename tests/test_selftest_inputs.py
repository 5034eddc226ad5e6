"""The boot self-check's inputs and stored expected values (CPU only).

The library draws the self-check's inputs on the GPU from SplitMix64; the
expected values were written by ``oracle/make_selftest_golden.py`` from the
same draws made by ``moe_synth``.  Pinned here: the generator against the
published test vector, the value recipe's exactness, and the stored header
against a fresh run of the oracle script."""
import numpy as np

import moe_synth as ms


def test_splitmix64_published_vector():
    # Reference output of SplitMix64 seeded with 1234567 (the test vector that
    # accompanies Vigna's public-domain splitmix64.c): successive outputs are
    # the "first output" of the states seed + j * 0x9E3779B97F4A7C15.
    gamma = 0x9E3779B97F4A7C15
    states = np.array([(1234567 + j * gamma) % 2 ** 64 for j in range(5)], np.uint64)
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    assert [int(v) for v in ms.splitmix64(states)] == want


def test_draw_streams_are_keyed_by_tag_and_index():
    a = ms.st_draw(5, 10)
    assert int(a[3]) == int(ms.splitmix64(np.array([(5 << 32) | 3], np.uint64))[0])
    assert np.array_equal(ms.st_draw(1, 8, period=4)[4:], ms.st_draw(1, 8, period=4)[:4])


def test_bell_values_are_small_integers():
    g = ms.st_bell(ms.st_draw(2, 1 << 16))
    assert g.min() >= -126 and g.max() <= 126
    # four independent 6-bit fields: mean 0, variance 4 * (64^2 - 1) / 12
    assert abs(g.mean()) < 0.5
    assert abs(g.var() - 4 * (64 ** 2 - 1) / 12) < 40


def test_recipe_values_are_exact_in_their_formats():
    x = ms.selftest_tokens(8)
    f = ms.bf16_to_f32(x).astype(np.float64)
    assert np.array_equal(f * 32, np.round(f * 32))          # g / 32, no rounding
    assert np.abs(f * 32).max() <= 126
    assert np.array_equal(x[4:], x[:4])                       # rows repeat the four tokens
    L = ms.SelftestLayer(mixed=True)
    w = ms.bf16_to_f32(L.w_router).astype(np.float64) * 2048
    assert np.array_equal(w, np.round(w))
    cb = L.codebook.view(np.float16).astype(np.float64) * 32
    assert np.array_equal(cb, np.round(cb))
    vq = L.expert(0)
    s = vq.scales[0].view(np.float16).astype(np.float64) * 8192
    assert np.array_equal(s, np.round(s)) and s.min() >= 40 and s.max() <= 163
    fp = L.expert(1)
    assert fp.fmt == ms.FMT_FP4 and vq.fmt == ms.FMT_VQ2
    assert fp.scales[2].min() >= 118 and fp.scales[2].max() <= 120
    assert [c.shape for c in fp.codes] == [(128, 128), (128, 128), (256, 64)]


def test_stored_expected_values_match_the_oracle_script():
    from oracle import make_selftest_golden as mk
    with open(mk.HEADER) as f:
        stored = f.read()
    assert stored == mk.render(), "selftest_expected.h is stale: rerun python -m oracle.make_selftest_golden"
