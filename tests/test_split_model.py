"""The decode's segment-count model (host arithmetic, no GPU).

Lecture 11 (sections 6.3-6.4) chooses the number of key segments with a
CTA-by-wave model, and its exercise 9 works one case on an A100 (108 SMs, a
CTA streaming at most 80 GB/s, 1555 GB/s of HBM): batch 1, 64K keys, 2 KV
heads.  With 32 segments the 64 CTAs run in one wave, each at 1555 / 64 = 24
GB/s, under the per-CTA cap; with 64 segments the 128 CTAs exceed the 108 SMs
and need two waves, the second paying a whole wave's time for 20 CTAs.  So 32
segments are faster.  attn_decode_model_time / _best (include/attn_test.h)
are the library's model with the machine given as arguments; these tests
replay the exercise, check the model's terms, and pin the GB300 fit to the
counts that measured best.
"""
import math

import pytest

import exact_attention_62_gb300 as pkg

A100 = dict(slots=108, cta=80e9, hbm=1555e9)


@pytest.fixture(scope="module")
def L():
    return pkg.lib()


def t(L, units, slots, Nk, d, S, cta, hbm, fixed=0.0, merge=0.0):
    return L.attn_decode_model_time(units, slots, Nk, d, S, cta, hbm, fixed, merge)


def test_exercise_9_one_wave_of_64_ctas_beats_two_waves_of_128(L):
    units, Nk, d = 2, 65536, 128  # one CTA per KV head per segment (its 8 query heads together)
    t32 = t(L, units, A100["slots"], Nk, d, 32, A100["cta"], A100["hbm"])
    t64 = t(L, units, A100["slots"], Nk, d, 64, A100["cta"], A100["hbm"])
    assert t32 < t64
    # 32 segments: 64 CTAs in one wave, each streaming 2048 keys x 4d bytes at
    # 1555 / 64 = 24.3 GB/s (under the 80 GB/s cap); then the merge traffic
    merge32 = 2 * units * 8 * 32 * (d + 1) * 4 / A100["hbm"]
    assert t32 == pytest.approx(2048 * 4 * d / (A100["hbm"] / 64) + merge32, rel=1e-12)
    assert A100["hbm"] / 64 / 1e9 == pytest.approx(24.3, abs=0.05)
    # 64 segments: 128 CTAs > 108 SMs, two waves at 1555 / 108 GB/s each
    merge64 = 2 * units * 8 * 64 * (d + 1) * 4 / A100["hbm"]
    assert t64 == pytest.approx(2 * 1024 * 4 * d / (A100["hbm"] / 108) + merge64, rel=1e-12)
    # the model's own choice keeps every CTA in one wave
    best = L.attn_decode_model_best(units, A100["slots"], Nk, d, A100["cta"], A100["hbm"], 0.0, 0.0, 0)
    assert 1 <= best and units * best <= A100["slots"]
    assert t(L, units, A100["slots"], Nk, d, best, A100["cta"], A100["hbm"]) <= t32 * 1.005


def test_model_terms(L):
    # one segment: no merge term; the per-CTA cap binds when few CTAs run
    one = t(L, 4, 152, 8192, 128, 1, 60e9, 6e12)
    assert one == pytest.approx(8192 * 512 / 60e9, rel=1e-12)
    # fixed costs: one start-up per wave, one merge launch for S > 1
    assert t(L, 4, 152, 8192, 128, 1, 60e9, 6e12, fixed=1e-6) == pytest.approx(one + 1e-6, rel=1e-12)
    base = t(L, 4, 152, 8192, 128, 8, 60e9, 6e12)
    assert t(L, 4, 152, 8192, 128, 8, 60e9, 6e12, merge=3e-6) == pytest.approx(base + 3e-6, rel=1e-12)
    # 152 slots: 38 segments of 4 CTAs fill one wave, 39 need two
    rate = 6e12 / 152   # per CTA when all 152 slots stream (under the 60 GB/s cap)
    mrg = lambda S: 2 * 4 * 8 * S * 129 * 4 / 6e12
    w1 = t(L, 4, 152, 8192, 128, 38, 60e9, 6e12)
    w2 = t(L, 4, 152, 8192, 128, 39, 60e9, 6e12)
    assert w1 == pytest.approx(math.ceil(8192 / 38) * 512 / rate + mrg(38), rel=1e-12)
    assert w2 == pytest.approx(2 * math.ceil(8192 / 39) * 512 / rate + mrg(39), rel=1e-12)
    # single_wave caps the count at one wave of CTAs (and whole 64-key tiles)
    assert L.attn_decode_model_best(4, 152, 8192, 128, 1e9, 6e12, 0.0, 0.0, 1) == 38
    assert L.attn_decode_model_best(4, 152, 1000, 128, 1e9, 6e12, 0.0, 0.0, 1) == 16
    # invalid arguments
    assert t(L, 0, 152, 8192, 128, 1, 60e9, 6e12) == -1.0
    assert L.attn_decode_model_best(1, 0, 8192, 128, 60e9, 6e12, 0.0, 0.0, 0) == -1


@pytest.mark.parametrize("B,Nk,want", [(1, 2048, 12), (1, 8192, 12), (1, 16384, 12), (1, 65536, 12),
                                       (4, 4096, 3), (4, 16384, 3), (8, 8192, 2), (16, 8192, 1),
                                       (32, 2048, 1)])
def test_gb300_fit_picks_the_measured_counts(L, B, Nk, want):
    """The contiguous-cache constants (80 GB/s per CTA, 7.5 TB/s, 0.5 us per
    wave, 4 us merge) on 152 SMs, one CTA per SM, Hq = 32, Hkv = 8 (four
    query heads per CTA): counts that measured best or within 2% of it on
    GB300 with L2 flushed clean (µs, 22 calls each: B = 1 x 64K 45.9 at 12,
    45.7 at 16, 47.5 at 9; B = 1 x 8K 14.6 at 12, 15.0 at 9; B = 1 x 2K
    10.6 at 12, 10.4 at 9; B = 4 x 16K 46.0 at 3, 45.9 at 4, 57.5 at 5;
    B = 8 x 8K 46.0 at 2, 45.7 at 1; B = 16 x 8K 79.5 at 1, 83.3 at 2)."""
    units = B * 8
    assert L.attn_decode_model_best(units, 152, Nk, 128, 8.0e10, 7.5e12, 0.5e-6, 4.0e-6, 0) == want
