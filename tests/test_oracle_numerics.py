"""Pins for the oracle's rounding helpers and its Philox generator."""

import numpy as np
import pytest
import torch

from oracle.numerics import bf16_round, widen
from oracle.philox import philox4x32_10, uniforms, gumbel_argmax


def test_bf16_round_matches_torch_on_fp32_inputs():
    # For inputs exactly representable in fp32, rounding straight to bf16
    # must agree with torch's fp32 -> bf16 conversion (round to nearest even).
    rng = np.random.default_rng(0)
    x32 = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(20000) * 1e-30).astype(np.float32),
        (rng.standard_normal(20000) * 1e30).astype(np.float32),
    ])
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = bf16_round(x32.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_bf16_round_ties_to_even():
    # 1 + 2**-8 lies halfway between 1 and 1 + 2**-7: ties go to the even mantissa (1.0)
    assert bf16_round(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3 * 2**-8 is halfway between 1 + 2**-7 and 1 + 2**-6: goes to 1 + 2**-6
    assert bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert bf16_round(-(1.0 + 2.0 ** -8)) == -1.0
    # just above the halfway point rounds up
    assert bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7
    assert bf16_round(0.0) == 0.0


def test_widen_matches_torch():
    rng = np.random.default_rng(1)
    t = torch.from_numpy(rng.standard_normal(1000).astype(np.float32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(widen(bits), t.to(torch.float64).numpy())


# Known-answer vectors published with the Random123 library for
# philox4x32 with 10 rounds: (counter words, key words) -> output words.
PHILOX_KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF),
     (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,expect", PHILOX_KAT)
def test_philox_known_answers(ctr, key, expect):
    out = philox4x32_10(tuple(np.uint64(c) for c in ctr), key)
    assert tuple(int(o) for o in out) == expect


def test_uniforms_range_and_moments():
    u = uniforms(seed=1234, pos=7, rnd=3, stream=0, n=400000)
    assert u.min() > 0.0 and u.max() < 1.0
    # exact in fp32
    np.testing.assert_array_equal(u.astype(np.float32).astype(np.float64), u)
    assert abs(u.mean() - 0.5) < 3e-3
    assert abs(u.var() - 1.0 / 12.0) < 2e-3
    # distinct streams / positions give distinct draws
    assert not np.array_equal(u[:64], uniforms(1234, 7, 3, 1, 64))
    assert not np.array_equal(u[:64], uniforms(1234, 8, 3, 0, 64))


def test_gumbel_argmax_frequencies():
    # Sampling frequencies of Gumbel-max follow the normalised weights (chi-square test).
    from scipy.stats import chisquare
    w = np.array([0.05, 0.1, 0.0, 0.25, 0.6])
    with np.errstate(divide="ignore"):
        logw = np.log(w)
    counts = np.zeros(5)
    for i in range(20000):
        counts[gumbel_argmax(logw, seed=99, pos=i, rnd=1, stream=2)] += 1
    assert counts[2] == 0
    keep = w > 0
    stat = chisquare(counts[keep], 20000 * w[keep])
    assert stat.pvalue > 1e-3


def test_uniform_table_matches_single_draws():
    # the table form (arrays of positions and rounds) gives every draw the
    # single-position form gives, in the same vocabulary order
    from oracle.philox import uniforms_table
    pos = np.array([0, 5, 1023])
    rnd = np.array([[0], [7]])
    tab = uniforms_table(99, pos[None, :], rnd, 2, 11)
    assert tab.shape == (2, 3, 11)
    for i in range(2):
        for j in range(3):
            np.testing.assert_array_equal(tab[i, j], uniforms(99, int(pos[j]), int(rnd[i, 0]), 2, 11))
