"""Pins for the oracle's bf16 conversion and Philox generator (CPU only)."""

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import bf16_bits_to_f64, f64_to_bf16_bits, philox4, philox4x32_10, uniform_from_u32
from oracle.philox import philox_uniform_pair
import spec_workloads as wl


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint16)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    ours = bf16_bits_to_f64(bits)
    finite = np.isfinite(t)
    assert np.array_equal(ours[finite], t[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(t))


def test_bf16_encode_matches_torch_on_float32_values():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 3,
                        rng.standard_normal(1000).astype(np.float32) * np.float32(1e-38),
                        np.array([0.0, -0.0, 1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)], dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(f64_to_bf16_bits(x.astype(np.float64)), ref)
    # the workload generator's encoder agrees too (it is a separate implementation)
    assert np.array_equal(wl.f32_to_bf16_bits(x), ref)


def test_bf16_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: even is 1.0
    assert bf16_bits_to_f64(f64_to_bf16_bits(np.array([1 + 2 ** -8])))[0] == 1.0
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6
    assert bf16_bits_to_f64(f64_to_bf16_bits(np.array([1 + 3 * 2 ** -8])))[0] == 1 + 2 ** -6
    # just above the halfway point rounds up (a float64 value no float32 holds)
    assert bf16_bits_to_f64(f64_to_bf16_bits(np.array([1 + 2 ** -8 + 2 ** -40])))[0] == 1 + 2 ** -7


def test_philox4x32_known_answers():
    for row in read_golden("philox4x32_10_kat.txt"):
        words = [int(w, 16) for w in row]
        assert philox4x32_10(words[0:4], words[4:6]) == tuple(words[6:10])


def test_philox4x64_matches_numpy():
    # NumPy's Philox is Philox4x64-10; it advances the counter before each block.
    for key in [(0, 0), (1, 2), (0xDEADBEEF12345678, 0x0123456789ABCDEF)]:
        for start in [0, 5, (1 << 64) - 3]:
            bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                                  counter=np.array([start, 7, 0, 1], dtype=np.uint64))
            raw = [int(x) for x in bg.random_raw(12)]
            ours = []
            c0, c1 = start, 7
            for _ in range(3):
                c0 = (c0 + 1) & ((1 << 64) - 1)
                if c0 == 0:
                    c1 += 1
                ours.extend(philox4((c0, c1, 0, 1), key, width=64))
            assert ours == raw


def test_uniform_conversion_range():
    assert uniform_from_u32(0) == 0.0
    assert uniform_from_u32(0xFFFFFFFF) == (2 ** 24 - 1) / 2 ** 24
    assert uniform_from_u32(0xFFFFFFFF) < 1.0
    u0, u1 = philox_uniform_pair(1234, 0, 3, 0)
    assert 0.0 <= u0 < 1.0 and 0.0 <= u1 < 1.0


def test_philox_uniforms_are_uniform():
    us = np.array([philox_uniform_pair(99, 0, c, b)[0] for c in range(100) for b in range(50)])
    hist = np.histogram(us, bins=10, range=(0, 1))[0]
    expected = len(us) / 10
    chi2 = ((hist - expected) ** 2 / expected).sum()
    assert chi2 < 27.9  # chi-square, 9 dof, p = 0.001
