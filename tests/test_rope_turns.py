"""The host conversion of a RoPE frequency into a 64-bit fixed-point turn rate
(csrc/rope_table.h, turn_rate_fixed64), checked against exact rational
arithmetic (CPU only).  The split pass forms a block token's rotary angle as
position * turn_rate mod 2^64 (the angle's fraction of a turn) instead of a
floating-point product and range reduction, so the table must be
round(f * 2^64 / (2 pi)) and a position times it must land on the exact
fraction of a turn.  The reference values come from sympy's pi at 60 digits,
not from the library's constant."""
import os
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decoding_drafter_k3_gb300", "csrc")

HARNESS = r"""
#include <cstdio>
#include <cstdlib>
#include "rope_table.h"
int main(int argc, char **argv) {
    for (int i = 1; i < argc; ++i) {
        const double f = std::strtod(argv[i], nullptr);
        std::printf("%llu\n", static_cast<unsigned long long>(k3da_host::turn_rate_fixed64(f)));
    }
    return 0;
}
"""


@pytest.fixture(scope="module")
def turn_rate(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    d = tmp_path_factory.mktemp("turns")
    src = d / "h.cpp"
    src.write_text(HARNESS)
    exe = d / "h"
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"), "-I", CSRC, str(src), "-o",
                    str(exe)], check=True)

    def run(values):
        out = subprocess.run([str(exe)] + [repr(float(v)) for v in values], check=True, capture_output=True,
                             text=True).stdout.split()
        return [int(x) for x in out]
    return run


def two_pi():
    sympy = pytest.importorskip("sympy")
    return Fraction(str(sympy.N(2 * sympy.pi, 60)))


def exact_rate(f):
    # round(f * 2^64 / (2 pi)) with f taken exactly (a double is a dyadic rational)
    return round(Fraction(f) * 2 ** 64 / two_pi())


def neox_freqs(base=10000.0, dims=64):
    return [base ** (-2.0 * j / dims) for j in range(dims // 2)]


def test_rates_are_the_rounded_exact_values(turn_rate):
    fs = neox_freqs() + neox_freqs(500000.0) + [1.0, 0.5, 0.75, 1e-9, 2.0 ** -40, 0.999999999]
    got = turn_rate(fs)
    for f, g in zip(fs, got):
        assert abs(g - exact_rate(f)) <= 1, (f, g, exact_rate(f))


def test_out_of_range_frequencies_give_zero(turn_rate):
    assert turn_rate([0.0, -1.0, 1.5, 2.0 ** -80]) == [0, 0, 0, 0]


def test_position_times_rate_is_the_fraction_of_a_turn(turn_rate):
    fs = neox_freqs()
    rates = turn_rate(fs)
    tp = two_pi()
    for p in [0, 1, 7, 2041, 131079, 2 ** 24 - 1, 2 ** 31 - 1]:
        for f, g in zip(fs, rates):
            turns = (p * g) % 2 ** 64 / Fraction(2 ** 64)
            exact = (Fraction(p) * Fraction(f) / tp) % 1
            err = abs(turns - exact)
            err = min(err, 1 - err)  # on the circle
            assert err <= Fraction(p + 1, 2 ** 64), (p, f)


def test_top_bits_give_the_angle_within_float_resolution(turn_rate):
    # What the kernel does with the product: its top 32 bits as a signed
    # fraction of a turn, scaled to half-turns for sincospif.
    fs = neox_freqs()
    rates = turn_rate(fs)
    for p in [3, 2049, 131000]:
        for f, g in zip(fs, rates):
            top = ((p * g) % 2 ** 64) >> 32
            top = top - 2 ** 32 if top >= 2 ** 31 else top
            half_turns = np.float32(top) * np.float32(2.0 ** -31)
            got = np.array([np.cos(np.pi * np.float64(half_turns)), np.sin(np.pi * np.float64(half_turns))])
            theta = p * f  # fp64 is exact enough here for the comparison
            want = np.array([np.cos(theta), np.sin(theta)])
            assert np.abs(got - want).max() < 4e-7, (p, f)
