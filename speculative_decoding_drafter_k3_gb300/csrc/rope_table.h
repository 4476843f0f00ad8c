// rope_table.h -- host side of the rotary frequencies shared by the library's
// kernels: the plain NeoX table and its YaRN rescaling (k3da_yarn in k3da.h).
#pragma once

#include <cmath>
#include <cstdint>

#include "k3da.h"

namespace k3da_host {

// True when `y` describes a usable YaRN rescaling.
inline bool yarn_valid(const k3da_yarn *y) {
    if (y == nullptr) return false;
    const float v[5] = {y->factor, y->original_max_position, y->beta_fast, y->beta_slow, y->mscale};
    for (float x : v)
        if (!std::isfinite(x)) return false;
    return y->factor >= 1.f && y->original_max_position > 0.f && y->beta_slow > 0.f &&
           y->beta_fast > y->beta_slow && y->mscale >= 0.f;
}

// Multiplier of the rotated q and k: the caller's mscale when it is
// positive, else the YaRN paper's sqrt(1/t) = 0.1 * ln(factor) + 1 (formed in
// fp64, rounded once to fp32).
inline float yarn_mscale(const k3da_yarn *y) {
    if (y->mscale > 0.f) return y->mscale;
    return static_cast<float>(0.1 * std::log(static_cast<double>(y->factor)) + 1.0);
}

// Frequencies of the `pairs` rotary pairs of a head of 2*pairs dims, in
// fp64.  Plain NeoX: theta_j = base^(-2j / dims).  With YaRN (factor != 1):
// r = original_max_position * theta_j / (2 pi) counts the pair's turns over
// the original context; pairs with r >= beta_fast keep theta_j, pairs with
// r <= beta_slow turn factor times slower, and a linear ramp joins the two.
inline void rope_frequencies(double *inv_freq, int pairs, float base, const k3da_yarn *yarn) {
    const double dims = 2.0 * pairs;
    for (int j = 0; j < pairs; ++j) {
        const double theta = std::pow(static_cast<double>(base), -2.0 * j / dims);
        if (yarn == nullptr || yarn->factor == 1.f) {
            inv_freq[j] = theta;
            continue;
        }
        const double turns = static_cast<double>(yarn->original_max_position) * theta / 6.283185307179586;
        double ramp = (turns - yarn->beta_slow) / (static_cast<double>(yarn->beta_fast) - yarn->beta_slow);
        ramp = ramp < 0.0 ? 0.0 : (ramp > 1.0 ? 1.0 : ramp);
        inv_freq[j] = theta * ramp + theta / static_cast<double>(yarn->factor) * (1.0 - ramp);
    }
}

// A rotary frequency f (radians per position, 0 < f <= 1) as a turn rate:
// round(f * 2^64 / (2 pi)), unsigned 64-bit fixed point with 2^64 = one
// turn.  For an integer position p, p * turn_rate mod 2^64 (plain wrapping
// integer arithmetic) is then p f / (2 pi) mod 1, the angle's fraction of a
// turn, exact up to p * 2^-65 turns: no floating-point range reduction.
// Formed exactly from the fp64 f with 128-bit integer arithmetic and
// floor(2^128 / (2 pi)) = kInv2PiHi * 2^64 + kInv2PiLo.
inline uint64_t turn_rate_fixed64(double f) {
    constexpr uint64_t kInv2PiHi = 0x28BE60DB9391054Aull;
    constexpr uint64_t kInv2PiLo = 0x7F09D5F47D4D3770ull;
    if (!(f > 0.0) || !(f <= 1.0)) return 0;
    int ex = 0;
    const double fr = std::frexp(f, &ex);  // f = fr * 2^ex, fr in [0.5, 1)
    const uint64_t m = static_cast<uint64_t>(std::ldexp(fr, 53));  // exact: f = m * 2^(ex - 53)
    // f * 2^64 / (2 pi) = m * K * 2^(ex - 53 - 128 + 64) with K = 2^128 / (2 pi):
    // the product m * K (up to 179 bits) is high * 2^64 + low, shifted right
    // by rs = 117 - ex bits (>= 116 since ex <= 1).
    const unsigned __int128 p1 = static_cast<unsigned __int128>(m) * kInv2PiHi;
    const unsigned __int128 p0 = static_cast<unsigned __int128>(m) * kInv2PiLo;
    const unsigned __int128 high = p1 + (p0 >> 64);
    const int rs = 117 - ex - 64;  // shift of `high`
    if (rs >= 127) return 0;
    const unsigned __int128 half = static_cast<unsigned __int128>(1) << (rs - 1);
    return static_cast<uint64_t>((high + half) >> rs);
}

}  // namespace k3da_host
