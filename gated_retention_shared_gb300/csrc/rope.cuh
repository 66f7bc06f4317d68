// rope.cuh -- rotary position encoding on the device (paper Section 3.1:
// Q (.) Theta, K (.) conj(Theta), Theta_n = e^{i n theta}; in the cross-decoder the
// shared K^ is rotated once when it is projected and every layer rotates its Q).
// Real-valued form: channel pair (2i, 2i+1) of the vector at position p turns by
// the angle p * theta_i, theta_i = base^(-2i/d).
//
// Positions reach 2^20 and more while theta_0 = 1, so the angle cannot be formed
// in fp32.  Two paths:
//   * rope_cs_exact: the angle formed and reduced modulo 2 pi in fp64 (for a few
//     positions per CTA, e.g. the base of a tile);
//   * rope_cs_offset: the angle of a small offset j (< 128) in fp32, reduced by a
//     two-constant Cody-Waite step (Cody & Waite, "Software Manual for the
//     Elementary Functions", 1980) to [-pi, pi] and handed to __sincosf;
// a position P0 + j combines the two by the angle-addition formulas.
#pragma once
#include <cmath>
#include <cstdint>

namespace yoco {

// theta_i = base^(-2i/d) for the d/2 <= 64 channel pairs, computed once on the host
// in fp64 and passed by value (kernels never evaluate the power)
struct RopeFreq {
    double theta[64];
};

inline RopeFreq make_rope_freq(float base, int d) {
    RopeFreq f{};
    if (base > 0.f)
        for (int i = 0; i < d / 2 && i < 64; ++i) f.theta[i] = std::exp2(-2.0 * i / d * std::log2((double)base));
    return f;
}

constexpr double kRopeTwoPi = 6.283185307179586476925286766559;
constexpr float kRopeInvTwoPiF = 0.15915494309189533577f;
constexpr float kRopeTwoPiHi = 6.28318548202514648438f;   // 2 pi rounded to float
constexpr float kRopeTwoPiLo = -1.7484555314695172e-07f;  // 2 pi - kRopeTwoPiHi

// (cos, sin) of pos * theta, reduced in fp64 (the reduced angle lies in [0, 2 pi))
__device__ __forceinline__ void rope_cs_exact(int64_t pos, double theta, float &c, float &s) {
    double a = (double)pos * theta;
    a = fma(-kRopeTwoPi, floor(a * (1.0 / kRopeTwoPi)), a);
    sincosf((float)a, &s, &c);
}

// (cos, sin) of j * theta for 0 <= j < 128, theta <= 1, in fp32 (angle error below
// 128 * 2^-23 rad)
__device__ __forceinline__ void rope_cs_offset(int j, float theta, float &c, float &s) {
    const float x = (float)j * theta;
    const float k = rintf(x * kRopeInvTwoPiF);
    float r = fmaf(-k, kRopeTwoPiHi, x);
    r = fmaf(-k, kRopeTwoPiLo, r);
    __sincosf(r, &s, &c);
}

// angle addition: (cos, sin)(a + b) from those of a and b
__device__ __forceinline__ void rope_cs_add(float ca, float sa, float cb, float sb, float &c, float &s) {
    c = ca * cb - sa * sb;
    s = sa * cb + ca * sb;
}

// turn the pair (x0, x1) by the angle with cosine c and sine s
__device__ __forceinline__ void rope_turn(float &x0, float &x1, float c, float s) {
    const float y0 = x0 * c - x1 * s;
    x1 = x0 * s + x1 * c;
    x0 = y0;
}

}  // namespace yoco
