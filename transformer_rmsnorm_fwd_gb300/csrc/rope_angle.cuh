// RoPE angle -> (cos, sign * sin), shared by the RoPE kernels and the fused
// RMSNorm + QKV + RoPE pre-pass.
//
// The angle phi = p * inv_freq is formed in double precision and reduced
// modulo 2 pi with a two-term 2 pi (Cody-Waite style), then cos/sin are taken
// in single precision on the reduced angle: fp32 p * inv_freq alone would err
// by about p ulp at long contexts.
#pragma once

#include <stdint.h>

namespace liger {

__device__ __forceinline__ float2 angle_cs(double p, double inv_freq, float sign) {
    const double two_pi_hi = 6.283185307179586232;      // nearest double to 2 pi
    const double two_pi_lo = 2.4492935982947064e-16;    // 2 pi - two_pi_hi
    const double phi = p * inv_freq;
    const double k = rint(phi * 0.15915494309189535);   // 1 / (2 pi)
    double r = fma(-k, two_pi_hi, phi);
    r = fma(-k, two_pi_lo, r);
    float s, c;
    sincosf(static_cast<float>(r), &s, &c);
    return make_float2(c, sign * s);
}

// The same angle in single precision for positions below 2^24 (exact as
// floats): inv_freq is passed as a float pair f_hi + f_lo (f_hi = fl(f),
// f_lo = fl(f - f_hi)); the product p * f_hi is made exact as a_hi + err by
// one FMA (two-product), and the reduction modulo 2 pi follows Cody and Waite
// (1980) with 2 pi split into c1 = fl(2 pi) and c2 = fl(2 pi - c1): each FMA
// below rounds only a result smaller than about pi, so r is (p f) mod 2 pi to
// within a few 1e-7 for every position below 2^24.  Larger positions take the
// double-precision path.
__device__ __forceinline__ float2 angle_cs32(int64_t p, float f_hi, float f_lo, double f, float sign) {
    if (p < 0 || p >= (int64_t{1} << 24)) return angle_cs(static_cast<double>(p), f, sign);
    const float c1 = 6.28318548202514648f;       // fl(2 pi)
    const float c2 = -1.74845553e-07f;           // fl(2 pi - c1)
    const float pf = static_cast<float>(p);
    const float a_hi = pf * f_hi;
    const float a_lo = fmaf(pf, f_lo, fmaf(pf, f_hi, -a_hi));
    const float k = rintf(a_hi * 0.159154943091895336f);   // 1 / (2 pi)
    float r = fmaf(-k, c1, a_hi);
    r = fmaf(-k, c2, r);
    r += a_lo;
    float s, c;
    sincosf(r, &s, &c);
    return make_float2(c, sign * s);
}

}  // namespace liger
