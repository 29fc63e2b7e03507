// RoPE angle -> (cos, sign * sin), shared by the RoPE kernels and the fused
// RMSNorm + QKV + RoPE pre-pass.
//
// The angle phi = p * inv_freq is formed in double precision and reduced
// modulo 2 pi with a two-term 2 pi (Cody-Waite style), then cos/sin are taken
// in single precision on the reduced angle: fp32 p * inv_freq alone would err
// by about p ulp at long contexts.
#pragma once

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

}  // namespace liger
