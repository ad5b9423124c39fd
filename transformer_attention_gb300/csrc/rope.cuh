// Rotation angles of RoPE ("Gemma 3 Attention Block", How it works: RoPE with
// the layer's base frequency and scale), shared by the prologue kernel and
// the fused projection epilogue.
//
// The angle of pair c at position p is (p / scale) * base^(-2c/d_h).  The
// frequency inv_scale * base^(-2c/d_h) is computed on the host in double and
// split into an fp32 (hi, lo) pair; the device forms p * freq as an exact
// fp32 two-product plus the lo term and reduces it modulo 2*pi by Cody-Waite
// with a two-part 2*pi, so positions up to 2^24 keep ~1e-6 rad of angle error
// without fp64 work on the device.  sin and cos of the reduced angle (about
// [-pi, pi]) come from the hardware approximation (absolute error ~2^-21).
#pragma once
#include <cmath>
#include <cuda_runtime.h>

namespace g3 {

struct RopeFreqs {
  float2 f[128];
};

inline RopeFreqs make_rope_freqs(int d_h, double rope_base, double rope_scale) {
  RopeFreqs r{};
  for (int c = 0; c < d_h / 2 && c < 128; ++c) {
    const double f = std::pow(rope_base, -2.0 * c / d_h) / rope_scale;
    r.f[c].x = static_cast<float>(f);
    r.f[c].y = static_cast<float>(f - static_cast<double>(r.f[c].x));
  }
  return r;
}

constexpr double kRopeTwoPi = 6.283185307179586476925286766559;
constexpr float kRopeTwoPiHi = static_cast<float>(kRopeTwoPi);
constexpr float kRopeTwoPiMid = static_cast<float>(kRopeTwoPi - static_cast<double>(kRopeTwoPiHi));
constexpr float kRopeInvTwoPi = static_cast<float>(1.0 / kRopeTwoPi);

// sin and cos of p * (f.x + f.y), p an integer position held exactly in fp32.
__device__ __forceinline__ void rope_sincos(float p, float2 f, float& sn, float& cs) {
  const float a_hi = p * f.x;
  const float a_err = fmaf(p, f.x, -a_hi);     // exact residual of the product
  const float a_lo = fmaf(p, f.y, a_err);
  const float k = rintf(a_hi * kRopeInvTwoPi);
  float r = fmaf(-k, kRopeTwoPiHi, a_hi);
  r = fmaf(-k, kRopeTwoPiMid, r);
  r += a_lo;
  __sincosf(r, &sn, &cs);
}

// The same for two pairs at once (frequencies fa and fb, one position p) in
// packed fp32x2 arithmetic: each lane performs exactly the operations of
// rope_sincos ((-k) * hi is k * (-hi) exactly), in half the instructions.
__device__ __forceinline__ void rope_sincos2(float p, float2 fa, float2 fb, float2& sn,
                                             float2& cs) {
  const float2 pp = make_float2(p, p);
  const float2 fh = make_float2(fa.x, fb.x), fl = make_float2(fa.y, fb.y);
  const float2 a_hi = __fmul2_rn(pp, fh);
  const float2 a_err = __ffma2_rn(pp, fh, make_float2(-a_hi.x, -a_hi.y));
  const float2 a_lo = __ffma2_rn(pp, fl, a_err);
  const float2 q = __fmul2_rn(a_hi, make_float2(kRopeInvTwoPi, kRopeInvTwoPi));
  const float2 k = make_float2(rintf(q.x), rintf(q.y));
  float2 r = __ffma2_rn(k, make_float2(-kRopeTwoPiHi, -kRopeTwoPiHi), a_hi);
  r = __ffma2_rn(k, make_float2(-kRopeTwoPiMid, -kRopeTwoPiMid), r);
  r = __fadd2_rn(r, a_lo);
  __sincosf(r.x, &sn.x, &cs.x);
  __sincosf(r.y, &sn.y, &cs.y);
}

}  // namespace g3
