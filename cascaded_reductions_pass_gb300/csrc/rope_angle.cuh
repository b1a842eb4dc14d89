// rope_angle.cuh -- the rotary-embedding angle p * base^(-2i/D) and its cosine
// and sine, shared by the separate RoPE pass (rope.cu) and the attention
// kernels that rotate Q and K rows as they load them (attn_fwd_tc.cu).
//
// Both call the same function, so a row rotated inside the attention kernel
// is bit for bit the row the separate pass writes.
//
// The host passes base^(-2i/D) computed in double and split into two floats
// (hi + lo).  The device forms p * (hi + lo) as a float pair (the product's
// rounding error recovered with an FMA) and reduces it modulo 2 pi by Cody and
// Waite's method with 2 pi split into three floats, so positions in the tens
// of thousands keep angle errors near 1e-7.  The reduced angle lies in
// [-pi, pi], where the hardware sine and cosine (__sincosf) are accurate to a
// few 1e-7 absolute; their error therefore does not grow with the position.
// (The library sincosf costs several times more per angle, which at one angle
// per element pair made the rotation inside the attention kernel cost more
// than a separate pass over Q and K.)
#pragma once

#include <math.h>

#include "rf_internal.h"

namespace rf {

struct RopeParams {
  float fhi[kRopeMaxHalf], flo[kRopeMaxHalf];  // base^(-2i/D) = fhi[i] + flo[i]
  float two_pi[3];                             // 2 pi = sum of the three floats
  float inv_two_pi;
};

inline RopeParams make_rope_params(double base, int D) {
  RopeParams prm;
  const int half = D / 2;
  for (int i = 0; i < kRopeMaxHalf; ++i) {
    const double f = i < half ? pow(base, -2.0 * i / D) : 0.0;
    prm.fhi[i] = static_cast<float>(f);
    prm.flo[i] = static_cast<float>(f - static_cast<double>(prm.fhi[i]));
  }
  const double two_pi = 2.0 * 3.14159265358979323846;
  prm.two_pi[0] = static_cast<float>(two_pi);
  prm.two_pi[1] = static_cast<float>(two_pi - static_cast<double>(prm.two_pi[0]));
  prm.two_pi[2] = static_cast<float>(two_pi - static_cast<double>(prm.two_pi[0]) - static_cast<double>(prm.two_pi[1]));
  prm.inv_two_pi = static_cast<float>(1.0 / two_pi);
  return prm;
}

// (cos, sin) of position p times base^(-2i/D).
__device__ __forceinline__ float2 rope_cs(float p, int i, const RopeParams& prm) {
  // theta = p * (fhi + flo) as th + tl, then th + tl - j * 2 pi with j = nearest integer
  const float th = p * prm.fhi[i];
  const float tl = fmaf(p, prm.flo[i], fmaf(p, prm.fhi[i], -th));
  const float j = rintf(th * prm.inv_two_pi);
  float r = fmaf(-j, prm.two_pi[0], th);
  r = fmaf(-j, prm.two_pi[1], r);
  r = fmaf(-j, prm.two_pi[2], r);
  r += tl;
  float s, c;
  __sincosf(r, &s, &c);
  return make_float2(c, s);
}

// One rotated pair: (a, b) -> (a cos - b sin, a sin + b cos).
__device__ __forceinline__ void rope_rotate(float a, float b, float2 cs, float& ya, float& yb) {
  ya = fmaf(a, cs.x, -b * cs.y);
  yb = fmaf(a, cs.y, b * cs.x);
}

}  // namespace rf
