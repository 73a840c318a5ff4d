// Device helpers shared by the router (router.cu) and the overflow re-route (reroute.cu).
#pragma once
#include <cmath>

#include "../../include/moe.h"

namespace moe {

// Half-width of the band around a score gap inside which the router GEMM's logits could misorder
// two experts. Those logits (a fresh tensor-core accumulator per 64-deep K block, the blocks
// added in fp32) differ from the exactly rounded dot product by at most 7.9e-7 x max(1, |largest
// logit of the row|) at d = 7168 (measured against float64 logits on 16384 x 7168 x 128,
// 8192 x 4096 x 16, 4096 x 2048 x 64 and 64 x 7168 x 128), so a logit difference by at most
// about 1.6e-6 on that scale; the band is about 9x that, scaled with sqrt(d) and with the row's
// largest |logit|.
__device__ __forceinline__ float router_band(int d, float max_abs_logit) {
  return 1.5e-5f * sqrtf((float)d * (1.0f / 7168.0f)) * fmaxf(1.0f, max_abs_logit);
}

// Selection score of one expert: the logit (PLAIN), logit + bias (BIAS_SELECT), or
// (logit - log(-log u)) / tau (GUMBEL). NaN ranks last.
__device__ __forceinline__ float selection_score(int mode, float l, float bias_e, float u_te,
                                                 float tau) {
  float s = l;
  if (mode == MOE_ROUTE_BIAS_SELECT) {
    s = l + bias_e;
  } else if (mode == MOE_ROUTE_GUMBEL) {
    const float g = -logf(-logf(u_te));
    s = (l + g) / tau;
  }
  return (s != s) ? -INFINITY : s;
}

// a beats b: higher score, or equal score and lower expert index
__device__ __forceinline__ bool beats(float sa, int ea, float sb, int eb) {
  return sa > sb || (sa == sb && ea < eb);
}

}  // namespace moe
