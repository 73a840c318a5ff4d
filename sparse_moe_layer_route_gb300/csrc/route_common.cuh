// Device helpers shared by the router (router.cu) and the overflow re-route (reroute.cu).
#pragma once
#include <cmath>

#include "../../include/moe.h"

namespace moe {

// Half-width of the band around a score gap inside which the tensor-core logits could misorder
// two experts: the tensor core's fp32 accumulation differs from an exactly rounded dot product by
// up to ~4e-5 on unit-scale logits at d = 7168 (measured); the band is about 6x that, scaled
// with sqrt(d) and with the row's largest |logit|.
__device__ __forceinline__ float router_band(int d, float max_abs_logit) {
  return 2.5e-4f * sqrtf((float)d * (1.0f / 7168.0f)) * fmaxf(1.0f, max_abs_logit);
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
