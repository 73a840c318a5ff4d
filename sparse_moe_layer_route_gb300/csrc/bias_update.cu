// Aux-loss-free expert-bias update after a forward pass.
//
// "AI架构演进从稀疏MoE到条件记忆的工程实践", gating-network code (its no_grad block): the load of each
// expert is the number of (token, j) selections it received (all top-k picks, before any capacity
// limit), and bias <- decay * bias - rate * load / (mean(load) + 1e-8); the page uses decay 0.99
// and rate 0.01 (its configuration lists bias_decay 0.99 and bias_update_rate 0.01).
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"

namespace moe {
namespace {

// One block. The load total is an exact integer sum; the mean and ratio are computed in fp64.
__global__ void __launch_bounds__(256) bias_update_kernel(const int32_t* __restrict__ counts,
                                                          float* __restrict__ bias, int E,
                                                          float decay, float rate) {
  griddep_wait();
  __shared__ long long total;
  if (threadIdx.x == 0) {
    long long s = 0;
    for (int e = 0; e < E; ++e) s += counts[e];
    total = s;
  }
  __syncthreads();
  const double mean = (double)total / (double)E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const double ratio = (double)counts[e] / (mean + 1e-8);
    bias[e] = (float)((double)decay * (double)bias[e] - (double)rate * ratio);
  }
}

}  // namespace

cudaError_t launch_bias_update(int E, const int32_t* counts, float* bias, float decay, float rate,
                               cudaStream_t st) {
  return launch_k(bias_update_kernel, dim3(1), dim3(256), 0, st, counts, bias, E, decay, rate);
}

}  // namespace moe
