// Combine: out[t] = sum over kept j of y_slot[t*k + j] (fp16, already gate-scaled by the down GEMM)
// + sum over shared s of y_slot[T*k + s*T + t], in that fixed order in fp32, one bf16 rounding.
//
// Weighted sum of the selected experts' outputs: "大模型MoE稀疏激活原理与工程实践", §3.1
// (output = sum(weights[i] * expert_i_output)); aggregation layer of
// "AI架构演进从稀疏MoE到条件记忆的工程实践" (layered-architecture figure), without its residual.
// Shared experts always added: "V4" rework page, §2.2.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;

// acc += 8 fp16 values (exact widening to fp32)
__device__ __forceinline__ void add8(float (&acc)[8], const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
    const float2 f = __half22float2(h);
    acc[2 * i] += f.x;
    acc[2 * i + 1] += f.y;
  }
}

// Grid (column blocks, tokens): thread = one 8-column group of one token. Without a capacity
// limit every slot is kept, so every row's 16-byte load is issued at once; with one, a row is
// loaded only when its slot was kept (dropped slots' rows are never written), the flags first.
// Then the fixed-order sum.
template <bool MAY_DROP, int KR, int SR>  // KR >= top_k, SR >= n_shared: the row registers
__global__ void __launch_bounds__(kThreads) combine_kernel(const uint16_t* __restrict__ y,
                                                           const int32_t* __restrict__ slot_pos,
                                                           uint16_t* __restrict__ out, int T,
                                                           int d, int k, int S) {
  griddep_wait();
  const int t = blockIdx.y;
  const int g = blockIdx.x * kThreads + threadIdx.x;
  if (g >= d / 8) return;
  const long long TK = (long long)T * k;
  const uint4* __restrict__ y4 = reinterpret_cast<const uint4*>(y);
  const long long d8 = d / 8;
  uint4 vr[KR], vs[SR > 0 ? SR : 1];
  bool kept[KR];
#pragma unroll
  for (int j = 0; j < KR; ++j)
    if (j < k) kept[j] = !MAY_DROP || slot_pos[(long long)t * k + j] >= 0;
#pragma unroll
  for (int j = 0; j < KR; ++j)
    if (j < k) vr[j] = kept[j] ? y4[((long long)t * k + j) * d8 + g] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int s = 0; s < SR; ++s)
    if (s < S) vs[s] = y4[(TK + (long long)s * T + t) * d8 + g];
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < KR; ++j)
    if (j < k && kept[j]) add8(acc, vr[j]);
#pragma unroll
  for (int s = 0; s < SR; ++s)
    if (s < S) add8(acc, vs[s]);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    o[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(out + (size_t)t * d + 8 * g) = make_uint4(o[0], o[1], o[2], o[3]);
}

template <bool MAY_DROP>
cudaError_t launch_combine_variant(const Shape& s, const uint16_t* y, const int32_t* slot_pos,
                                   uint16_t* out, cudaStream_t st) {
  const dim3 grid((s.d / 8 + kThreads - 1) / kThreads, s.T);
  const dim3 block(kThreads);
  if (s.k <= 2 && s.S <= 1)
    return launch_k(combine_kernel<MAY_DROP, 2, 1>, grid, block, 0, st, y, slot_pos, out, s.T,
                    s.d, s.k, s.S);
  if (s.S <= 1)
    return launch_k(combine_kernel<MAY_DROP, 8, 1>, grid, block, 0, st, y, slot_pos, out, s.T,
                    s.d, s.k, s.S);
  return launch_k(combine_kernel<MAY_DROP, 8, 4>, grid, block, 0, st, y, slot_pos, out, s.T, s.d,
                  s.k, s.S);
}

// dst[i] = fp16(bf16 src[i]), round to nearest even, saturating; 8 elements per thread.
__global__ void __launch_bounds__(kThreads) pack_f16_kernel(const uint16_t* __restrict__ src,
                                                            uint16_t* __restrict__ dst, size_t n) {
  const size_t n8 = n / 8;
  for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < n8;
       i += (size_t)gridDim.x * kThreads) {
    const uint4 v = reinterpret_cast<const uint4*>(src)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
      asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(o[j]) : "f"(hi), "f"(lo));
    }
    reinterpret_cast<uint4*>(dst)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  // tail (n not a multiple of 8)
  const size_t t = n8 * 8 + (size_t)blockIdx.x * kThreads + threadIdx.x;
  if (blockIdx.x == 0 && t < n) {
    const float v = __uint_as_float(((uint32_t)src[t]) << 16);
    uint32_t o;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(o) : "f"(0.0f), "f"(v));
    dst[t] = (uint16_t)(o & 0xFFFFu);
  }
}

}  // namespace

cudaError_t launch_pack_f16(const uint16_t* src, uint16_t* dst, size_t n, cudaStream_t st) {
  long long grid = (long long)((n / 8 + kThreads - 1) / kThreads);
  const long long cap = (long long)num_sms() * 32;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  pack_f16_kernel<<<(unsigned)grid, kThreads, 0, st>>>(src, dst, n);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Shape& s, const uint16_t* y, const int32_t* slot_pos,
                           uint16_t* out, cudaStream_t st) {
  if (s.C < s.TK)  // a slot may be dropped
    return launch_combine_variant<true>(s, y, slot_pos, out, st);
  return launch_combine_variant<false>(s, y, slot_pos, out, st);
}

}  // namespace moe
