// Combine: out[t] = sum over kept j of y_slot[t*k + j] (fp16 or fp32, already gate-scaled by the
// down GEMM) + sum over shared s of y_slot[T*k + s*T + t], in that fixed order in fp32, one bf16
// rounding.
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

// One thread's 8 columns of one slot row: fp16 (16 bytes) or fp32 (32 bytes).
template <bool F32>
struct Row8 {
  uint4 v[F32 ? 2 : 1];
};

template <bool F32>
__device__ __forceinline__ Row8<F32> load8(const void* y, long long row, long long d, int g) {
  Row8<F32> r;
  if constexpr (F32) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(y) + row * d) + 2 * g;
    r.v[0] = p[0];
    r.v[1] = p[1];
  } else {
    r.v[0] = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(y) + row * d)[g];
  }
  return r;
}

template <bool F32>
__device__ __forceinline__ Row8<F32> zero8() {
  Row8<F32> r;
#pragma unroll
  for (int i = 0; i < (F32 ? 2 : 1); ++i) r.v[i] = make_uint4(0u, 0u, 0u, 0u);
  return r;
}

// acc += the row's 8 values (fp16 widened exactly to fp32, or fp32 as they are)
template <bool F32>
__device__ __forceinline__ void add8(float (&acc)[8], const Row8<F32>& r) {
  if constexpr (F32) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t w[4] = {r.v[h].x, r.v[h].y, r.v[h].z, r.v[h].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[4 * h + i] += __uint_as_float(w[i]);
    }
  } else {
    const uint32_t w[4] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 hv = *reinterpret_cast<const __half2*>(&w[i]);
      const float2 f = __half22float2(hv);
      acc[2 * i] += f.x;
      acc[2 * i + 1] += f.y;
    }
  }
}

// Grid (column blocks, tokens): thread = one 8-column group of one token. Without a capacity
// limit every slot is kept, so every row's load is issued at once; with one, a row is loaded only
// when its slot was kept (dropped slots' rows are never written), the flags first. Then the
// fixed-order sum. F32: the slot rows are fp32 (bf16 down path), else fp16.
template <bool MAY_DROP, int KR, int SR, bool F32>  // KR >= top_k, SR >= n_shared
__global__ void __launch_bounds__(kThreads) combine_kernel(const void* __restrict__ y,
                                                           const int32_t* __restrict__ slot_pos,
                                                           uint16_t* __restrict__ out, int T,
                                                           int d, int k, int S) {
  griddep_wait();
  const int t = blockIdx.y;
  const int g = blockIdx.x * kThreads + threadIdx.x;
  if (g >= d / 8) return;
  const long long TK = (long long)T * k;
  Row8<F32> vr[KR], vs[SR > 0 ? SR : 1];
  bool kept[KR];
#pragma unroll
  for (int j = 0; j < KR; ++j)
    if (j < k) kept[j] = !MAY_DROP || slot_pos[(long long)t * k + j] >= 0;
#pragma unroll
  for (int j = 0; j < KR; ++j)
    if (j < k) vr[j] = kept[j] ? load8<F32>(y, (long long)t * k + j, d, g) : zero8<F32>();
#pragma unroll
  for (int s = 0; s < SR; ++s)
    if (s < S) vs[s] = load8<F32>(y, TK + (long long)s * T + t, d, g);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < KR; ++j)
    if (j < k && kept[j]) add8<F32>(acc, vr[j]);
#pragma unroll
  for (int s = 0; s < SR; ++s)
    if (s < S) add8<F32>(acc, vs[s]);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    o[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(out + (size_t)t * d + 8 * g) = make_uint4(o[0], o[1], o[2], o[3]);
}

// One CTA per token, for rows of 2 to 4 column groups per thread (d / 8 in (256, 1024]): thread
// i takes groups i, i + 256, ... (at most G), and every row load of every group is issued before
// the adds. Against a CTA per (token, 256 groups) this keeps several loads in flight per thread
// behind one read of the token's slot flags: the skewed prefill's combine (T = 16384, d = 7168,
// top_k = 2) went from 72 to 57 us in the bench.
template <bool MAY_DROP, int KR, int SR, bool F32, int G>
__global__ void __launch_bounds__(kThreads) combine_tok_kernel(const void* __restrict__ y,
                                                               const int32_t* __restrict__ slot_pos,
                                                               uint16_t* __restrict__ out, int T,
                                                               int d, int k, int S) {
  griddep_wait();
  const int t = blockIdx.x;
  const int d8 = d / 8;
  const long long TK = (long long)T * k;
  bool kept[KR];
#pragma unroll
  for (int j = 0; j < KR; ++j)
    if (j < k) kept[j] = !MAY_DROP || slot_pos[(long long)t * k + j] >= 0;
  Row8<F32> vr[G][KR], vs[G][SR > 0 ? SR : 1];
#pragma unroll
  for (int q = 0; q < G; ++q) {
    const int g = threadIdx.x + q * kThreads;
    if (g < d8) {
#pragma unroll
      for (int j = 0; j < KR; ++j)
        if (j < k) vr[q][j] = kept[j] ? load8<F32>(y, (long long)t * k + j, d, g) : zero8<F32>();
#pragma unroll
      for (int s2 = 0; s2 < SR; ++s2)
        if (s2 < S) vs[q][s2] = load8<F32>(y, TK + (long long)s2 * T + t, d, g);
    }
  }
#pragma unroll
  for (int q = 0; q < G; ++q) {
    const int g = threadIdx.x + q * kThreads;
    if (g < d8) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < KR; ++j)
        if (j < k && kept[j]) add8<F32>(acc, vr[q][j]);
#pragma unroll
      for (int s2 = 0; s2 < SR; ++s2)
        if (s2 < S) add8<F32>(acc, vs[q][s2]);
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        o[i] = *reinterpret_cast<const uint32_t*>(&b);
      }
      *reinterpret_cast<uint4*>(out + (size_t)t * d + 8 * g) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

template <bool MAY_DROP, bool F32>
cudaError_t launch_combine_variant(const Shape& s, const void* y, const int32_t* slot_pos,
                                   uint16_t* out, cudaStream_t st) {
  const int d8 = s.d / 8;
  // a CTA per token when the rows span 2-4 groups per thread and the tokens fill the GPU
  if (s.k <= 2 && s.S <= 1 && d8 > kThreads && d8 <= 4 * kThreads && s.T >= 2 * num_sms()) {
    if (d8 <= 2 * kThreads)
      return launch_k(combine_tok_kernel<MAY_DROP, 2, 1, F32, 2>, dim3(s.T), dim3(kThreads), 0,
                      st, y, slot_pos, out, s.T, s.d, s.k, s.S);
    return launch_k(combine_tok_kernel<MAY_DROP, 2, 1, F32, 4>, dim3(s.T), dim3(kThreads), 0, st,
                    y, slot_pos, out, s.T, s.d, s.k, s.S);
  }
  const dim3 grid((s.d / 8 + kThreads - 1) / kThreads, s.T);
  const dim3 block(kThreads);
  if (s.k <= 2 && s.S <= 1)
    return launch_k(combine_kernel<MAY_DROP, 2, 1, F32>, grid, block, 0, st, y, slot_pos, out,
                    s.T, s.d, s.k, s.S);
  if (s.S <= 1)
    return launch_k(combine_kernel<MAY_DROP, 8, 1, F32>, grid, block, 0, st, y, slot_pos, out,
                    s.T, s.d, s.k, s.S);
  return launch_k(combine_kernel<MAY_DROP, 8, 4, F32>, grid, block, 0, st, y, slot_pos, out, s.T,
                  s.d, s.k, s.S);
}

// dst[i] = fp16(bf16 src[i]), round to nearest even, saturating; 8 elements per thread. A
// source whose magnitude would round past 65504 (|w| >= 65520: a bf16 of 65536 or more, or not
// finite) is clamped, and the call ORs MOE_DEVFAULT_FP16_RANGE into *fault (when given), once per
// warp that met one.
__device__ __forceinline__ uint32_t mag_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }
constexpr uint32_t kF16Clamp = 0x477FF000u;  // 65520.0f

__global__ void __launch_bounds__(kThreads) pack_f16_kernel(const uint16_t* __restrict__ src,
                                                            uint16_t* __restrict__ dst, size_t n,
                                                            int* fault) {
  uint32_t mx = 0u;
  const size_t n8 = n / 8;
  for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < n8;
       i += (size_t)gridDim.x * kThreads) {
    const uint4 v = reinterpret_cast<const uint4*>(src)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
      mx = max(mx, max(mag_bits(lo), mag_bits(hi)));
      asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(o[j]) : "f"(hi), "f"(lo));
    }
    reinterpret_cast<uint4*>(dst)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  // tail (n not a multiple of 8)
  const size_t t = n8 * 8 + (size_t)blockIdx.x * kThreads + threadIdx.x;
  if (blockIdx.x == 0 && t < n) {
    const float v = __uint_as_float(((uint32_t)src[t]) << 16);
    mx = max(mx, mag_bits(v));
    uint32_t o;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(o) : "f"(0.0f), "f"(v));
    dst[t] = (uint16_t)(o & 0xFFFFu);
  }
  if (fault != nullptr && __any_sync(0xffffffffu, mx >= kF16Clamp) && (threadIdx.x & 31) == 0)
    atomicOr(fault, MOE_DEVFAULT_FP16_RANGE);
}

}  // namespace

cudaError_t launch_pack_f16(const uint16_t* src, uint16_t* dst, size_t n, int* fault,
                            cudaStream_t st) {
  long long grid = (long long)((n / 8 + kThreads - 1) / kThreads);
  const long long cap = (long long)num_sms() * 32;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  pack_f16_kernel<<<(unsigned)grid, kThreads, 0, st>>>(src, dst, n, fault);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Shape& s, const void* y, bool y_f32, const int32_t* slot_pos,
                           uint16_t* out, cudaStream_t st) {
  const bool may_drop = s.C < s.TK;  // a slot may be dropped
  if (y_f32)
    return may_drop ? launch_combine_variant<true, true>(s, y, slot_pos, out, st)
                    : launch_combine_variant<false, true>(s, y, slot_pos, out, st);
  return may_drop ? launch_combine_variant<true, false>(s, y, slot_pos, out, st)
                  : launch_combine_variant<false, false>(s, y, slot_pos, out, st);
}

}  // namespace moe
