// Router: logits = x . W_g in fp32 (CUDA-core FFMA), selection score, top-k with lower-index
// tie-breaking, softmax gates. One kernel; logits never leave shared memory.
//
// Method: "大模型MoE稀疏激活原理与工程实践", §3.1 路由器 (linear router without bias, top-k with
// sorted=True, softmax over the selected logits); bias-adjusted selection from
// "AI架构演进从稀疏MoE到条件记忆的工程实践" (gating-network code); Gumbel scores from
// "GPT-4 Has 1.8 Trillion Parameters. It Uses 2% of Them Per Token", §3.1 门控网络.
#include <cuda_runtime.h>
#include <cstdint>
#include <climits>
#include <cmath>

#include "internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kKC = 32;  // d-chunk per shared-memory stage

struct RouterArgs {
  const uint16_t* x;
  const uint16_t* W_g;
  const float* bias;
  const float* u;
  int32_t* topk_idx;
  float* topk_w;
  int T, d, E, k, mode;
  float tau;
  int EL;  // threads along experts (each covers 4 consecutive experts per 4*EL block)
  int EQ;  // 4*EL-wide expert blocks per thread
  int EP;  // padded expert row length in shared memory = 4*EL*EQ
  int TM;  // tokens per CTA = 4 * (kThreads / EL)
};

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// a beats b: higher score, or equal score and lower expert index
__device__ __forceinline__ bool beats(float sa, int ea, float sb, int eb) {
  return sa > sb || (sa == sb && ea < eb);
}

__global__ void __launch_bounds__(kThreads) router_kernel(RouterArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* xs = sm;                          // [kKC][TM]   x chunk, token-minor
  float* wsm = xs + kKC * a.TM;            // [kKC][EP]   W_g chunk, zero-padded past E
  float* lg = wsm + kKC * a.EP;            // [TM][E + 1] logits of this CTA's tokens

  const int tid = threadIdx.x;
  const int el = tid % a.EL, tg = tid / a.EL;
  const int t0 = blockIdx.x * a.TM;

  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[i][c] = 0.f;

  for (int k0 = 0; k0 < a.d; k0 += kKC) {
    // x chunk: each thread moves 8 bf16 (16 B) of one token row
    for (int idx = tid; idx < a.TM * (kKC / 8); idx += kThreads) {
      const int q = idx % (kKC / 8), i = idx / (kKC / 8);
      const int t = t0 + i;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < a.T) v = *reinterpret_cast<const uint4*>(a.x + (size_t)t * a.d + k0 + 8 * q);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        xs[(8 * q + 2 * r) * a.TM + i] = bf16f(w4[r] & 0xFFFFu);
        xs[(8 * q + 2 * r + 1) * a.TM + i] = bf16f(w4[r] >> 16);
      }
    }
    for (int idx = tid; idx < kKC * a.EP; idx += kThreads) {
      const int j = idx / a.EP, e = idx % a.EP;
      wsm[idx] = (e < a.E) ? bf16f(a.W_g[(size_t)(k0 + j) * a.E + e]) : 0.f;
    }
    __syncthreads();
    // two-level fp32 summation: a fresh partial per chunk, then added to the running sum
    float part[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < 8; ++c) part[i][c] = 0.f;
#pragma unroll 4
    for (int j = 0; j < kKC; ++j) {
      const float4 xv = *reinterpret_cast<const float4*>(xs + j * a.TM + 4 * tg);
      const float xr[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (q < a.EQ) {
          const float4 wv =
              *reinterpret_cast<const float4*>(wsm + j * a.EP + 4 * el + 4 * a.EL * q);
          const float wr[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) part[i][4 * q + c] = fmaf(xr[i], wr[c], part[i][4 * q + c]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[i][c] += part[i][c];
    __syncthreads();
  }

  // logits to shared memory
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = 4 * el + 4 * a.EL * q + c;
        if (q < a.EQ && e < a.E) lg[(4 * tg + i) * (a.E + 1) + e] = acc[i][4 * q + c];
      }
  __syncthreads();

  // top-k + gates: one warp per token
  const int warp = tid >> 5, lane = tid & 31;
  for (int i = warp; i < a.TM; i += kThreads / 32) {
    const int t = t0 + i;
    if (t >= a.T) break;
    float sv[8], av[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = lane + 32 * q;
      sv[q] = -INFINITY;
      av[q] = 0.f;
      if (e < a.E) {
        const float l = lg[i * (a.E + 1) + e];
        float s = l;
        if (a.mode == MOE_ROUTE_BIAS_SELECT) {
          s = l + a.bias[e];
        } else if (a.mode == MOE_ROUTE_GUMBEL) {
          const float g = -logf(-logf(a.u[(size_t)t * a.E + e]));
          s = (l + g) / a.tau;
        }
        if (s != s) s = -INFINITY;  // NaN ranks last
        sv[q] = s;
        av[q] = (a.mode == MOE_ROUTE_GUMBEL) ? s : l;
      }
    }
    uint32_t used = 0;
    int esel[8];
    float asel[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      esel[j] = 0;
      asel[j] = 0.f;
      if (j < a.k) {
        float bs = -INFINITY, ba = 0.f;
        int be = INT_MAX;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int e = lane + 32 * q;
          if (e < a.E && !((used >> q) & 1u) && beats(sv[q], e, bs, be)) {
            bs = sv[q];
            be = e;
            ba = av[q];
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float os = __shfl_xor_sync(0xffffffffu, bs, off);
          const int oe = __shfl_xor_sync(0xffffffffu, be, off);
          const float oa = __shfl_xor_sync(0xffffffffu, ba, off);
          if (beats(os, oe, bs, be)) {
            bs = os;
            be = oe;
            ba = oa;
          }
        }
        if ((be & 31) == lane) used |= 1u << (be >> 5);
        esel[j] = be;
        asel[j] = ba;
      }
    }
    float m = asel[0];
#pragma unroll
    for (int j = 1; j < 8; ++j)
      if (j < a.k) m = fmaxf(m, asel[j]);
    float ex[8], sum = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ex[j] = (j < a.k) ? expf(asel[j] - m) : 0.f;
      sum += ex[j];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < a.k && lane == j) {
        a.topk_idx[(size_t)t * a.k + j] = esel[j];
        a.topk_w[(size_t)t * a.k + j] = ex[j] / sum;
      }
    }
  }
}

}  // namespace

cudaError_t launch_router(const Shape& s, const uint16_t* x, const uint16_t* W_g,
                          const float* bias, const float* u, int32_t* topk_idx, float* topk_w,
                          cudaStream_t st) {
  RouterArgs a;
  a.x = x;
  a.W_g = W_g;
  a.bias = bias;
  a.u = u;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.T = s.T;
  a.d = s.d;
  a.E = s.E;
  a.k = s.k;
  a.mode = s.mode;
  a.tau = s.tau;
  int need = (s.E + 3) / 4;
  int el = 1;
  while (el < need && el < 32) el *= 2;
  a.EL = el;
  a.EQ = (s.E + 4 * el - 1) / (4 * el);  // <= 2 for E <= 256
  a.EP = 4 * el * a.EQ;
  a.TM = 4 * (kThreads / el);
  const size_t smem = sizeof(float) * ((size_t)kKC * a.TM + (size_t)kKC * a.EP +
                                       (size_t)a.TM * (s.E + 1));
  cudaError_t err =
      cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int grid = (s.T + a.TM - 1) / a.TM;
  router_kernel<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
