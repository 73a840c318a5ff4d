// Router: logits = x . W_g on the tensor cores (bf16 inputs, fp32 accumulation in TMEM), then
// per token the selection score, top-k with lower-index tie-breaking and softmax gates, all in the
// epilogue. Logits never leave the chip.
//
// Method: "大模型MoE稀疏激活原理与工程实践", §3.1 路由器 (linear router without bias, top-k with
// sorted=True, softmax over the selected logits); bias-adjusted selection from
// "AI架构演进从稀疏MoE到条件记忆的工程实践" (gating-network code); Gumbel scores
// (logits - log(-log u)) / tau from "GPT-4 Has 1.8 Trillion Parameters. It Uses 2% of Them Per
// Token", §3.1 门控网络.
//
// One CTA per 128 tokens. Warp 0 streams x tiles [128 x 64] (K-major) and W_g chunks [64 x 64]
// (expert-major, i.e. N-major) with TMA into a 4-stage ring; warp 1 issues
// tcgen05.mma (M=128, N=E rounded up to 64, K=16); warps 4-7 each own 32 tokens (TMEM lanes):
// a thread turns its token's logits into selection scores 32 columns at a time, stages them in
// shared memory (its own row, bank-conflict-free), then takes the top-(k+1) by k+1 branch-free
// argmax passes over that row.
//
// Exactness. The tensor core's fp32 accumulation differs from an exactly rounded dot product by
// up to ~4e-5 on unit-scale logits at d = 7168 (measured), which is above the 1e-5 near-tie
// margin of the parity contract. So a token whose top-(k+1) scores have an adjacent gap below a
// conservative band (router_band: 2.5e-4 x sqrt(d / 7168) x max(1, |largest logit of the row|),
// about 6x the largest measured error) is flagged together with its candidate experts: every
// expert whose tensor-core score lies within the band of the k-th score (only those can be in
// the exact top-k). refine_kernel recomputes the candidates' logits as plain fp32 dot products
// (error ~1e-7) and re-decides the token's top-k and gates. Tokens outside the band cannot change
// their selection or order under the tensor-core error.
#include <cuda.h>
#include <cuda_runtime.h>
#include <climits>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB
constexpr int kChunkBytes = kBK * 64 * 2;  // 8 KB: 64 k-rows x 64 experts
constexpr int kMaxK = 8;
constexpr int kList = kMaxK + 1;  // top-(k+1) list: the (k+1)-th score bounds the selection gap
constexpr int kMaxCand = 16;      // candidate experts recorded per near-tie token
constexpr uint64_t kWaitLimitNs = 2000000000ull;

template <int NCH>
struct RCfg {
  static constexpr int EP = 64 * NCH;  // MMA N
  static constexpr int kStageBytes = kABytes + NCH * kChunkBytes;
  static constexpr int kStages = (192 * 1024 / kStageBytes) > 8 ? 8 : (192 * 1024 / kStageBytes);
  static constexpr int kTmemCols = EP <= 64 ? 64 : (EP <= 128 ? 128 : 256);
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256 + 256 * 4;
  // the epilogue stages scores [128 tokens][EP + 1] and the selection scratch (9 x 128 words)
  // in the (then idle) stage buffers
  static_assert((128 * (EP + 1) + 9 * 128) * 4 <= kStages * kStageBytes, "score staging fits");
};

struct RouterArgs {
  const float* bias;
  const float* u;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* ncand;  // [T]: 0 = decided; n > 0 = near-tie with n candidates; -1 = recompute all E
  int32_t* cand;   // [T, kMaxCand] candidate experts of near-tie tokens
  int* status;
  int T, E, k, mode, k_blocks, d;
  float tau;
};

// Half-width of the band around a gap inside which the tensor-core logits could misorder two
// experts (see the file comment).
__device__ __forceinline__ float router_band(int d, float max_abs_logit) {
  return 2.5e-4f * sqrtf((float)d * (1.0f / 7168.0f)) * fmaxf(1.0f, max_abs_logit);
}

__device__ __forceinline__ float selection_score(int mode, float l, float bias_e, float u_te,
                                                 float tau) {
  float s = l;
  if (mode == MOE_ROUTE_BIAS_SELECT) {
    s = l + bias_e;
  } else if (mode == MOE_ROUTE_GUMBEL) {
    const float g = -logf(-logf(u_te));
    s = (l + g) / tau;
  }
  return (s != s) ? -INFINITY : s;  // NaN ranks last
}

// a beats b: higher score, or equal score and lower expert index
__device__ __forceinline__ bool beats(float sa, int ea, float sb, int eb) {
  return sa > sb || (sa == sb && ea < eb);
}

template <int NCH>
__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW, const RouterArgs a) {
  using C = RCfg<NCH>;
  constexpr int kStages = C::kStages;
  constexpr uint32_t IDESC = ptx::idesc_f16kind_f32(kBM, C::EP, 0, 1, 1);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + kStages * C::kStageBytes;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t acc_bar = bar0 + 8u * (2 * kStages);
  const uint32_t done_bar = bar0 + 8u * (2 * kStages + 1);
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(gbase + kStages * C::kStageBytes + 8 * (2 * kStages + 2));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* never = reinterpret_cast<volatile int*>(tmem_slot + 2);  // stays 0
  float* bias_s = reinterpret_cast<float*>(gbase + kStages * C::kStageBytes + 256);
  // selection scratch (valid once the MMAs are done): scores [128][kLD], per-token max |logit|,
  // and the two halves' per-pass picks (double-buffered by pass parity)
  constexpr int kLD = C::EP + 1;
  float* sel_maxl = reinterpret_cast<float*>(gbase) + kBM * kLD;
  float(*sel_s)[2][kBM] = reinterpret_cast<float(*)[2][kBM]>(sel_maxl + kBM);
  int(*sel_e)[2][kBM] = reinterpret_cast<int(*)[2][kBM]>(sel_maxl + kBM + 4 * kBM);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kBM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    ptx::mbar_init(acc_bar, 1);
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    *never = 0;
    ptx::fence_mbarrier_init();
    ptx::prefetch_tmap(&tmX);
    ptx::prefetch_tmap(&tmW);
  }
  if (warp == 2) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  griddep_wait();  // the setup above touched only shared memory, TMEM and parameters
  if (warp == 3) {
    for (int e = lane; e < a.E; e += 32)
      bias_s[e] = (a.mode == MOE_ROUTE_BIAS_SELECT) ? a.bias[e] : 0.f;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------------- TMA producer
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      for (int kb = 0; kb < a.k_blocks; ++kb) {
        if (!ptx::mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, a.status,
                                    MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs))
          break;
        const uint32_t sA = base + stage * C::kStageBytes;
        const uint32_t fb = full_bar(stage);
        ptx::mbar_arrive_expect_tx(fb, C::kStageBytes);
        ptx::tma_load_2d(sA, &tmX, fb, kb * kBK, m0);
#pragma unroll
        for (int c = 0; c < NCH; ++c)
          ptx::tma_load_2d(sA + kABytes + c * kChunkBytes, &tmW, fb, c * 64, kb * kBK);
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      for (int s = 0; s < kStages; ++s)
        if (issued & (1u << s)) {
          ptx::mbar_wait_bounded(full_bar(s), (last_par >> s) & 1u, never, a.status,
                                 MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs / 4);
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < a.k_blocks; ++kb) {
        if (!ptx::mbar_wait_bounded(full_bar(stage), phase, abort_flag, a.status,
                                    MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sA = base + stage * C::kStageBytes;
        const uint32_t sB = sA + kABytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t adesc = ptx::smem_desc_sw128(sA + kk * 32, 16, 1024);
          const uint64_t bdesc = ptx::smem_desc_sw128(sB + kk * 2048, kChunkBytes, 1024);
          ptx::umma_f16(tmem_base, adesc, bdesc, IDESC, (kb | kk) != 0 ? 1u : 0u);
        }
        ptx::umma_commit(empty_bar(stage));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) ptx::umma_commit(acc_bar);
      ptx::umma_commit(done_bar);
      ptx::mbar_wait_bounded(done_bar, 0, never, a.status, MOE_DEVFAULT_PIPELINE_TIMEOUT,
                             kWaitLimitNs / 4);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue 1: stage scores
    const int q = warp - 4;
    const int r = 32 * q + lane;  // this thread's token within the tile
    const int t = m0 + r;
    const bool ok = ptx::mbar_wait_bounded(acc_bar, 0, abort_flag, a.status,
                                           MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs);
    if (ok) {
      ptx::tc_fence_after();
      // every MMA has completed, so the stage buffers are free: scores [128][EP + 1]
      float* srow = reinterpret_cast<float*>(gbase) + r * kLD;
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16);
      const bool row_ok = t < a.T;
      const bool gumbel = a.mode == MOE_ROUTE_GUMBEL;
      float max_abs_l = 0.f;
#pragma unroll 1
      for (int c = 0; c < C::EP / 32; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(taddr + c * 32, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c * 32 + i;
          const float l = __uint_as_float(v[i]);
          float sc = -INFINITY;
          if (row_ok && e < a.E) {
            max_abs_l = fmaxf(max_abs_l, fabsf(l));
            sc = selection_score(a.mode, l, bias_s[e], gumbel ? a.u[(size_t)t * a.E + e] : 0.f,
                                 a.tau);
          }
          srow[e] = sc;
        }
      }
      sel_maxl[r] = max_abs_l;
    }
  }

  // ------------------------------------------------------------------ epilogue 2: selection
  // All 256 threads: thread (r, h) scans half h of token r's experts; each pass picks the best
  // expert strictly after the previous pick in (score desc, index asc) order, with four
  // independent chains per thread; the two halves merge through shared memory.
  __syncthreads();
  if (!*abort_flag) {
    const int r = threadIdx.x & (kBM - 1), h = threadIdx.x >> 7;
    const int t = m0 + r;
    const bool row_ok = t < a.T;
    const float* srow = reinterpret_cast<const float*>(gbase) + r * kLD;
    const int k = a.k;
    const int nl = k < a.E ? k + 1 : k;  // top-(k+1), or all E when k == E
    const int half = (a.E + 1) / 2;
    const int e_lo = h * half, e_hi = min(a.E, e_lo + half);
    float ts[kList];
    int te[kList];
    float ps = INFINITY;
    int pe = -1;
#pragma unroll
    for (int j = 0; j < kList; ++j) {
      ts[j] = -INFINITY;
      te[j] = INT_MAX;
      if (j < nl) {  // uniform: nl depends on k and E only
        float bs[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        int be[4] = {INT_MAX, INT_MAX, INT_MAX, INT_MAX};
        if (row_ok) {
          for (int e = e_lo; e < e_hi; e += 4) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int ee = e + c;
              if (ee < e_hi) {
                const float sc = srow[ee];
                const bool after = sc < ps || (sc == ps && ee > pe);
                if (after && beats(sc, ee, bs[c], be[c])) {
                  bs[c] = sc;
                  be[c] = ee;
                }
              }
            }
          }
        }
#pragma unroll
        for (int c = 1; c < 4; ++c)
          if (beats(bs[c], be[c], bs[0], be[0])) {
            bs[0] = bs[c];
            be[0] = be[c];
          }
        sel_s[j & 1][h][r] = bs[0];
        sel_e[j & 1][h][r] = be[0];
        __syncthreads();
        const float os = sel_s[j & 1][h ^ 1][r];
        const int oe = sel_e[j & 1][h ^ 1][r];
        if (beats(os, oe, bs[0], be[0])) {
          bs[0] = os;
          be[0] = oe;
        }
        ts[j] = bs[0];
        te[j] = be[0];
        ps = bs[0];
        pe = be[0];
      }
    }
    if (row_ok && h == 0) {
      const bool gumbel = a.mode == MOE_ROUTE_GUMBEL;
      // near-tie test (scores in their own units: GUMBEL scores carry 1/tau)
      float min_gap = INFINITY, sk = ts[0];
#pragma unroll
      for (int j = 1; j < kList; ++j) {
        if (j < nl) min_gap = fminf(min_gap, ts[j - 1] - ts[j]);
        if (j == k - 1) sk = ts[j];
      }
      float band = router_band(a.d, sel_maxl[r]);
      if (gumbel) band /= a.tau;
      int nc = 0;
      if (min_gap < band) {
        // candidates: every expert scoring within the band of the k-th score
        for (int e = 0; e < a.E; ++e) {
          if (srow[e] >= sk - band) {
            if (nc < kMaxCand) a.cand[(size_t)t * kMaxCand + nc] = e;
            ++nc;
          }
        }
        nc = nc <= kMaxCand ? nc : -1;
      }
      a.ncand[t] = nc;
      // gates: softmax over the selected logits (PLAIN: the score; BIAS_SELECT: score - bias,
      // within one rounding of the logit) or over the selected scores (GUMBEL)
      float av[kMaxK];
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        av[j] = (a.mode == MOE_ROUTE_BIAS_SELECT && j < k) ? ts[j] - bias_s[te[j]] : ts[j];
      float mx = av[0];
#pragma unroll
      for (int j = 1; j < kMaxK; ++j)
        if (j < k) mx = fmaxf(mx, av[j]);
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        av[j] = (j < k) ? expf(av[j] - mx) : 0.f;
        sum += av[j];
      }
      const float inv = 1.0f / sum;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
          a.topk_idx[(size_t)t * k + j] = te[j];
          a.topk_w[(size_t)t * k + j] = av[j] * inv;
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// Router weight preparation, per call: WgT[e, j] = W_g[j, e] (each expert's weights contiguous,
// for the exact re-decision of near-tie tokens) and, when E is not a multiple of 64,
// Wp[j, e] = e < E ? W_g[j, e] : 0 for e < EP (zero columns for the MMA's padding experts).
// 32 x 32 tiles through shared memory so both sides are coalesced.
__global__ void __launch_bounds__(kThreads) prep_router_kernel(const uint16_t* __restrict__ W,
                                                               uint16_t* __restrict__ WgT,
                                                               uint16_t* __restrict__ Wp, int d,
                                                               int E, int EP) {
  __shared__ uint16_t tile[32][33];
  griddep_wait();
  const int j0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int r = ty; r < 32; r += 8) {
    const int j = j0 + r, e = e0 + tx;
    const uint16_t v = (j < d && e < E) ? W[(size_t)j * E + e] : (uint16_t)0;
    tile[r][tx] = v;
    if (Wp != nullptr && j < d && e < EP) Wp[(size_t)j * EP + e] = v;
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int e = e0 + r, j = j0 + tx;
    if (e < E && j < d) WgT[(size_t)e * d + j] = tile[tx][r];
  }
}

// Exact re-decision of the near-tie tokens, one CTA per token at a time: the logits of the
// token's candidate experts (all E when there were too many) as plain fp32 dot products over the
// transposed weights. Thread i sums its 8-column groups i, i + 256, ... in order; the 256
// partials are added by a fixed tree (warp shuffles, then the eight warp sums in warp order), so
// equal W_g columns give equal logits.
__global__ void __launch_bounds__(kThreads) refine_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ WT, const float* __restrict__ bias,
    const float* __restrict__ u, const int32_t* __restrict__ ncand,
    const int32_t* __restrict__ cand, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, int T, int d, int E, int k, int mode, float tau) {
  __shared__ float red[kThreads / 32][kMaxCand];
  __shared__ int ce[256];
  __shared__ float cl[256], cs[256];
  __shared__ int flagged[kThreads];
  __shared__ int n_flagged;
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's contiguous chunk of tokens; their flags are read 256 at a time in one round
  const int chunk = (T + gridDim.x - 1) / gridDim.x;
  const int t_begin = blockIdx.x * chunk;
  const int t_end = min(T, t_begin + chunk);
  for (int base = t_begin; base < t_end; base += kThreads) {
    if (threadIdx.x == 0) n_flagged = 0;
    __syncthreads();
    {
      const int tt = base + threadIdx.x;
      if (tt < t_end && ncand[tt] != 0) flagged[atomicAdd(&n_flagged, 1)] = tt;
    }
    __syncthreads();
    const int nf = n_flagged;
  for (int fi = 0; fi < nf; ++fi) {
    const int t = flagged[fi];
    const int n_c = ncand[t];
    const int nc = n_c > 0 ? n_c : E;
    for (int i = threadIdx.x; i < nc; i += kThreads)
      ce[i] = n_c > 0 ? cand[(size_t)t * kMaxCand + i] : i;
    __syncthreads();
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    const int d8 = d / 8;
    for (int c0 = 0; c0 < nc; c0 += kMaxCand) {
      const int cn = min(kMaxCand, nc - c0);
      float acc[kMaxCand];
#pragma unroll
      for (int c = 0; c < kMaxCand; ++c) acc[c] = 0.f;
      // thread i takes 8-column groups i, i + 256, ...: one 16-byte load of x and of each
      // candidate's contiguous row per group, all issued before the arithmetic
      for (int g = threadIdx.x; g < d8; g += kThreads) {
        const uint4 xv = xr[g];
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int c = 0; c < kMaxCand; ++c) {
          if (c < cn) {
            const uint4 wv =
                reinterpret_cast<const uint4*>(WT + (size_t)ce[c0 + c] * d)[g];
            const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
            float sacc = acc[c];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              sacc = fmaf(__uint_as_float(xw[h] << 16), __uint_as_float(ww[h] << 16), sacc);
              sacc = fmaf(__uint_as_float(xw[h] & 0xFFFF0000u), __uint_as_float(ww[h] & 0xFFFF0000u),
                          sacc);
            }
            acc[c] = sacc;
          }
        }
      }
#pragma unroll
      for (int c = 0; c < kMaxCand; ++c) {
        float v = acc[c];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) red[warp][c] = v;
      }
      __syncthreads();
      if (threadIdx.x < cn) {
        float l = 0.f;
        for (int w = 0; w < kThreads / 32; ++w) l += red[w][threadIdx.x];
        const int e = ce[c0 + threadIdx.x];
        cl[c0 + threadIdx.x] = l;
        cs[c0 + threadIdx.x] =
            selection_score(mode, l, mode == MOE_ROUTE_BIAS_SELECT ? bias[e] : 0.f,
                            mode == MOE_ROUTE_GUMBEL ? u[(size_t)t * E + e] : 0.f, tau);
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      // selection among the candidates by (score desc, index asc)
      uint32_t used[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      int esel[kMaxK];
      float asel[kMaxK];
      for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int i = 0; i < nc; ++i) {
          if ((used[i >> 5] >> (i & 31)) & 1u) continue;
          if (best < 0 || beats(cs[i], ce[i], cs[best], ce[best])) best = i;
        }
        used[best >> 5] |= 1u << (best & 31);
        esel[j] = ce[best];
        asel[j] = (mode == MOE_ROUTE_GUMBEL) ? cs[best] : cl[best];
      }
      float mx = asel[0];
      for (int j = 1; j < k; ++j) mx = fmaxf(mx, asel[j]);
      float ex[kMaxK], sum = 0.f;
      for (int j = 0; j < k; ++j) {
        ex[j] = expf(asel[j] - mx);
        sum += ex[j];
      }
      const float inv = 1.0f / sum;
      for (int j = 0; j < k; ++j) {
        topk_idx[(size_t)t * k + j] = esel[j];
        topk_w[(size_t)t * k + j] = ex[j] * inv;
      }
    }
    __syncthreads();
  }
    __syncthreads();  // the flag list is rebuilt for the next chunk only after every reader
  }
}

template <int NCH>
cudaError_t launch_tc(const CUtensorMap& mx, const CUtensorMap& mw, const RouterArgs& a, int grid,
                      cudaStream_t st) {
  using C = RCfg<NCH>;
  cudaError_t err = cudaFuncSetAttribute(router_tc_kernel<NCH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
  if (err != cudaSuccess) return err;
  return launch_k(router_tc_kernel<NCH>, dim3(grid), dim3(kThreads), C::kSmemBytes, st, mx, mw,
                  a);
}

}  // namespace

cudaError_t launch_router(const Shape& s, const uint16_t* x, const uint16_t* W_g,
                          const float* bias, const float* u, int32_t* topk_idx, float* topk_w,
                          uint16_t* wg_pad, uint16_t* wg_t, int32_t* ncand, int32_t* cand,
                          int* status, cudaStream_t st) {
  const int EP = (s.E + 63) / 64 * 64;
  const uint16_t* W = EP != s.E ? wg_pad : W_g;
  {
    const dim3 grid((s.d + 31) / 32, (EP + 31) / 32);
    const cudaError_t e = launch_k(prep_router_kernel, grid, dim3(kThreads), 0, st, W_g, wg_t,
                                   EP != s.E ? wg_pad : nullptr, s.d, s.E, EP);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mx, mw;
  if (!make_tmap_2d(&mx, x, s.T, s.d, kBK, kBM) || !make_tmap_2d(&mw, W, s.d, EP, 64, kBK))
    return cudaErrorInvalidValue;
  RouterArgs a;
  a.bias = bias;
  a.u = u;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.ncand = ncand;
  a.cand = cand;
  a.status = status;
  a.d = s.d;
  a.T = s.T;
  a.E = s.E;
  a.k = s.k;
  a.mode = s.mode;
  a.k_blocks = s.d / kBK;
  a.tau = s.tau;
  const int grid = (s.T + kBM - 1) / kBM;
  cudaError_t err;
  switch (EP / 64) {
    case 1: err = launch_tc<1>(mx, mw, a, grid, st); break;
    case 2: err = launch_tc<2>(mx, mw, a, grid, st); break;
    case 3: err = launch_tc<3>(mx, mw, a, grid, st); break;
    default: err = launch_tc<4>(mx, mw, a, grid, st); break;
  }
  if (err != cudaSuccess) return err;
  const int rgrid = s.T < 2 * num_sms() ? s.T : 2 * num_sms();
  return launch_k(refine_kernel, dim3(rgrid), dim3(kThreads), 0, st, x, (const uint16_t*)wg_t,
                  bias, u, (const int32_t*)ncand, (const int32_t*)cand, topk_idx, topk_w, s.T, s.d,
                  s.E, s.k, s.mode, s.tau);
}

}  // namespace moe
