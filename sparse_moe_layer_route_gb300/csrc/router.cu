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
// Two kernels (plus the per-call weight preparation):
//  * router_gemm_kernel: CTA (row tile of 128 tokens, K slice). Warp 0 streams x tiles [128 x 64]
//    (K-major) and W_g chunks [64 x 64] (expert-major, i.e. N-major) with TMA; warp 1 issues
//    tcgen05.mma (M=128, N=E rounded up to 64, K=16) into TMEM; warps 4-7 write the fp32 partial
//    logits of the slice. Splitting K fills the GPU when T is small (one row tile at decode).
//  * select_kernel: 32 tokens per CTA, 8 threads per token. The K-slice partials summed in slice
//    order, selection scores, top-(k+1) by k+1 argmax passes (each thread over its eighth of the
//    experts, then a 3-step shuffle reduction), softmax gates and the near-tie test.
//  * refine_kernel: the exact re-decision of the near-tie tokens (below).
//
// Exactness. The tensor core's fp32 accumulation differs from an exactly rounded dot product by
// up to ~4e-5 on unit-scale logits at d = 7168 (measured), which is above the 1e-5 near-tie
// margin of the parity contract. So a token whose top-(k+1) scores have an adjacent gap below a
// conservative band (router_band: 2.5e-4 x sqrt(d / 7168) x max(1, |largest logit of the row|),
// about 6x the largest measured error) is flagged together with its candidate experts: every
// expert whose tensor-core score lies within the band of the k-th score (only those can be in
// the exact top-k), or all experts when there are more than 16 of them or the group decision of
// group-limited routing is itself that close. refine_kernel recomputes the candidates' logits as
// plain fp32 dot products (error ~1e-7) and re-decides the token's top-k and gates. Tokens outside
// the band cannot change their selection or order under the tensor-core error. Flagged tokens are
// appended to a list (order irrelevant: each token is re-decided on its own) and spread over all
// refine CTAs, a whole CTA per token, which keeps the pass short however the flags cluster.
#include <cuda.h>
#include <cuda_runtime.h>
#include <climits>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "route_common.cuh"

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
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
};

// Partial logits of one K slice: part[split][t][0, EP) (fp32; columns >= E are zero).
template <int NCH>
__global__ void __launch_bounds__(kThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmW, float* __restrict__ part, int T,
                       int kb_per_split, int k_blocks, int* status) {
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

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kBM;
  const int split = blockIdx.y;
  const int kb0 = split * kb_per_split;
  const int kb1 = min(k_blocks, kb0 + kb_per_split);

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
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();  // the setup above touched only shared memory, TMEM and parameters

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------------- TMA producer
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!ptx::mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, status,
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
        if (issued & (1u << s))
          ptx::mbar_wait_bounded(full_bar(s), (last_par >> s) & 1u, never, status,
                                 MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs / 4);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!ptx::mbar_wait_bounded(full_bar(stage), phase, abort_flag, status,
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
          ptx::umma_f16(tmem_base, adesc, bdesc, IDESC, (kb > kb0 || kk) ? 1u : 0u);
        }
        ptx::umma_commit(empty_bar(stage));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) ptx::umma_commit(acc_bar);
      ptx::umma_commit(done_bar);
      ptx::mbar_wait_bounded(done_bar, 0, never, status, MOE_DEVFAULT_PIPELINE_TIMEOUT,
                             kWaitLimitNs / 4);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue: partials out
    const int q = warp - 4;
    const int t = m0 + 32 * q + lane;
    if (ptx::mbar_wait_bounded(acc_bar, 0, abort_flag, status, MOE_DEVFAULT_PIPELINE_TIMEOUT,
                               kWaitLimitNs)) {
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16);
      float* dst = part + ((size_t)split * T + t) * C::EP;
#pragma unroll 1
      for (int c = 0; c < C::EP / 32; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(taddr + c * 32, v);
        ptx::tmem_wait_ld();
        if (t < T) {
          float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
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

struct SelectArgs {
  const float* part;   // [splits, T, EP]
  const float* bias;
  const float* u;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* ncand;     // [T]: 0 = decided; n > 0 = near-tie with n candidates; -1 = all E
  int32_t* cand;      // [T, kMaxCand]
  int32_t* rlist;     // near-tie tokens, appended
  int* rcount;        // their number (reset to 0 by the refine kernel when it finishes)
  float* sfull;       // [T, E] selection scores for the overflow re-route, or nullptr
  float* maxl_out;    // [T] largest |logit| of each row (with sfull)
  int T, E, EP, k, mode, d, splits;
  int G, Gk;          // group-limited routing (G = 0: off)
  float tau;
};

constexpr int kSelRows = 32;              // tokens per selection CTA
constexpr int kSelP = 8;                  // threads per token
constexpr int kSelThreads = kSelRows * kSelP;

// Group-limited routing: group scores (largest member score), the Gk best groups (ties to the
// lower group) as a bit mask, and the gap between the Gk-th and the next group score.
__device__ __forceinline__ unsigned long long pick_groups(const float* gm, int G, int Gk,
                                                          float* gap) {
  unsigned long long sel = 0ull;
  float ps_g = INFINITY, kth = INFINITY, next = -INFINITY;
  int pg = -1;
  const int passes = Gk < G ? Gk + 1 : Gk;
  for (int j = 0; j < passes; ++j) {
    float bs = -INFINITY;
    int bg = INT_MAX;
    for (int gi = 0; gi < G; ++gi) {
      const float v = gm[gi];
      const bool after = v < ps_g || (v == ps_g && gi > pg);
      if (after && beats(v, gi, bs, bg)) {
        bs = v;
        bg = gi;
      }
    }
    if (j < Gk) {
      sel |= 1ull << bg;
      kth = bs;
    } else {
      next = bs;
    }
    ps_g = bs;
    pg = bg;
  }
  *gap = Gk < G ? kth - next : INFINITY;
  return sel;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelectArgs a) {
  extern __shared__ __align__(16) float ssm[];
  const int LD = a.EP + 4;  // rows stay 16-byte aligned; 128-bit reads of consecutive rows
                            // hit distinct banks
  float* scores = ssm;                                        // [32][LD]
  float* maxl = scores + kSelRows * LD;                       // [32]
  float* gmax = maxl + kSelRows;                              // [32][G]
  unsigned long long* gsel =
      reinterpret_cast<unsigned long long*>(gmax + kSelRows * (a.G > 0 ? a.G : 0));  // [32]
  float* gmarg = reinterpret_cast<float*>(gsel + kSelRows);   // [32]
  griddep_wait();
  const bool gumbel = a.mode == MOE_ROUTE_GUMBEL;
  const int t0 = blockIdx.x * kSelRows;
  const int rows = min(kSelRows, a.T - t0);
  // phase 1: the block's partial-logit tiles with coalesced 16-byte loads (every K slice of four
  // groups in flight together), summed in slice order and turned into selection scores
  int* maxl_bits = reinterpret_cast<int*>(maxl);  // |logit| >= 0: int order = float order
  if (threadIdx.x < kSelRows) maxl_bits[threadIdx.x] = 0;
  __syncthreads();
  {
    const int ep4 = a.EP / 4;
    const float4* __restrict__ P = reinterpret_cast<const float4*>(a.part);
#pragma unroll 4
    for (int i = threadIdx.x; i < rows * ep4; i += kSelThreads) {
      const int rr = i / ep4, c = (i - rr * ep4) * 4;
      const int tt = t0 + rr;
      float4 v[8];
#pragma unroll
      for (int sp = 0; sp < 8; ++sp)
        if (sp < a.splits) v[sp] = __ldg(P + ((size_t)sp * a.T + tt) * ep4 + c / 4);
      float4 acc = v[0];
#pragma unroll
      for (int sp = 1; sp < 8; ++sp)
        if (sp < a.splits) {
          acc.x += v[sp].x;
          acc.y += v[sp].y;
          acc.z += v[sp].z;
          acc.w += v[sp].w;
        }
      const float lv[4] = {acc.x, acc.y, acc.z, acc.w};
      float m = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = c + q;
        float sc = -INFINITY;
        if (e < a.E) {
          m = fmaxf(m, fabsf(lv[q]));
          sc = selection_score(a.mode, lv[q],
                               a.mode == MOE_ROUTE_BIAS_SELECT ? __ldg(a.bias + e) : 0.f,
                               gumbel ? __ldg(a.u + (size_t)tt * a.E + e) : 0.f, a.tau);
        }
        scores[rr * LD + e] = sc;
      }
      atomicMax(&maxl_bits[rr], __float_as_int(m));
    }
  }
  __syncthreads();
  if (a.sfull != nullptr) {
    // the overflow re-route ranks every expert of a token: keep the scores and the row scale
    for (int i = threadIdx.x; i < rows * a.E; i += kSelThreads) {
      const int rr = i / a.E, e = i - rr * a.E;
      a.sfull[(size_t)(t0 + rr) * a.E + e] = scores[rr * LD + e];
    }
    if (threadIdx.x < rows) a.maxl_out[t0 + threadIdx.x] = maxl[threadIdx.x];
  }
  const int r = threadIdx.x / kSelP, h = threadIdx.x % kSelP;
  const int t = t0 + r;
  const bool row_ok = r < rows;
  float* srow = scores + r * LD;
  const int chunk = ((a.E + kSelP - 1) / kSelP + 3) & ~3;  // multiple of 4: float4 reads
  const int e_lo = h * chunk, e_hi = min(a.E, e_lo + chunk);
  if (a.G > 0) {
    // group-limited routing: experts outside the kept groups get -inf
    const int gsz = a.E / a.G;
    if (row_ok)
      for (int gi = h; gi < a.G; gi += kSelP) {
        float m = -INFINITY;
        for (int e = gi * gsz; e < (gi + 1) * gsz; ++e) m = fmaxf(m, srow[e]);
        gmax[r * a.G + gi] = m;
      }
    __syncthreads();
    if (row_ok && h == 0) gsel[r] = pick_groups(gmax + r * a.G, a.G, a.Gk, &gmarg[r]);
    __syncthreads();
    if (row_ok) {
      const unsigned long long sel = gsel[r];
      for (int e = e_lo; e < e_hi; ++e)
        if (!((sel >> (e / gsz)) & 1ull)) srow[e] = -INFINITY;
    }
    __syncwarp();
  }
  const int k = a.k;
  const int nl = k < a.E ? k + 1 : k;  // top-(k+1), or all E when k == E
  // pass j: the best expert strictly after pick j-1 in (score desc, index asc) order; each of
  // the token's 8 threads scans its experts, then a shuffle reduction over the 8 lanes
  float pick_s[kList];
  int pick_e[kList];
  float ps = INFINITY;
  int pe = -1;
#pragma unroll
  for (int j = 0; j < kList; ++j) {
    if (j < nl) {
      float bs[2] = {-INFINITY, -INFINITY};
      int be[2] = {INT_MAX, INT_MAX};
      if (row_ok) {
        const float4* s4 = reinterpret_cast<const float4*>(srow);
#pragma unroll 1
        for (int e = e_lo; e < e_hi; e += 8) {
          // may read up to 7 floats past this thread's range (still inside the row's padded
          // storage or the next row); those lanes fail the ee < e_hi test below
          const float4 v0 = s4[e >> 2], v1 = s4[(e >> 2) + 1];
          const float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int ee = e + q;
            const float sc = vv[q];
            const bool after = sc < ps || (sc == ps && ee > pe);
            if (ee < e_hi && after && beats(sc, ee, bs[q & 1], be[q & 1])) {
              bs[q & 1] = sc;
              be[q & 1] = ee;
            }
          }
        }
      }
      if (beats(bs[1], be[1], bs[0], be[0])) {
        bs[0] = bs[1];
        be[0] = be[1];
      }
#pragma unroll
      for (int off = kSelP / 2; off > 0; off >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, bs[0], off);
        const int oe = __shfl_xor_sync(0xffffffffu, be[0], off);
        if (beats(os, oe, bs[0], be[0])) {
          bs[0] = os;
          be[0] = oe;
        }
      }
      pick_s[j] = bs[0];
      pick_e[j] = be[0];
      ps = bs[0];
      pe = be[0];
    }
  }
  if (row_ok && h == 0) {
    // near-tie test (scores in their own units: GUMBEL scores carry 1/tau)
    float min_gap = INFINITY;
#pragma unroll
    for (int j = 1; j < kList; ++j)
      if (j < nl) min_gap = fminf(min_gap, pick_s[j - 1] - pick_s[j]);
    float sk = pick_s[0];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j == k - 1) sk = pick_s[j];
    float band = router_band(a.d, maxl[r]);
    if (gumbel) band /= a.tau;
    int nc = 0;
    if (a.G > 0 && gmarg[r] < band) {
      nc = -1;  // the group decision itself is uncertain: recompute every expert exactly
      a.rlist[atomicAdd(a.rcount, 1)] = t;
    } else if (min_gap < band) {
      // candidates: every expert scoring within the band of the k-th score
      for (int e = 0; e < a.E; ++e) {
        if (srow[e] >= sk - band) {
          if (nc < kMaxCand) a.cand[(size_t)t * kMaxCand + nc] = e;
          ++nc;
        }
      }
      nc = nc <= kMaxCand ? nc : -1;
      a.rlist[atomicAdd(a.rcount, 1)] = t;
    }
    a.ncand[t] = nc;
    {
      // gates: softmax over the selected logits (PLAIN: the score; BIAS_SELECT: score - bias,
      // within one rounding of the logit) or over the selected scores (GUMBEL)
      float av[kMaxK];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < k) {
          av[j] = a.mode == MOE_ROUTE_BIAS_SELECT ? pick_s[j] - a.bias[pick_e[j]] : pick_s[j];
          mx = fmaxf(mx, av[j]);
        }
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < k) {
          av[j] = expf(av[j] - mx);
          sum += av[j];
        }
      const float inv = 1.0f / sum;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < k) {
          a.topk_idx[(size_t)t * k + j] = pick_e[j];
          a.topk_w[(size_t)t * k + j] = av[j] * inv;
        }
    }
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
    const int32_t* __restrict__ cand, const int32_t* __restrict__ rlist, int* rcount, int* rdone,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int T, int d, int E, int k,
    int mode, float tau, int G, int Gk) {
  __shared__ float red[kThreads / 32][kMaxCand];
  __shared__ int ce[256];
  __shared__ float cl[256], cs[256];
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nf = *(volatile int*)rcount;
  for (int fi = blockIdx.x; fi < nf; fi += gridDim.x) {
    const int t = rlist[fi];
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
    if (threadIdx.x == 0 && n_c < 0 && G > 0) {
      // all experts recomputed (candidates are 0..E-1 in order): redo the group decision
      const int gsz = E / G;
      unsigned long long sel = 0ull;
      float ps_g = INFINITY;
      int pg = -1;
      for (int j = 0; j < Gk; ++j) {
        float bs = -INFINITY;
        int bg = INT_MAX;
        for (int gi = 0; gi < G; ++gi) {
          float v = -INFINITY;
          for (int e = gi * gsz; e < (gi + 1) * gsz; ++e) v = fmaxf(v, cs[e]);
          const bool after = v < ps_g || (v == ps_g && gi > pg);
          if (after && beats(v, gi, bs, bg)) {
            bs = v;
            bg = gi;
          }
        }
        sel |= 1ull << bg;
        ps_g = bs;
        pg = bg;
      }
      for (int e = 0; e < E; ++e)
        if (!((sel >> (e / gsz)) & 1ull)) cs[e] = -INFINITY;
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
  // the last CTA to finish resets the list for the next call (all CTAs have read the count)
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(rdone, 1) == (int)gridDim.x - 1) {
      *rcount = 0;
      *rdone = 0;
    }
  }
}

template <int NCH>
cudaError_t launch_gemm(const CUtensorMap& mx, const CUtensorMap& mw, float* part, int T,
                        int n_mt, int splits, int kb_per_split, int k_blocks, int* status,
                        cudaStream_t st) {
  using C = RCfg<NCH>;
  cudaError_t err = cudaFuncSetAttribute(router_gemm_kernel<NCH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
  if (err != cudaSuccess) return err;
  return launch_k(router_gemm_kernel<NCH>, dim3(n_mt, splits), dim3(kThreads), C::kSmemBytes, st,
                  mx, mw, part, T, kb_per_split, k_blocks, status);
}

}  // namespace

int router_splits(int T, int d) {
  const int n_mt = (T + kBM - 1) / kBM;
  const int k_blocks = d / kBK;
  int sp = 152 / n_mt;  // fill the GPU's SMs with (row tile, K slice) CTAs
  // at most 8 slices (the selection reads every slice) and at least 4 K blocks per slice
  const int cap = k_blocks / 4 < 8 ? (k_blocks / 4 > 1 ? k_blocks / 4 : 1) : 8;
  if (sp > cap) sp = cap;
  if (sp < 1) sp = 1;
  const int kbs = (k_blocks + sp - 1) / sp;  // no empty slice
  return (k_blocks + kbs - 1) / kbs;
}

cudaError_t launch_router(const Shape& s, const uint16_t* x, const uint16_t* W_g,
                          const float* bias, const float* u, int32_t* topk_idx, float* topk_w,
                          const RouterScratch& rs, int* status, cudaStream_t st) {
  const int EP = (s.E + 63) / 64 * 64;
  const uint16_t* W = EP != s.E ? rs.wg_pad : W_g;
  {
    const dim3 grid((s.d + 31) / 32, (EP + 31) / 32);
    const cudaError_t e = launch_k(prep_router_kernel, grid, dim3(kThreads), 0, st, W_g, rs.wg_t,
                                   EP != s.E ? rs.wg_pad : nullptr, s.d, s.E, EP);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mx, mw;
  if (!make_tmap_2d(&mx, x, s.T, s.d, kBK, kBM) || !make_tmap_2d(&mw, W, s.d, EP, 64, kBK))
    return cudaErrorInvalidValue;
  const int n_mt = (s.T + kBM - 1) / kBM;
  const int k_blocks = s.d / kBK;
  const int splits = router_splits(s.T, s.d);
  const int kbs = (k_blocks + splits - 1) / splits;
  cudaError_t err;
  switch (EP / 64) {
    case 1: err = launch_gemm<1>(mx, mw, rs.part, s.T, n_mt, splits, kbs, k_blocks, status, st); break;
    case 2: err = launch_gemm<2>(mx, mw, rs.part, s.T, n_mt, splits, kbs, k_blocks, status, st); break;
    case 3: err = launch_gemm<3>(mx, mw, rs.part, s.T, n_mt, splits, kbs, k_blocks, status, st); break;
    default: err = launch_gemm<4>(mx, mw, rs.part, s.T, n_mt, splits, kbs, k_blocks, status, st); break;
  }
  if (err != cudaSuccess) return err;
  SelectArgs a;
  a.part = rs.part;
  a.bias = bias;
  a.u = u;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.ncand = rs.ncand;
  a.cand = rs.cand;
  a.rlist = rs.rlist;
  a.rcount = rs.rcount;
  a.sfull = rs.sfull;
  a.maxl_out = rs.maxl;
  a.T = s.T;
  a.E = s.E;
  a.EP = EP;
  a.k = s.k;
  a.mode = s.mode;
  a.d = s.d;
  a.splits = splits;
  a.G = s.G;
  a.Gk = s.Gk;
  a.tau = s.tau;
  const size_t smem =
      sizeof(float) * ((size_t)kSelRows * (EP + 4) + kSelRows + (size_t)kSelRows * s.G +
                       2 * kSelRows + kSelRows);
  err = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
  if (err != cudaSuccess) return err;
  err = launch_k(select_kernel, dim3((s.T + kSelRows - 1) / kSelRows), dim3(kSelThreads), smem,
                 st, a);
  if (err != cudaSuccess) return err;
  const int rgrid = 2 * num_sms();
  return launch_k(refine_kernel, dim3(rgrid), dim3(kThreads), 0, st, x, (const uint16_t*)rs.wg_t,
                  bias, u, (const int32_t*)rs.ncand, (const int32_t*)rs.cand,
                  (const int32_t*)rs.rlist, rs.rcount, rs.rdone, topk_idx, topk_w, s.T, s.d, s.E,
                  s.k, s.mode, s.tau, s.G, s.Gk);
}

}  // namespace moe
