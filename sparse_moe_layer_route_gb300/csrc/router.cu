// Router: logits = x . W_g on the tensor cores (bf16 inputs, fp32 accumulation in TMEM), then
// per token the selection score, top-k with lower-index tie-breaking and softmax gates. The GEMM
// writes fp32 partial logits per K slice ([splits, T, EP], a few MB that stay in L2) and the
// selection kernel adds them; the full logits exist only in the selection's registers.
//
// Method: "大模型MoE稀疏激活原理与工程实践", §3.1 路由器 (linear router without bias, top-k with
// sorted=True, softmax over the selected logits); bias-adjusted selection from
// "AI架构演进从稀疏MoE到条件记忆的工程实践" (gating-network code); Gumbel scores
// (logits - log(-log u)) / tau from "GPT-4 Has 1.8 Trillion Parameters. It Uses 2% of Them Per
// Token", §3.1 门控网络.
//
// Three kernels, after the one-time transpose of W_g (transpose_router_kernel, through
// moe_prepare_router, or per call when the caller has no transposed copy):
//  * router_gemm_kernel: CTA (row tile of 128 tokens, K slice). Warp 0 streams x tiles [128 x 64]
//    and W_g^T tiles [E rounded up to 64 x 64] (both K-major) with TMA; warp 1 issues tcgen05.mma
//    (M=128, N=E rounded up to 64, K=16) into TMEM, one fresh accumulator per 64-deep K block;
//    warps 4-11 add the blocks in fp32 registers and write the slice's partial logits. Splitting
//    K fills the GPU when T is small (one row tile at decode).
//  * select_kernel: one warp per token. The K-slice partials summed in slice order, selection
//    scores, top-(k+1) by k+1 warp-wide key reductions (largest key, then the lowest expert index
//    holding it), softmax gates and the near-tie test.
//  * refine_kernel: the exact re-decision of the near-tie tokens (below).
//
// Exactness. The logits differ from exactly rounded dot products by at most 7.9e-7 x max(1,
// |largest logit of the row|) at d = 7168 (measured; see router_gemm_kernel for why each K block
// gets its own accumulator), so the gates, a softmax over the selected logits, stay within 1e-5
// of exact. An order decided on a score gap below that error could still differ from the exact
// one, and the parity contract exempts only gaps below 1e-5. So a token whose top-(k+1) scores
// have an adjacent gap below a band (router_band: 1.5e-5 x sqrt(d / 7168) x max(1, |largest
// logit of the row|), about 9x the largest measured error of a logit difference) is flagged
// together with its candidate experts: every expert whose score lies within the band of the
// k-th score (only those can be in the exact top-k), or all experts when there are more than 16
// of them or the group decision of group-limited routing is itself that close. refine_kernel
// recomputes the candidates' logits as plain fp32 dot products (error ~1e-7) and re-decides the
// token's top-k and gates. Tokens outside the band cannot change their selection or order under
// the GEMM's error. Flagged tokens are appended to a list (order irrelevant: each token is
// re-decided on its own) and spread over all refine CTAs, a whole CTA per token, which keeps the
// pass short however the flags cluster.
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

constexpr int kThreads = 256;      // selection-side kernels
constexpr int kGemmThreads = 384;  // router GEMM: warps 0 TMA, 1 MMA, 2 TMEM, 4-11 epilogue
constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB
constexpr int kMaxK = 8;
constexpr int kList = kMaxK + 1;  // top-(k+1) list: the (k+1)-th score bounds the selection gap
constexpr int kMaxCand = 16;      // candidate experts recorded per near-tie token
constexpr uint64_t kWaitLimitNs = 2000000000ull;

template <int NCH>
struct RCfg {
  static constexpr int EP = 64 * NCH;                  // MMA N (experts rounded up to 64)
  static constexpr int kBBytes = EP * kBK * 2;         // W_g^T rows [EP experts x 64 k]
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (192 * 1024 / kStageBytes) > 8 ? 8 : (192 * 1024 / kStageBytes);
  // one fresh accumulator per K block; the epilogue adds each into fp32 registers while the
  // next blocks accumulate in the other buffers
  static constexpr int kNAcc = EP <= 128 ? 4 : 2;
  static constexpr int kTmemCols = kNAcc * EP <= 256 ? 256 : 512;
  static constexpr int kHalf = EP / 2;                 // columns per epilogue thread
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
};

// Partial logits of one K slice: part[split][t][0, EP) (fp32; columns >= E are zero).
//
// Accumulation. tcgen05.mma adds its products into the fp32 accumulator after aligning them
// to the accumulator's exponent, and the bits shifted out are lost; summed over the d/16 MMAs of
// a long dot product against a growing accumulator this drifts by up to ~4e-5 on unit-scale
// logits at d = 7168 (measured). So every 64-deep K block starts from a zero accumulator (its
// partial sum stays small, and so does that loss), and the epilogue adds the blocks in K order
// in fp32 registers with round-to-nearest adds. Four (EP <= 128) or two accumulators rotate so
// the MMAs of later blocks run while the epilogue reads earlier ones.
template <int NCH>
__global__ void __launch_bounds__(kGemmThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmW, float* __restrict__ part, int T,
                       int kb_per_split, int k_blocks, int* status, int* rcount) {
  using C = RCfg<NCH>;
  constexpr int kStages = C::kStages;
  constexpr int NACC = C::kNAcc;
  constexpr int HALF = C::kHalf;
  // A = x rows (K-major), B = W_g^T rows (K-major): both 128-byte swizzled [rows][64 k]
  constexpr uint32_t IDESC = ptx::idesc_f16kind_f32(kBM, C::EP, 0, 0, 1);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + kStages * C::kStageBytes;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto afull_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto aempty_bar = [&](int b) { return bar0 + 8u * (2 * kStages + NACC + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * kStages + 2 * NACC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kStages * C::kStageBytes +
                                                    8 * (2 * kStages + 2 * NACC + 1));
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
    for (int b = 0; b < NACC; ++b) {
      ptx::mbar_init(afull_bar(b), 1);
      ptx::mbar_init(aempty_bar(b), 8);  // the eight epilogue warps
    }
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
  // the near-tie list of this call starts empty: the selection (the next kernel) appends to it
  // and the previous call's refine pass, which read it, has completed
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *rcount = 0;

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
        // experts >= E lie past the map's rows: the copy fills them with zeros
        ptx::tma_load_2d(sA + kABytes, &tmW, fb, kb * kBK, 0);
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
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!ptx::mbar_wait_bounded(aempty_bar(acc), acc_phase ^ 1u, abort_flag, status,
                                    MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs))
          break;
        if (!ptx::mbar_wait_bounded(full_bar(stage), phase, abort_flag, status,
                                    MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs))
          break;
        ptx::tc_fence_after();
        const uint32_t sA = base + stage * C::kStageBytes;
        const uint32_t sB = sA + kABytes;
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::EP);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t adesc = ptx::smem_desc_sw128(sA + kk * 32, 16, 1024);
          const uint64_t bdesc = ptx::smem_desc_sw128(sB + kk * 32, 16, 1024);
          ptx::umma_f16(d_tmem, adesc, bdesc, IDESC, kk ? 1u : 0u);
        }
        ptx::umma_commit(empty_bar(stage));
        ptx::umma_commit(afull_bar(acc));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++acc == NACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      ptx::umma_commit(done_bar);
      ptx::mbar_wait_bounded(done_bar, 0, never, status, MOE_DEVFAULT_PIPELINE_TIMEOUT,
                             kWaitLimitNs / 4);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------ epilogue: K blocks summed, partials out
    const int q = warp & 3;          // TMEM lanes [32q, 32q + 32): rows of the tile
    const int h = (warp - 4) >> 2;   // columns [h * HALF, h * HALF + HALF)
    const int t = m0 + 32 * q + lane;
    float sum[HALF];
#pragma unroll
    for (int i = 0; i < HALF; ++i) sum[i] = 0.f;
    const uint32_t trow = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * HALF);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!ptx::mbar_wait_bounded_warp(afull_bar(acc), acc_phase, abort_flag, status,
                                       MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
#pragma unroll
      for (int c = 0; c < HALF / 32; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(trow + (uint32_t)(acc * C::EP + c * 32), v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) sum[c * 32 + i] += __uint_as_float(v[i]);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(aempty_bar(acc));
      if (++acc == NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (ok && t < T) {
      float4* d4 = reinterpret_cast<float4*>(part + ((size_t)split * T + t) * C::EP + h * HALF);
#pragma unroll
      for (int i = 0; i < HALF / 4; ++i)
        d4[i] = make_float4(sum[4 * i], sum[4 * i + 1], sum[4 * i + 2], sum[4 * i + 3]);
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
  int32_t* rrec;      // near-tie records, appended (layout: kRouterRecInts)
  int* rcount;        // their number (cleared by the router GEMM before this kernel runs)
  float* sfull;       // [T, E] selection scores for the overflow re-route, or nullptr
  float* maxl_out;    // [T] largest |logit| of each row (with sfull)
  int T, E, EP, k, mode, d, splits;
  int G, Gk;          // group-limited routing (G = 0: off)
  float tau;
};

constexpr int kSelWarps = 8;              // tokens per selection CTA: one warp each
constexpr int kSelThreads = kSelWarps * 32;
constexpr int kSelMaxPerLane = 8;         // experts per lane: E <= 256

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

// Order-preserving 32-bit key of a selection score (NaN already mapped to -inf): a larger score
// gives a larger key, -0 and +0 the same key, and every score a key above 0, which marks experts
// that are taken or do not exist.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t b = __float_as_uint(s);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// One warp per token. Lane l holds experts [l*m, l*m + m) (m = ceil(E/32)): it sums their
// partial logits over the K slices in slice order, forms their selection scores, and keeps their
// keys. Each of the k+1 picks, in (score desc, index asc) order, is the warp's largest key, then
// the smallest expert index among the lanes holding that key; the owner marks it taken.
// M >= m is the compiled bound on experts per lane (1, 2, 4 or 8): the per-expert loops are
// unrolled to M rather than to the largest supported E, so small E runs no predicated-off work.
// v[i] = p[i] for i < n (else 0): one or M / 4 vector loads when the whole run is there and
// aligned, scalar loads otherwise.
template <int M>
__device__ __forceinline__ void load_run(const float* p, int n, float (&v)[M]) {
  constexpr int VB = M % 4 == 0 ? 16 : (M == 2 ? 8 : 0);  // vector bytes
  if (VB != 0 && n == M && (reinterpret_cast<uintptr_t>(p) % VB) == 0) {
    if (M == 2) {
      const float2 f = __ldg(reinterpret_cast<const float2*>(p));
      v[0] = f.x;
      v[M - 1] = f.y;
    } else {
#pragma unroll
      for (int c = 0; c < M / 4; ++c) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(p) + c);
        v[4 * c] = f.x;
        v[4 * c + 1] = f.y;
        v[4 * c + 2] = f.z;
        v[4 * c + 3] = f.w;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < M; ++i) v[i] = i < n ? __ldg(p + i) : 0.f;
  }
}

// p[i] = v[i] for i < n, the same way.
template <int M>
__device__ __forceinline__ void store_run(float* p, int n, const float (&v)[M]) {
  constexpr int VB = M % 4 == 0 ? 16 : (M == 2 ? 8 : 0);
  if (VB != 0 && n == M && (reinterpret_cast<uintptr_t>(p) % VB) == 0) {
    if (M == 2) {
      *reinterpret_cast<float2*>(p) = make_float2(v[0], v[M - 1]);
    } else {
#pragma unroll
      for (int c = 0; c < M / 4; ++c)
        reinterpret_cast<float4*>(p)[c] =
            make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < M; ++i)
      if (i < n) p[i] = v[i];
  }
}

template <int M>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelectArgs a) {
  static_assert(M >= 1 && M <= kSelMaxPerLane, "experts per lane");
  __shared__ uint32_t gkey[kSelWarps][64];  // group-limited routing: group maxima
  __shared__ float gsc[kSelWarps][64];
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSelWarps + warp;
  if (t >= a.T) return;
  const bool gumbel = a.mode == MOE_ROUTE_GUMBEL;
  const int m = (a.E + 31) >> 5;
  const int e0 = lane * m;
  float sc[M];
  uint32_t key[M];
  float maxabs = 0.f;
  // this lane's logits: the slices added in slice order; when the lane holds exactly M experts
  // (e0 = lane * M, 4 M-byte aligned) each slice comes in M / 4 float4 (or one float2) loads
  float lg[M];
  {
    const float* p = a.part + (size_t)t * a.EP + e0;
    const size_t stride = (size_t)a.T * a.EP;
    if (m == M && (M == 2 || M % 4 == 0)) {
      // every slice's load issued before the first add
      float v[8][M];
#pragma unroll
      for (int sp = 0; sp < 8; ++sp) {
        const float* q = p + sp * stride;
        if (M == 2) {
          const float2 f = sp < a.splits ? __ldg(reinterpret_cast<const float2*>(q))
                                         : make_float2(0.f, 0.f);
          v[sp][0] = f.x;
          v[sp][M - 1] = f.y;
        } else {
#pragma unroll
          for (int c = 0; c < M / 4; ++c) {
            const float4 f = sp < a.splits ? __ldg(reinterpret_cast<const float4*>(q) + c)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
            v[sp][4 * c] = f.x;
            v[sp][4 * c + 1] = f.y;
            v[sp][4 * c + 2] = f.z;
            v[sp][4 * c + 3] = f.w;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < M; ++i) {
        lg[i] = v[0][i];
#pragma unroll
        for (int sp = 1; sp < 8; ++sp)
          if (sp < a.splits) lg[i] += v[sp][i];
      }
    } else {
#pragma unroll
      for (int i = 0; i < M; ++i) {
        lg[i] = 0.f;
        if (i < m && e0 + i < a.E) {
          float v[8];
#pragma unroll
          for (int sp = 0; sp < 8; ++sp)
            v[sp] = sp < a.splits ? __ldg(p + i + sp * stride) : 0.f;
          float l = v[0];
#pragma unroll
          for (int sp = 1; sp < 8; ++sp)
            if (sp < a.splits) l += v[sp];
          lg[i] = l;
        }
      }
    }
  }
  // this lane's experts [e0, e0 + nv) and their bias or Gumbel draws
  const int nv = max(0, min(m, a.E - e0));
  float bv[M], uv[M];
#pragma unroll
  for (int i = 0; i < M; ++i) bv[i] = uv[i] = 0.f;
  if (a.mode == MOE_ROUTE_BIAS_SELECT) load_run<M>(a.bias + e0, nv, bv);
  if (gumbel) load_run<M>(a.u + (size_t)t * a.E + e0, nv, uv);
#pragma unroll
  for (int i = 0; i < M; ++i) {
    sc[i] = -INFINITY;
    key[i] = 0u;
    if (i < nv) {
      const float l = lg[i];
      maxabs = fmaxf(maxabs, fabsf(l));
      sc[i] = selection_score(a.mode, l, bv[i], uv[i], a.tau);
      key[i] = score_key(sc[i]);
    }
  }
  // |logit| >= 0: its bits order as the value
  maxabs = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(maxabs)));
  if (a.sfull != nullptr) {
    // the overflow re-route ranks every expert of a token: keep the scores and the row scale
    store_run<M>(a.sfull + (size_t)t * a.E + e0, nv, sc);
    if (lane == 0) a.maxl_out[t] = maxabs;
  }
  float gmarg = INFINITY;
  if (a.G > 0) {
    // group-limited routing: experts outside the Gk best groups get -inf
    const int gsz = a.E / a.G;
    for (int g = lane; g < a.G; g += 32) gkey[warp][g] = 0u;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < M; ++i)
      if (i < m && e0 + i < a.E) atomicMax(&gkey[warp][(e0 + i) / gsz], key[i]);
    __syncwarp();
    for (int g = lane; g < a.G; g += 32) gsc[warp][g] = key_score(gkey[warp][g]);
    __syncwarp();
    unsigned long long sel = 0ull;
    if (lane == 0) sel = pick_groups(gsc[warp], a.G, a.Gk, &gmarg);
    sel = __shfl_sync(0xffffffffu, sel, 0);
    gmarg = __shfl_sync(0xffffffffu, gmarg, 0);
#pragma unroll
    for (int i = 0; i < M; ++i)
      if (i < m && e0 + i < a.E && !((sel >> ((e0 + i) / gsz)) & 1ull)) {
        sc[i] = -INFINITY;
        key[i] = score_key(-INFINITY);
      }
  }
  // this lane's best remaining expert (lowest index among equal keys)
  auto lane_best = [&](uint32_t& bk, int& be) {
    bk = 0u;
    be = INT_MAX;
#pragma unroll
    for (int i = 0; i < M; ++i) {
      const bool better = i < m && key[i] > bk;
      bk = better ? key[i] : bk;
      be = better ? e0 + i : be;
    }
  };
  uint32_t bk;
  int be;
  lane_best(bk, be);
  const int k = a.k;
  const int nl = k < a.E ? k + 1 : k;  // top-(k+1), or all E when k == E
  float prev = 0.f, min_gap = INFINITY, sk = -INFINITY;
  float my_s = 0.f;  // lane j < k: pick j
  int my_e = 0;
#pragma unroll
  for (int j = 0; j < kList; ++j) {
    if (j >= nl) break;  // uniform over the warp
    const uint32_t K = __reduce_max_sync(0xffffffffu, bk);
    const int W = (int)__reduce_min_sync(0xffffffffu, bk == K ? (uint32_t)be : 0xffffffffu);
    const float s_j = key_score(K);
    my_s = lane == j ? s_j : my_s;
    my_e = lane == j ? W : my_e;
    if (j > 0) min_gap = fminf(min_gap, prev - s_j);
    if (j == k - 1) sk = s_j;
    prev = s_j;
    // every lane drops the pick (only its owner holds it) and rescans: no divergent branch
#pragma unroll
    for (int i = 0; i < M; ++i) key[i] = e0 + i == W ? 0u : key[i];
    lane_best(bk, be);
  }
  // near-tie test (scores in their own units: GUMBEL scores carry 1/tau)
  float band = router_band(a.d, maxabs);
  if (gumbel) band /= a.tau;
  // a listed token gets a record: the token, then -1 (re-decide every expert) or its candidates,
  // every expert scoring within the band of the k-th score, in index order
  const bool group_tie = a.G > 0 && gmarg < band;
  if (group_tie || min_gap < band) {
    int mine = 0;
    if (!group_tie) {
#pragma unroll
      for (int i = 0; i < M; ++i)
        if (i < m && e0 + i < a.E && sc[i] >= sk - band) ++mine;
    }
    int before = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, before, off);
      if (lane >= off) before += o;
    }
    int nc = __shfl_sync(0xffffffffu, before, 31);
    before -= mine;
    nc = (!group_tie && nc <= kMaxCand) ? nc : -1;
    int slot = 0;
    if (lane == 0) slot = atomicAdd(a.rcount, 1);
    int32_t* rec = a.rrec + (size_t)__shfl_sync(0xffffffffu, slot, 0) * kRouterRecInts;
    if (lane == 0) {
      rec[0] = t;
      rec[1] = nc;
    }
    if (nc > 0) {
#pragma unroll
      for (int i = 0; i < M; ++i)
        if (i < m && e0 + i < a.E && sc[i] >= sk - band) rec[2 + before++] = e0 + i;
    }
  }
  // gates: softmax over the selected logits (PLAIN: the score; BIAS_SELECT: score - bias,
  // within one rounding of the logit) or over the selected scores (GUMBEL); lane j holds pick j
  float av = -INFINITY;
  if (lane < k) av = a.mode == MOE_ROUTE_BIAS_SELECT ? my_s - __ldg(a.bias + my_e) : my_s;
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j)
    if (j < k) mx = fmaxf(mx, __shfl_sync(0xffffffffu, av, j));
  const float ex = lane < k ? expf(av - mx) : 0.f;
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j)
    if (j < k) sum += __shfl_sync(0xffffffffu, ex, j);
  if (lane < k) {
    a.topk_idx[(size_t)t * k + lane] = my_e;
    a.topk_w[(size_t)t * k + lane] = ex * (1.0f / sum);
  }
}

// Router weight transpose: WgT[e, j] = W_g[j, e], each expert's weights contiguous. The router
// GEMM reads it as its K-major B operand and the exact passes (near-tie re-decision, overflow
// re-route) read one expert's row at a time. Weight preparation: once per weight set through
// moe_prepare_router, or per call when the caller passes no transposed copy.
// 32 x 32 tiles through shared memory so both sides are coalesced.
__global__ void __launch_bounds__(kThreads) transpose_router_kernel(
    const uint16_t* __restrict__ W, uint16_t* __restrict__ WgT, int d, int E) {
  __shared__ uint16_t tile[32][33];
  griddep_wait();
  // the router GEMM may start its setup; it waits for this kernel before reading WgT
  griddep_launch_dependents();
  const int j0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int r = ty; r < 32; r += 8) {
    const int j = j0 + r, e = e0 + tx;
    tile[r][tx] = (j < d && e < E) ? W[(size_t)j * E + e] : (uint16_t)0;
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
    const float* __restrict__ u, const int32_t* __restrict__ rrec, const int* rcount,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int T, int d, int E, int k,
    int mode, float tau, int G, int Gk) {
  __shared__ float red[kThreads / 32][kMaxCand];
  __shared__ int ce[256];
  __shared__ float cl[256], cs[256];
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the first record is read together with the count (a record past the count is never used)
  int4 rv[(2 + kMaxCand) / 4 + 1];
  auto load_rec = [&](int fi) {
    const int4* rp = reinterpret_cast<const int4*>(rrec + (size_t)fi * kRouterRecInts);
#pragma unroll
    for (int i = 0; i < (2 + kMaxCand) / 4 + 1; ++i) rv[i] = rp[i];
  };
  if (blockIdx.x < T) load_rec(blockIdx.x);
  const int nf = *rcount;
  for (int fi = blockIdx.x; fi < nf; fi += gridDim.x) {
    if (fi != (int)blockIdx.x) load_rec(fi);
    const int* rec = reinterpret_cast<const int*>(rv);
    const int t = rec[0];
    const int n_c = rec[1];
    const int nc = n_c > 0 ? n_c : E;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    const int d8 = d / 8;
    for (int c0 = 0; c0 < nc; c0 += kMaxCand) {
      const int cn = min(kMaxCand, nc - c0);
      // this chunk's experts, read by every thread (the candidate list is 64 bytes)
      // this chunk's experts (a listed chunk is the record's whole list: c0 = 0)
      int ec[kMaxCand];
#pragma unroll
      for (int c = 0; c < kMaxCand; ++c) ec[c] = c < cn ? (n_c > 0 ? rec[2 + c] : c0 + c) : 0;
      // warp 0's lane c < cn: its expert's bias / noise, loaded while the dot products run
      float bias_c = 0.f, u_c = 0.f;
      if (warp == 0 && lane < cn) {
        int e = c0 + lane;
#pragma unroll
        for (int c = 0; c < kMaxCand; ++c)
          if (c == lane) e = ec[c];
        if (mode == MOE_ROUTE_BIAS_SELECT) bias_c = bias[e];
        if (mode == MOE_ROUTE_GUMBEL) u_c = u[(size_t)t * E + e];
        ce[c0 + lane] = e;
      }
      float acc[kMaxCand];
#pragma unroll
      for (int c = 0; c < kMaxCand; ++c) acc[c] = 0.f;
      // thread i takes 8-column groups i, i + 256, ...: one 16-byte load of x and of each
      // candidate's contiguous row per group, all issued before the arithmetic
      for (int g = threadIdx.x; g < d8; g += kThreads) {
        const uint4 xv = xr[g];
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        uint4 wv[kMaxCand];
#pragma unroll
        for (int c = 0; c < kMaxCand; ++c)
          if (c < cn) wv[c] = reinterpret_cast<const uint4*>(WT + (size_t)ec[c] * d)[g];
#pragma unroll
        for (int c = 0; c < kMaxCand; ++c) {
          if (c < cn) {
            const uint32_t ww[4] = {wv[c].x, wv[c].y, wv[c].z, wv[c].w};
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
      if (warp == 0 && lane < cn) {
        float l = 0.f;
        for (int w = 0; w < kThreads / 32; ++w) l += red[w][lane];
        cl[c0 + lane] = l;
        cs[c0 + lane] = selection_score(mode, l, bias_c, u_c, tau);
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
    if (n_c < 0 && G > 0) __syncthreads();
    if (warp == 0) {
      // selection among the candidates by (score desc, index asc): lane l holds candidates
      // l, l + 32, ...; each pick is the warp's largest key, then the smallest expert index
      uint32_t key[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = lane + 32 * i;
        key[i] = c < nc ? score_key(cs[c]) : 0u;
      }
      float my_a = 0.f;
      int my_e = 0;
      for (int j = 0; j < k; ++j) {
        uint32_t bk = 0u;
        int be = INT_MAX, bi = -1;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = lane + 32 * i;
          if (key[i] > bk || (key[i] == bk && key[i] != 0u && ce[c] < be)) {
            bk = key[i];
            be = ce[c];
            bi = i;
          }
        }
        const uint32_t K = __reduce_max_sync(0xffffffffu, bk);
        const int W = (int)__reduce_min_sync(0xffffffffu, bk == K ? (uint32_t)be : 0xffffffffu);
        const bool mine = bk == K && be == W;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (mine && i == bi) key[i] = 0u;
        // the pick's gate input: the logit, or the score for GUMBEL
        const unsigned ow = __ballot_sync(0xffffffffu, mine);
        const int src = __ffs(ow) - 1;
        float av = 0.f;
        if (mine) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i == bi) av = mode == MOE_ROUTE_GUMBEL ? cs[lane + 32 * i] : cl[lane + 32 * i];
        }
        av = __shfl_sync(0xffffffffu, av, src);
        if (lane == j) {
          my_a = av;
          my_e = W;
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < k) mx = fmaxf(mx, __shfl_sync(0xffffffffu, my_a, j));
      const float ex = lane < k ? expf(my_a - mx) : 0.f;
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < k) sum += __shfl_sync(0xffffffffu, ex, j);
      if (lane < k) {
        topk_idx[(size_t)t * k + lane] = my_e;
        topk_w[(size_t)t * k + lane] = ex * (1.0f / sum);
      }
    }
    __syncthreads();
  }
}

template <int NCH>
cudaError_t launch_gemm(const CUtensorMap& mx, const CUtensorMap& mw, float* part, int T,
                        int n_mt, int splits, int kb_per_split, int k_blocks, int* status,
                        int* rcount, cudaStream_t st) {
  using C = RCfg<NCH>;
  cudaError_t err = cudaFuncSetAttribute(router_gemm_kernel<NCH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
  if (err != cudaSuccess) return err;
  return launch_k(router_gemm_kernel<NCH>, dim3(n_mt, splits), dim3(kGemmThreads), C::kSmemBytes,
                  st, mx, mw, part, T, kb_per_split, k_blocks, status, rcount);
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

cudaError_t launch_router_transpose(int d, int E, const uint16_t* W_g, uint16_t* W_g_t,
                                    cudaStream_t st) {
  const dim3 grid((d + 31) / 32, (E + 31) / 32);
  return launch_k(transpose_router_kernel, grid, dim3(kThreads), 0, st, W_g, W_g_t, d, E);
}

cudaError_t launch_router(const Shape& s, const uint16_t* x, const uint16_t* W_g,
                          const uint16_t* W_g_t, const float* bias, const float* u,
                          int32_t* topk_idx, float* topk_w, const RouterScratch& rs, int* status,
                          cudaStream_t st) {
  const int EP = (s.E + 63) / 64 * 64;
  cudaError_t err;
  if (W_g_t == nullptr) {
    // no prepared transpose: make one in the workspace for this call
    if ((err = launch_router_transpose(s.d, s.E, W_g, rs.wg_t, st)) != cudaSuccess) return err;
    W_g_t = rs.wg_t;
  }
  CUtensorMap mx, mw;
  if (!make_tmap_2d(&mx, x, s.T, s.d, kBK, kBM) || !make_tmap_2d(&mw, W_g_t, s.E, s.d, kBK, EP))
    return cudaErrorInvalidValue;
  const int n_mt = (s.T + kBM - 1) / kBM;
  const int k_blocks = s.d / kBK;
  const int splits = router_splits(s.T, s.d);
  const int kbs = (k_blocks + splits - 1) / splits;
  switch (EP / 64) {
    case 1: err = launch_gemm<1>(mx, mw, rs.part, s.T, n_mt, splits, kbs, k_blocks, status, rs.rcount, st); break;
    case 2: err = launch_gemm<2>(mx, mw, rs.part, s.T, n_mt, splits, kbs, k_blocks, status, rs.rcount, st); break;
    case 3: err = launch_gemm<3>(mx, mw, rs.part, s.T, n_mt, splits, kbs, k_blocks, status, rs.rcount, st); break;
    default: err = launch_gemm<4>(mx, mw, rs.part, s.T, n_mt, splits, kbs, k_blocks, status, rs.rcount, st); break;
  }
  if (err != cudaSuccess) return err;
  SelectArgs a;
  a.part = rs.part;
  a.bias = bias;
  a.u = u;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.rrec = rs.rrec;
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
  const int m = (s.E + 31) / 32;  // experts per lane
  const dim3 sgrid((s.T + kSelWarps - 1) / kSelWarps), sblock(kSelThreads);
  if (m <= 1)
    err = launch_k(select_kernel<1>, sgrid, sblock, 0, st, a);
  else if (m <= 2)
    err = launch_k(select_kernel<2>, sgrid, sblock, 0, st, a);
  else if (m <= 4)
    err = launch_k(select_kernel<4>, sgrid, sblock, 0, st, a);
  else
    err = launch_k(select_kernel<8>, sgrid, sblock, 0, st, a);
  if (err != cudaSuccess) return err;
  const int rgrid = num_sms();  // one CTA per SM (its registers allow no second)
  return launch_k(refine_kernel, dim3(rgrid), dim3(kThreads), 0, st, x, W_g_t,
                  bias, u, (const int32_t*)rs.rrec, (const int*)rs.rcount, topk_idx, topk_w, s.T,
                  s.d, s.E,
                  s.k, s.mode, s.tau, s.G, s.Gk);
}

}  // namespace moe
