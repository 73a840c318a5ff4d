// Level-2 overflow re-route ("参数规模与稀疏激活的真相拆解", §3.2 专家容量: overflow tokens are not
// dropped but handed to a fallback router that picks the next-best expert that is not full).
//
// Definition (the oracle's): after the Level-1 walk, the dropped slots are visited in slot order
// and each takes the best-scoring expert that still has room and that its token does not already
// use. That walk is sequential; the GPU computes the same assignment with token-proposing
// deferred acceptance, which reaches it because every expert ranks its proposers by one shared
// priority (the token number):
//
//   reroute_prep_kernel     one warp per token. A token with dropped slots sorts the experts it
//                           may still take (not its own, not already full after Level 1) by the
//                           router's tensor-core selection scores (a bitonic sort in registers),
//                           and orders the first window of that list exactly: every run of
//                           positions whose adjacent gaps lie inside the tensor-core error band
//                           is re-ordered by exact fp32 dot products. Also resets the per-expert
//                           state and the proposal bitmaps.
//   reroute_exact_kernel    the first windows that need exact dot products, a CTA per token
//                           (the prep kernel lists them instead of computing them per warp).
//   reroute_da_kernel       cooperative (all CTAs resident), rounds of
//                             A. every token with unmet demand proposes to its next experts,
//                                skipping experts already full with better tokens; a token that
//                                reaches the end of its exactly ordered window stops and is
//                                listed;
//                             B. every expert that got proposals keeps its `room` best (lowest
//                                token numbers; a bitmap over tokens, so ranks are popcounts) and
//                                turns the rest away; listed tokens get their next window ordered;
//                           until a round turns nobody away and lists nobody. Grid barriers wait
//                           with a bound.
//   reroute_finalize_kernel one warp per token: the experts that kept the token, in its
//                           preference order, fill its dropped slots in slot order; the gates of
//                           a re-routed token are the softmax over its final experts.
//
// Why windows: a token consumes a short prefix of its list (on the skewed prefill layer about 12
// positions on average, at most ~40 of 126), and ordering the whole list exactly would cost about
// five 7168-long dot products per token instead of under one.
//
// The caller then runs the dispatch again on the final expert indices.
#include <cuda_runtime.h>
#include <climits>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "route_common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxRounds = 1024;
constexpr int kWindow = 32;    // positions ordered exactly per window (then to the end of a run)
constexpr int kDotBatch = 4;   // exact dot products computed together
constexpr uint64_t kBarrierLimitNs = 2000000000ull;

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16); no completion to wait on.
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// float -> uint32 with the same order (every float but NaN; scores are never NaN here)
__device__ __forceinline__ uint32_t ordered_bits(float s) {
  const uint32_t b = __float_as_uint(s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Bitonic sort of 32 * V keys held by one warp (key i in register i / 32 of lane i % 32),
// descending: position 0 gets the largest key.
template <int V>
__device__ __forceinline__ void warp_sort_desc(uint32_t (&k)[V], int lane) {
  constexpr int N = 32 * V;
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
      if (j >= 32) {
        const int jv = j >> 5;
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const int pv = v ^ jv;
          if (pv > v) {
            const bool desc = ((v * 32 + lane) & size) == 0;
            const uint32_t x = k[v], y = k[pv];
            if (desc ? (x < y) : (x > y)) {
              k[v] = y;
              k[pv] = x;
            }
          }
        }
      } else {
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const uint32_t p = __shfl_xor_sync(0xffffffffu, k[v], j);
          const bool lower = (lane & j) == 0;
          const bool desc = ((v * 32 + lane) & size) == 0;
          k[v] = (lower == desc) ? max(k[v], p) : min(k[v], p);
        }
      }
    }
  }
}

// Per-warp scratch for one window: TC scores, experts and exact scores by window position,
// and the member positions whose exact score is needed.
struct WarpScratch {
  float* sw;
  float* ex;
  int* pe;
  int* mpos;
};

__device__ __forceinline__ WarpScratch warp_scratch(uint8_t* smem, int warp, int E) {
  float* base = reinterpret_cast<float*>(smem) + (size_t)warp * 4 * E;
  WarpScratch w;
  w.sw = base;
  w.ex = base + E;
  w.pe = reinterpret_cast<int*>(base + 2 * E);
  w.mpos = reinterpret_cast<int*>(base + 3 * E);
  return w;
}

__device__ __forceinline__ float window_band(const RerouteArgs& a, int t) {
  float band = router_band(a.d, a.maxl[t]);
  if (a.mode == MOE_ROUTE_GUMBEL) band /= a.tau;
  return band;
}

// Window positions [0, n) with a neighbour (inside the window) closer than the band, compacted
// into ws.mpos; returns their number. One warp; all lanes call it.
__device__ __forceinline__ int window_members(const WarpScratch& ws, int n, float band, int lane) {
  int nm = 0;
  for (int c0 = 0; c0 < n; c0 += 32) {
    const int i = c0 + lane;
    bool mem = false;
    if (i < n) {
      if (i > 0) mem = ws.sw[i - 1] - ws.sw[i] < band;
      if (i + 1 < n) mem = mem || ws.sw[i] - ws.sw[i + 1] < band;
    }
    const unsigned mm = __ballot_sync(0xffffffffu, mem);
    if (mem) ws.mpos[nm + __popc(mm & ((1u << lane) - 1u))] = i;
    nm += __popc(mm);
  }
  return nm;
}

// Each member moves to its exact rank inside its run (ws.ex holds the members' exact scores):
// pref[w0 + rank] = its expert. Threads j = first, first + step, ... take member j.
__device__ __forceinline__ void rank_members(const RerouteArgs& a, int t, int w0, int n,
                                             float band, const WarpScratch& ws, int nm,
                                             int first, int step) {
  uint8_t* prefw = a.pref + (size_t)t * a.PS;
  for (int m = first; m < nm; m += step) {
    const int i = ws.mpos[m];
    int lo = i, hi = i;
    while (lo > 0 && ws.sw[lo - 1] - ws.sw[lo] < band) --lo;
    while (hi + 1 < n && ws.sw[hi] - ws.sw[hi + 1] < band) ++hi;
    int r = lo;
    for (int i2 = lo; i2 <= hi; ++i2) r += beats(ws.ex[i2], ws.pe[i2], ws.ex[i], ws.pe[i]) ? 1 : 0;
    prefw[w0 + r] = (uint8_t)ws.pe[i];
  }
}

// Orders positions [w0, w1) of token t's list exactly, where w1 = min(L, w0 + kWindow) moved on
// to the end of the run it falls in; returns w1. Positions before w0 are already final and w0
// starts a run. The caller has put the experts and tensor-core scores of positions w0..L-1 into
// ws.pe / ws.sw (index = position - w0). One warp; all lanes call it. With defer (first windows,
// w0 = 0), a window that needs exact dot products is left in tensor-core order and its token
// listed for reroute_exact_kernel, which orders it the same way with a whole CTA.
__device__ int refine_window(const RerouteArgs& a, int t, int w0, int L, const WarpScratch& ws,
                             int lane, bool defer = false) {
  if (w0 >= L) return L;
  const int E = a.E;
  const float band = window_band(a, t);
  // window end: extend while the gap across it is inside the band
  const int m = L - w0;  // positions available
  int n = min(m, kWindow);
  while (n < m) {
    const int i = n + lane;  // gap between window positions i - 1 and i
    const bool linked = i < m && ws.sw[i - 1] - ws.sw[i] < band;
    const unsigned closed = ~__ballot_sync(0xffffffffu, linked);  // lanes past the list: closed
    if (closed) {
      n = min(m, n + __ffs(closed) - 1);
      break;
    }
    n = min(m, n + 32);
  }
  const int w1 = w0 + n;
  // members: positions with a neighbour inside the band
  const int nm = window_members(ws, n, band, lane);
  if (nm == 0) return w1;
  if (defer) {
    if (lane == 0) a.ex_list[atomicAdd(a.ex_count, 1)] = t;
    return w1;
  }
  __syncwarp();
  // exact selection scores of the members, kDotBatch dot products per pass over x
  const uint4* x4 = reinterpret_cast<const uint4*>(a.x + (size_t)t * a.d);
  const int d8 = a.d / 8;
  for (int b0 = 0; b0 < nm; b0 += kDotBatch) {
    const int nb = min(kDotBatch, nm - b0);
    const uint4* w4[kDotBatch];
#pragma unroll
    for (int c = 0; c < kDotBatch; ++c)
      w4[c] = reinterpret_cast<const uint4*>(
          a.WgT + (size_t)ws.pe[ws.mpos[b0 + (c < nb ? c : 0)]] * a.d);
    float acc[kDotBatch];
#pragma unroll
    for (int c = 0; c < kDotBatch; ++c) acc[c] = 0.f;
#pragma unroll 4
    for (int g = lane; g < d8; g += 32) {
      const uint4 xv = x4[g];
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int c = 0; c < kDotBatch; ++c) {
        if (c < nb) {
          const uint4 wv = w4[c][g];
          const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
          float s = acc[c];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            s = fmaf(__uint_as_float(xw[h] << 16), __uint_as_float(ww[h] << 16), s);
            s = fmaf(__uint_as_float(xw[h] & 0xFFFF0000u), __uint_as_float(ww[h] & 0xFFFF0000u),
                     s);
          }
          acc[c] = s;
        }
      }
    }
#pragma unroll
    for (int c = 0; c < kDotBatch; ++c) {
      float v = acc[c];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == c && c < nb) {
        const int i = ws.mpos[b0 + c];
        const int e = ws.pe[i];
        ws.ex[i] = selection_score(a.mode, v, a.mode == MOE_ROUTE_BIAS_SELECT ? a.bias[e] : 0.f,
                                   a.mode == MOE_ROUTE_GUMBEL ? a.u[(size_t)t * E + e] : 0.f,
                                   a.tau);
      }
    }
  }
  __syncwarp();
  rank_members(a, t, w0, n, band, ws, nm, lane, 32);
  __syncwarp();
  return w1;
}

// ws.pe / ws.sw for positions w0..L-1 of token t's list, from global memory
__device__ void load_list(const RerouteArgs& a, int t, int w0, int L, const WarpScratch& ws,
                          int lane) {
  for (int i = lane; i < L - w0; i += 32) {
    const int e = a.pref[(size_t)t * a.PS + w0 + i];
    ws.pe[i] = e;
    ws.sw[i] = a.sfull[(size_t)t * a.E + e];
  }
  __syncwarp();
}

template <int V>
__device__ void prep_token(const RerouteArgs& a, int t, int lane, const WarpScratch& ws) {
  int dropped = 0, own_e = -1;
  if (lane < a.k) {
    dropped = a.slot_pos[(size_t)t * a.k + lane] < 0;
    own_e = a.topk_idx[(size_t)t * a.k + lane];
  }
  const unsigned dmask = __ballot_sync(0xffffffffu, dropped);
  int own[8];  // the token's experts (k <= 8), the same in every lane
#pragma unroll
  for (int j = 0; j < 8; ++j) own[j] = __shfl_sync(0xffffffffu, own_e, j);
  if (lane == 0) {
    a.dem[t] = __popc(dmask);
    a.ptr[t] = 0;
    a.held[t] = 0;
  }
  if (dmask == 0u) return;
  // keys of the experts the token may still take (not its own, not full after Level 1): the
  // score's order-preserving bits with the low 8 replaced by 255 - e. Two scores that this
  // truncation puts out of order land next to each other with a negative gap, which is inside
  // the band, so the exact pass below orders them.
  uint32_t key[V];
  int L = 0;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int e = v * 32 + lane;
    bool ok = e < a.E;
    if (ok) {
      ok = a.counts[e] < a.C;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < a.k && own[j] == e) ok = false;
    }
    key[v] = ok ? (ordered_bits(a.sfull[(size_t)t * a.E + e]) & 0xFFFFFF00u) | (255u - e) : 0u;
    L += __popc(__ballot_sync(0xffffffffu, ok));
  }
  warp_sort_desc<V>(key, lane);
  uint8_t* pref = a.pref + (size_t)t * a.PS;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int i = v * 32 + lane;
    if (i < L) {
      const int e = 255 - (int)(key[v] & 0xFFu);
      pref[i] = (uint8_t)e;
      ws.pe[i] = e;
      ws.sw[i] = a.sfull[(size_t)t * a.E + e];
    }
  }
  __syncwarp();
  const int r = refine_window(a, t, 0, L, ws, lane, /*defer=*/true);
  if (lane == 0) {
    a.plen[t] = L;
    a.rlen[t] = r;
  }
}

template <int V>
__global__ void __launch_bounds__(kThreads) reroute_prep_kernel(const RerouteArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WarpScratch ws = warp_scratch(smem, warp, a.E);
  griddep_wait();
  // per-call reset of the shared state of the proposal rounds
  const int gtid = blockIdx.x * kThreads + threadIdx.x;
  const int nthr = gridDim.x * kThreads;
  const size_t nbits = (size_t)a.E * a.W;
  for (size_t i = gtid; i < nbits; i += nthr) a.bits[i] = 0u;
  for (int e = gtid; e < a.E; e += nthr) {
    const int kept = a.counts[e] < a.C ? a.counts[e] : a.C;
    a.room[e] = a.C - kept;
    a.cut[e] = INT_MAX;
    a.touched[e] = 0;
  }
  for (int i = gtid; i < kMaxRounds; i += nthr) {
    a.rejected[i] = 0;
    a.extended[i] = 0;
  }
  if (gtid == 0) {
    a.ctl[0] = 0;  // barrier arrivals
    a.ctl[1] = 0;  // barrier generation
  }
  for (int t = blockIdx.x * kWarps + warp; t < a.T; t += gridDim.x * kWarps)
    prep_token<V>(a, t, lane, ws);
}

// The first windows the prep kernel listed: the same ordering as refine_window, with the exact
// dot products spread over a whole CTA (each thread a strided share of the d / 8 16-byte chunks,
// one round of loads for d up to 8192) instead of one warp (seven dependent rounds at d = 7168).
// A CTA per listed token at a time; the partial sums are added by a fixed tree (shuffles, then
// the warps in order), so results are deterministic.
__global__ void __launch_bounds__(kThreads) reroute_exact_kernel(const RerouteArgs a) {
  __shared__ float s_sw[256], s_ex[256];
  __shared__ int s_pe[256], s_mpos[256];
  __shared__ float red[kWarps][kDotBatch];
  __shared__ int s_nm;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WarpScratch ws;
  ws.sw = s_sw;
  ws.ex = s_ex;
  ws.pe = s_pe;
  ws.mpos = s_mpos;
  griddep_wait();
  const int count = *a.ex_count;
  const int d8 = a.d / 8;
  if (threadIdx.x == 0 && blockIdx.x < count)
    l2_prefetch(a.x + (size_t)a.ex_list[blockIdx.x] * a.d, (uint32_t)a.d * 2u);
  for (int li = blockIdx.x; li < count; li += gridDim.x) {
    const int t = a.ex_list[li];
    // the next listed token's x row comes into L2 while this one is ordered
    if (threadIdx.x == 0 && li + gridDim.x < count)
      l2_prefetch(a.x + (size_t)a.ex_list[li + gridDim.x] * a.d, (uint32_t)a.d * 2u);
    const int n = a.rlen[t];  // the window the prep kernel closed, positions [0, n)
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const int e = a.pref[(size_t)t * a.PS + i];
      s_pe[i] = e;
      s_sw[i] = a.sfull[(size_t)t * a.E + e];
    }
    __syncthreads();
    const float band = window_band(a, t);
    if (warp == 0) {
      const int nm = window_members(ws, n, band, lane);
      if (lane == 0) s_nm = nm;
    }
    __syncthreads();
    const int nm = s_nm;
    const uint4* x4 = reinterpret_cast<const uint4*>(a.x + (size_t)t * a.d);
    for (int b0 = 0; b0 < nm; b0 += kDotBatch) {
      const int nb = min(kDotBatch, nm - b0);
      const uint4* w4[kDotBatch];
#pragma unroll
      for (int c = 0; c < kDotBatch; ++c)
        w4[c] = reinterpret_cast<const uint4*>(a.WgT + (size_t)s_pe[s_mpos[b0 + (c < nb ? c : 0)]] *
                                                          a.d);
      float acc[kDotBatch];
#pragma unroll
      for (int c = 0; c < kDotBatch; ++c) acc[c] = 0.f;
#pragma unroll 4
      for (int g = threadIdx.x; g < d8; g += kThreads) {
        const uint4 xv = x4[g];
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int c = 0; c < kDotBatch; ++c) {
          if (c < nb) {
            const uint4 wv = w4[c][g];
            const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
            float v = acc[c];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              v = fmaf(__uint_as_float(xw[h] << 16), __uint_as_float(ww[h] << 16), v);
              v = fmaf(__uint_as_float(xw[h] & 0xFFFF0000u), __uint_as_float(ww[h] & 0xFFFF0000u),
                       v);
            }
            acc[c] = v;
          }
        }
      }
#pragma unroll
      for (int c = 0; c < kDotBatch; ++c) {
        float v = acc[c];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) red[warp][c] = v;
      }
      __syncthreads();
      if (threadIdx.x < nb) {
        const int c = threadIdx.x;
        float v = red[0][c];
        for (int w = 1; w < kWarps; ++w) v += red[w][c];
        const int i = s_mpos[b0 + c];
        const int e = s_pe[i];
        s_ex[i] = selection_score(a.mode, v, a.mode == MOE_ROUTE_BIAS_SELECT ? a.bias[e] : 0.f,
                                  a.mode == MOE_ROUTE_GUMBEL ? a.u[(size_t)t * a.E + e] : 0.f,
                                  a.tau);
      }
      __syncthreads();
    }
    rank_members(a, t, 0, n, band, ws, nm, threadIdx.x, kThreads);
    __syncthreads();
  }
}

// Grid-wide barrier for the cooperative launch. Returns false when the wait ran past limit_ns
// (status bit set); the caller then leaves the rounds.
__device__ bool grid_barrier(unsigned* arrive, volatile unsigned* gen, unsigned& my_gen,
                             int* status, volatile int* fail,
                             uint64_t limit_ns = kBarrierLimitNs) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned g = my_gen;
    __threadfence();
    if (atomicAdd(arrive, 1u) == gridDim.x - 1) {
      atomicExch(arrive, 0u);
      __threadfence();
      atomicExch(const_cast<unsigned*>(gen), g + 1);
    } else {
      const uint64_t t0 = globaltimer();
      while (*gen == g) {
        if (globaltimer() - t0 > limit_ns) {
          atomicOr(status, MOE_DEVFAULT_PIPELINE_TIMEOUT);
          *fail = 1;
          break;
        }
        __nanosleep(32);
      }
    }
    __threadfence();
    my_gen = g + 1;
  }
  __syncthreads();
  return *fail == 0;
}

// Failure-detection check (moe_check_bounded_waits): the two kinds of bounded device wait, each
// against a condition that never comes true, with a short limit. CTA 0 waits on an mbarrier
// nobody arrives on (the wait of every tcgen05 pipeline, ptx::mbar_wait_bounded); CTA 1 enters
// the grid barrier of the proposal rounds, on which CTA 0 never arrives. Both must give up after
// limit_ns, record MOE_DEVFAULT_PIPELINE_TIMEOUT and return; expired[i] = 1 says wait i did.
// Nothing else is in flight, so nothing is left behind.
__global__ void __launch_bounds__(32) wait_check_kernel(uint64_t limit_ns, int* status,
                                                        int32_t* expired, unsigned* arrive,
                                                        unsigned* gen) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int flag;
  griddep_wait();
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) {
      const uint32_t b = ptx::smem_u32(&bar);
      ptx::mbar_init(b, 1);
      ptx::fence_mbarrier_init();
      flag = 0;  // the abort flag of the CTA's other roles: never raised here
      const bool ok = ptx::mbar_wait_bounded(b, 0u, &flag, status, MOE_DEVFAULT_PIPELINE_TIMEOUT,
                                             limit_ns);
      expired[0] = ok ? 0 : 1;
    }
  } else {
    if (threadIdx.x == 0) flag = 0;
    unsigned my_gen = *reinterpret_cast<volatile unsigned*>(gen);
    const bool ok = grid_barrier(arrive, gen, my_gen, status, &flag, limit_ns);
    if (threadIdx.x == 0) {
      expired[1] = ok ? 0 : 1;
      atomicExch(arrive, 0u);  // this CTA's arrival is withdrawn: the counter is clean again
    }
  }
}

__global__ void __launch_bounds__(kThreads) reroute_da_kernel(const RerouteArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int wsum[kWarps];
  __shared__ int s_cut_word, s_cut_bit;
  __shared__ int s_cut[256];
  __shared__ int s_touched[256];
  __shared__ volatile int fail;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WarpScratch wscr = warp_scratch(smem, warp, a.E);
  if (threadIdx.x == 0) fail = 0;
  unsigned my_gen = 0;
  unsigned* arrive = reinterpret_cast<unsigned*>(a.ctl);
  volatile unsigned* gen = reinterpret_cast<volatile unsigned*>(a.ctl + 1);
  const int gtid = blockIdx.x * kThreads + threadIdx.x;
  const int nthr = gridDim.x * kThreads;
  __syncthreads();
  for (int round = 0; round < kMaxRounds; ++round) {
    // A. proposals (state other CTAs update between rounds is read past L1: ld.global.cg)
    for (int e = threadIdx.x; e < a.E; e += kThreads) {
      s_cut[e] = __ldcg(&a.cut[e]);
      s_touched[e] = 0;
    }
    __syncthreads();
    for (int t = gtid; t < a.T; t += nthr) {
      const int dem = a.dem[t];
      if (dem == 0) continue;
      int held = __ldcg(&a.held[t]), p = __ldcg(&a.ptr[t]);
      const int len = a.plen[t], rl = __ldcg(&a.rlen[t]);
      const uint4* row4 = reinterpret_cast<const uint4*>(a.pref + (size_t)t * a.PS);
      uint4 chunk = make_uint4(0u, 0u, 0u, 0u);
      int chunk_at = -1;
      while (held < dem && p < len) {
        if (p >= rl) {  // next window first
          a.ext_list[atomicAdd(&a.extended[round], 1)] = t;
          break;
        }
        if ((p >> 4) != chunk_at) {  // 16 list positions per load (rows are 16-byte aligned)
          chunk_at = p >> 4;
          chunk = __ldcg(row4 + chunk_at);
        }
        const int q = (p >> 2) & 3;
        const uint32_t wd = q == 0 ? chunk.x : q == 1 ? chunk.y : q == 2 ? chunk.z : chunk.w;
        const int e = (wd >> (8 * (p & 3))) & 0xFF;
        ++p;
        if (s_cut[e] < t) continue;  // full with better tokens
        atomicOr(&a.bits[(size_t)e * a.W + (t >> 5)], 1u << (t & 31));
        s_touched[e] = 1;
        ++held;
      }
      a.ptr[t] = p;
      a.held[t] = held;
    }
    __syncthreads();  // one global flag store per expert and CTA, not one per proposal
    for (int e = threadIdx.x; e < a.E; e += kThreads)
      if (s_touched[e]) a.touched[e] = 1;
    if (!grid_barrier(arrive, gen, my_gen, a.status, &fail)) return;
    // B. every expert with new proposals keeps its `room` lowest tokens
    for (int e = blockIdx.x; e < a.E; e += gridDim.x) {
      if (!__ldcg(&a.touched[e])) continue;
      const int room = a.room[e];
      unsigned* row = a.bits + (size_t)e * a.W;
      const int per = (a.W + kThreads - 1) / kThreads;
      const int w0 = threadIdx.x * per, w1 = min(a.W, w0 + per);
      int cnt = 0;
      for (int w = w0; w < w1; ++w) cnt += __popc(__ldcg(row + w));
      int incl = cnt;  // block exclusive scan of cnt
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      if (lane == 31) wsum[warp] = incl;
      if (threadIdx.x == 0) s_cut_word = -1;
      __syncthreads();
      int before = 0, total = 0;
      for (int w = 0; w < kWarps; ++w) {
        if (w < warp) before += wsum[w];
        total += wsum[w];
      }
      const int excl = before + incl - cnt;
      // the room-th set bit (1-based) lies in this thread's words when excl < room <= excl+cnt
      if (total >= room && excl < room && room <= excl + cnt) {
        int seen = excl;
        for (int w = w0; w < w1; ++w) {
          unsigned v = __ldcg(row + w);
          const int c = __popc(v);
          if (seen + c >= room) {
            for (int need = room - seen; need > 1; --need) v &= v - 1u;
            s_cut_word = w;
            s_cut_bit = __ffs(v) - 1;
            break;
          }
          seen += c;
        }
      }
      __syncthreads();
      if (total >= room && s_cut_word >= 0) {
        const int cw = s_cut_word, bit = s_cut_bit;
        if (total > room) {
          // turn away every proposer after the room-th
          for (int w = max(w0, cw); w < w1; ++w) {
            unsigned m = __ldcg(row + w);
            if (w == cw) m &= (bit == 31) ? 0u : (0xFFFFFFFFu << (bit + 1));
            if (m == 0u) continue;
            atomicAnd(row + w, ~m);
            while (m) {
              const int b = __ffs(m) - 1;
              m &= m - 1u;
              atomicSub(&a.held[w * 32 + b], 1);
            }
          }
          if (threadIdx.x == 0) atomicAdd(&a.rejected[round], 1);
        }
        if (threadIdx.x == 0) a.cut[e] = cw * 32 + bit;
      }
      if (threadIdx.x == 0) a.touched[e] = 0;
      __syncthreads();
    }
    // ... and the listed tokens get their next window ordered exactly
    const int n_ext = __ldcg(&a.extended[round]);
    for (int i = blockIdx.x * kWarps + warp; i < n_ext; i += gridDim.x * kWarps) {
      const int t = __ldcg(&a.ext_list[i]);
      const int w0 = __ldcg(&a.rlen[t]);
      load_list(a, t, w0, a.plen[t], wscr, lane);
      const int r = refine_window(a, t, w0, a.plen[t], wscr, lane);
      if (lane == 0) a.rlen[t] = r;
    }
    if (!grid_barrier(arrive, gen, my_gen, a.status, &fail)) return;
    if (__ldcg(&a.rejected[round]) == 0 && n_ext == 0) {
      if (gtid == 0) *a.rounds_out = round + 1;
      return;
    }
  }
  if (gtid == 0) atomicOr(a.status, MOE_DEVFAULT_PIPELINE_TIMEOUT);  // rounds exhausted
}

__global__ void __launch_bounds__(kThreads) reroute_finalize_kernel(const RerouteArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();
  // the exact pass's list is empty again for the next call (the pass has completed)
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.ex_count = 0;
  for (int t = blockIdx.x * kWarps + warp; t < a.T; t += gridDim.x * kWarps) {
    if (a.dem[t] == 0) continue;
    const int len = a.ptr[t];
    // experts that kept the token, in its preference order, to its dropped slots in slot order
    int dropped = 0;
    if (lane < a.k) dropped = a.slot_pos[(size_t)t * a.k + lane] < 0;
    unsigned dmask = __ballot_sync(0xffffffffu, dropped);
    int placed = 0;
    for (int c0 = 0; c0 < len && dmask; c0 += 32) {
      const int i = c0 + lane;
      int e = -1;
      bool got = false;
      if (i < len) {
        e = a.pref[(size_t)t * a.PS + i];
        got = (a.bits[(size_t)e * a.W + (t >> 5)] >> (t & 31)) & 1u;
      }
      unsigned gm = __ballot_sync(0xffffffffu, got);
      while (gm && dmask) {
        const int src = __ffs(gm) - 1;
        gm &= gm - 1u;
        const int j = __ffs(dmask) - 1;
        dmask &= dmask - 1u;
        const int ee = __shfl_sync(0xffffffffu, e, src);
        if (lane == 0) a.topk_idx[(size_t)t * a.k + j] = ee;
        ++placed;
      }
    }
    __syncwarp();
    if (placed == 0) continue;
    // gates over the final experts: unbiased logits (PLAIN, BIAS_SELECT) or scores (GUMBEL)
    float v = -INFINITY;
    if (lane < a.k) {
      const int e = a.topk_idx[(size_t)t * a.k + lane];
      const float s = a.sfull[(size_t)t * a.E + e];
      v = a.mode == MOE_ROUTE_BIAS_SELECT ? s - a.bias[e] : s;
    }
    float mx = v;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float ev = lane < a.k ? expf(v - mx) : 0.f;
    float sum = ev;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < a.k) a.topk_w[(size_t)t * a.k + lane] = ev / sum;
  }
}

}  // namespace

cudaError_t launch_reroute(const RerouteArgs& args, cudaStream_t st) {
  RerouteArgs a = args;
  const int sms = num_sms();
  const size_t smem = (size_t)kWarps * 4 * a.E * sizeof(float);
  void (*prep)(const RerouteArgs) = a.E <= 32   ? reroute_prep_kernel<1>
                                    : a.E <= 64  ? reroute_prep_kernel<2>
                                    : a.E <= 128 ? reroute_prep_kernel<4>
                                                 : reroute_prep_kernel<8>;
  cudaError_t err =
      cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(reroute_da_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
  if (err != cudaSuccess) return err;
  const int tok_blocks = (a.T + kWarps - 1) / kWarps;
  err = launch_k(prep, dim3(tok_blocks < 8 * sms ? tok_blocks : 8 * sms), dim3(kThreads), smem,
                 st, a);
  if (err != cudaSuccess) return err;
  err = launch_k(reroute_exact_kernel, dim3(8 * sms), dim3(kThreads), 0, st, a);
  if (err != cudaSuccess) return err;
  // proposal rounds: every CTA resident (cooperative launch), one CTA per SM at most
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reroute_da_kernel, kThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int grid = sms;
  const int need = max((a.T + kThreads - 1) / kThreads, a.E);
  if (grid > need) grid = need;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, reroute_da_kernel, a);
  if (err != cudaSuccess) return err;
  return launch_k(reroute_finalize_kernel, dim3(tok_blocks < 4 * sms ? tok_blocks : 4 * sms),
                  dim3(kThreads), 0, st, a);
}

cudaError_t launch_wait_check(uint64_t limit_ns, int* status, int32_t* expired,
                              unsigned* arrive, unsigned* gen, cudaStream_t st) {
  return launch_k(wait_check_kernel, dim3(2), dim3(32), 0, st, limit_ns, status, expired, arrive,
                  gen);
}

}  // namespace moe
