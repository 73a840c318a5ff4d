// Dispatch: histogram -> capacity clamp -> exclusive scan -> stable scatter, then the grouped
// GEMM's row-tile list and the gather of x rows into expert order.
//
// Capacity rule: "参数规模与稀疏激活的真相拆解", §3.2 专家容量 (capacity = tokens*k/E*factor;
// Level 1: slots past the limit are marked overflow). Slots claim capacity in slot order
// (t ascending, then j), which inside one expert is token order. Dispatch into per-expert
// contiguous segments follows the dispatch layer of "AI架构演进从稀疏MoE到条件记忆的工程实践"
// (layered-architecture figure: gather -> expert dispatch).
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kSlotsPerThread = kPermuteBlock / kThreads;  // 4
constexpr int kMaxE = 256;

// Row-tile list of the grouped GEMMs: routed experts' segments cut into tile_m-row tiles, then
// each shared expert's identity segment over all T tokens. Thread e < E holds expert e's
// segment [o0, o0 + kept); n_kept is the sum of kept over all experts. Called by every thread of
// one CTA of kThreads threads.
__device__ void build_tiles(int o0, int kept, int n_kept, int E, int S, int T, long long TK,
                            int tile_m, TileEntry* __restrict__ tiles, Meta* meta,
                            int* warp_tot) {
  const int e = threadIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nt = (kept + tile_m - 1) / tile_m;
  int v = nt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += n;
  }
  __syncthreads();  // warp_tot may still be read by the caller's previous scan
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  int wbase = 0, total = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) wbase += warp_tot[w];
    total += warp_tot[w];
  }
  const int start = wbase + v - nt;
  for (int i = 0; i < nt; ++i) {
    TileEntry te;
    te.expert = e;
    te.row0 = o0 + i * tile_m;
    te.rows = min(tile_m, kept - i * tile_m);
    te.arow0 = te.row0;
    te.g0 = start;
    te.gn = nt;
    tiles[start + i] = te;
  }
  const int per_shared = (T + tile_m - 1) / tile_m;
  for (int i = threadIdx.x; i < S * per_shared; i += kThreads) {
    const int s = i / per_shared, m = i % per_shared;
    TileEntry te;
    te.expert = E + s;
    te.row0 = (int)(TK + (long long)s * T + (long long)m * tile_m);
    te.rows = min(tile_m, T - m * tile_m);
    te.arow0 = m * tile_m;
    te.g0 = total + s * per_shared;
    te.gn = per_shared;
    tiles[total + i] = te;
  }
  if (threadIdx.x == 0) {
    meta->n_tiles = total + S * per_shared;
    meta->n_kept = n_kept;
    meta->work[0] = 0;  // work counters of the quantized FFN passes
    meta->work[1] = 0;
  }
}

// The tile list the last dispatch CTA builds as well (tiles == nullptr: none).
struct TileJob {
  TileEntry* tiles;
  Meta* meta;
  int S, T, tile_m;
};

// Per-block expert histogram of kPermuteBlock consecutive slots. The last CTA to finish (a ticket
// counter, which it resets for the next call) then takes the per-expert running sums over the
// blocks (blk_base), the counts, the capacity clamp and the exclusive scan of kept counts
// (offsets), and, when asked, the row-tile list.
__global__ void __launch_bounds__(kThreads) hist_kernel(const int32_t* __restrict__ topk_idx,
                                                        long long TK, int E, int C,
                                                        int32_t* __restrict__ blk_hist,
                                                        int32_t* __restrict__ blk_base,
                                                        int32_t* __restrict__ counts,
                                                        int32_t* __restrict__ offsets,
                                                        int* ticket, int* status, TileJob tj) {
  constexpr int kBatchInts = 8192;  // 32 KB staging of blk_hist rows
  __shared__ int h[kMaxE];
  __shared__ int stage[kBatchInts];
  __shared__ int warp_tot[kThreads / 32];
  __shared__ int is_last;
  griddep_wait();
  for (int e = threadIdx.x; e < E; e += kThreads) h[e] = 0;
  __syncthreads();
  const long long base = (long long)blockIdx.x * kPermuteBlock;
  bool bad = false;
#pragma unroll
  for (int r = 0; r < kSlotsPerThread; ++r) {
    const long long s = base + r * kThreads + threadIdx.x;
    if (s < TK) {
      const int e = topk_idx[s];
      if (e >= 0 && e < E)
        atomicAdd(&h[e], 1);
      else
        bad = true;
    }
  }
  if (bad) atomicOr(status, MOE_DEVFAULT_BAD_EXPERT_INDEX);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads)
    blk_hist[(size_t)blockIdx.x * E + e] = h[e];
  // publish this block's row, then take a ticket; the last block sees every row
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(ticket, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const int n_blk = gridDim.x;
  const int e = threadIdx.x;
  const int rows_per_batch = kBatchInts / E;
  int run = 0;
  for (int b0 = 0; b0 < n_blk; b0 += rows_per_batch) {
    const int nb = min(rows_per_batch, n_blk - b0);
    __syncthreads();
    for (int i = threadIdx.x; i < nb * E; i += kThreads)
      stage[i] = __ldcg(blk_hist + (size_t)b0 * E + i);
    __syncthreads();
    if (e < E) {
      for (int b = 0; b < nb; ++b) {
        blk_base[(size_t)(b0 + b) * E + e] = run;
        run += stage[b * E + e];
      }
    }
  }
  int kept = 0;
  if (e < E) {
    counts[e] = run;
    kept = min(run, C);
  }
  // block-wide exclusive scan of kept over experts 0..E-1 (warp shuffles, then warp totals)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int v = kept;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  int wbase = 0, n_kept = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) wbase += warp_tot[w];
    n_kept += warp_tot[w];
  }
  const int incl = wbase + v;
  if (e < E) {
    offsets[e] = incl - kept;
    if (e == E - 1) offsets[E] = incl;
  }
  if (threadIdx.x == 0) *ticket = 0;  // every block has taken its ticket
  if (tj.tiles != nullptr)
    build_tiles(incl - kept, kept, n_kept, E, tj.S, tj.T, TK, tj.tile_m, tj.tiles, tj.meta,
                warp_tot);
}

// Stable scatter: the rank of a slot inside its expert is (slots of that expert in earlier
// blocks) + (earlier slots of this block). Ranks >= C are dropped.
__global__ void __launch_bounds__(kThreads) scatter_kernel(
    const int32_t* __restrict__ topk_idx, long long TK, int E, int C,
    const int32_t* __restrict__ blk_base, const int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm_slot, int32_t* __restrict__ slot_pos) {
  __shared__ int wcnt[kThreads / 32][kMaxE];
  __shared__ int running[kMaxE];
  __shared__ int base[kMaxE];
  __shared__ int offs[kMaxE];
  griddep_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += kThreads) {
    running[e] = 0;
    base[e] = blk_base[(size_t)blockIdx.x * E + e];
    offs[e] = offsets[e];
  }
  const unsigned lt_mask = (1u << lane) - 1u;
  const long long blk0 = (long long)blockIdx.x * kPermuteBlock;
  for (int r = 0; r < kSlotsPerThread; ++r) {
    const long long s = blk0 + r * kThreads + threadIdx.x;
    int e = -1;
    if (s < TK) {
      e = topk_idx[s];
      if (e < 0 || e >= E) e = -1;  // reported by hist_kernel; the slot is dropped
    }
    for (int i = threadIdx.x; i < (kThreads / 32) * E; i += kThreads)
      wcnt[i / E][i % E] = 0;
    __syncthreads();
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank_w = __popc(peers & lt_mask);
    if (e >= 0 && (peers & lt_mask) == 0) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (s < TK) {
      if (e >= 0) {
        int rank = base[e] + running[e] + rank_w;
        for (int w = 0; w < warp; ++w) rank += wcnt[w][e];
        if (rank < C) {
          const int pos = offs[e] + rank;
          perm_slot[pos] = (int32_t)s;
          slot_pos[s] = pos;
        } else {
          slot_pos[s] = -1;
        }
      } else {
        slot_pos[s] = -1;
      }
    }
    __syncthreads();
    for (int ee = threadIdx.x; ee < E; ee += kThreads) {
      int add = 0;
      for (int w = 0; w < kThreads / 32; ++w) add += wcnt[w][ee];
      running[ee] += add;
    }
    __syncthreads();
  }
  // positions past the last kept slot hold -1
  const int n_kept = offsets[E];
  for (int r = 0; r < kSlotsPerThread; ++r) {
    const long long p = blk0 + r * kThreads + threadIdx.x;
    if (p < TK && p >= n_kept) perm_slot[p] = -1;
  }
}

// The row-tile list from given expert offsets (the FFN entry point without a dispatch).
__global__ void __launch_bounds__(kThreads) tiles_kernel(const int32_t* __restrict__ offsets,
                                                         int E, int S, int T, long long TK,
                                                         int tile_m,
                                                         TileEntry* __restrict__ tiles,
                                                         Meta* meta) {
  __shared__ int warp_tot[kThreads / 32];
  griddep_wait();
  const int e = threadIdx.x;
  int o0 = 0, kept = 0;
  if (e < E) {
    o0 = offsets[e];
    kept = offsets[e + 1] - o0;
  }
  build_tiles(o0, kept, offsets[E], E, S, T, TK, tile_m, tiles, meta, warp_tot);
}

// xp[p, :] = x[perm_slot[p] / k, :] for p < N. One warp per row, 16-byte vectors.
__global__ void __launch_bounds__(kThreads) gather_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ perm_slot,
                                                          const int32_t* __restrict__ offsets,
                                                          int E, int k, int d, long long TK,
                                                          uint16_t* __restrict__ xp) {
  griddep_wait();
  const long long p = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (p >= TK || p >= offsets[E]) return;
  const int t = perm_slot[p] / k;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
  uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)p * d);
  const int lane = threadIdx.x & 31, n = d / 8;
  // eight 16-byte loads in flight per lane before their stores
  for (int c0 = 0; c0 < n; c0 += 8 * 32) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = c0 + i * 32 + lane;
      if (c < n) v[i] = src[c];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = c0 + i * 32 + lane;
      if (c < n) __stcs(dst + c, v[i]);
    }
  }
}

}  // namespace

cudaError_t launch_permute(const Shape& s, const int32_t* topk_idx, int32_t* counts,
                           int32_t* offsets, int32_t* perm_slot, int32_t* slot_pos,
                           int32_t* blk_hist, int32_t* blk_base, int* ticket, int* status,
                           TileEntry* tiles, Meta* meta, cudaStream_t st) {
  const TileJob tj{tiles, meta, s.S, s.T, s.tile_m};
  cudaError_t e = launch_k(hist_kernel, dim3(s.n_pblk), dim3(kThreads), 0, st, topk_idx, s.TK,
                           s.E, s.C, blk_hist, blk_base, counts, offsets, ticket, status, tj);
  if (e == cudaSuccess)
    e = launch_k(scatter_kernel, dim3(s.n_pblk), dim3(kThreads), 0, st, topk_idx, s.TK, s.E, s.C,
                 (const int32_t*)blk_base, (const int32_t*)offsets, perm_slot, slot_pos);
  return e;
}

// ---- allocation-free dispatch -----------------------------------------------------------
// Scratch of moe_permute_noalloc for callers that cannot allocate: 64 ints (256 B) hold a status
// word used when the caller passes no fault word ([0]) and the dispatch's ticket counter ([1],
// zero at load and after every dispatch), then the per-block histograms and the per-block
// running sums, each up to (MOE_NOALLOC_MAX_SLOTS / kPermuteBlock) x 256 ints.
namespace {
constexpr int kNoallocBlocks = MOE_NOALLOC_MAX_SLOTS / kPermuteBlock;
constexpr int kNoallocInts = 64 + 2 * kNoallocBlocks * kMaxE;
static_assert(MOE_NOALLOC_MAX_SLOTS % kPermuteBlock == 0, "whole dispatch blocks");
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoallocInts];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {nullptr};

// Device address of g_noalloc_scratch on the current device. In host code the array's name is
// only a host-side stand-in, so the address comes from cudaGetSymbolAddress with the device
// current. It is looked up afresh on every call made outside stream capture (a device reset, or
// another context on the device, may have loaded the module at another address) and remembered
// per device; a call made while `st` is capturing uses the address remembered from the last call
// outside capture, and looks it up only if there is none yet.
cudaError_t noalloc_scratch(cudaStream_t st, int32_t** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if ((err = cudaStreamIsCapturing(st, &cs)) != cudaSuccess) return err;
  const bool slot = dev >= 0 && dev < 64;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  void* p = slot ? g_noalloc_addr[dev] : nullptr;
  if (cs == cudaStreamCaptureStatusNone || p == nullptr) {
    if ((err = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess) return err;
    if (slot) g_noalloc_addr[dev] = p;
  }
  *out = static_cast<int32_t*>(p);
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_permute_noalloc(const Shape& s, const int32_t* topk_idx, int32_t* counts,
                                   int32_t* offsets, int32_t* perm_slot, int32_t* slot_pos,
                                   int* fault_bits, cudaStream_t st) {
  if (s.TK > MOE_NOALLOC_MAX_SLOTS || s.E > kMaxE) return cudaErrorInvalidValue;
  int32_t* scratch = nullptr;
  cudaError_t err = noalloc_scratch(st, &scratch);
  if (err != cudaSuccess) return err;
  int* status = fault_bits;
  if (status != nullptr) {
    if ((err = cudaMemsetAsync(status, 0, sizeof(int), st)) != cudaSuccess) return err;
  } else {
    status = scratch;  // nobody reads it
  }
  // every entry of both tables is written before it is read, so nothing needs clearing
  int32_t* blk_hist = scratch + 64;
  int32_t* blk_base = blk_hist + (size_t)kNoallocBlocks * kMaxE;
  return launch_permute(s, topk_idx, counts, offsets, perm_slot, slot_pos, blk_hist, blk_base,
                        scratch + 1, status, nullptr, nullptr, st);
}

cudaError_t launch_tiles(const Shape& s, const int32_t* offsets, TileEntry* tiles, Meta* meta,
                         cudaStream_t st) {
  return launch_k(tiles_kernel, dim3(1), dim3(kThreads), 0, st, offsets, s.E, s.S, s.T, s.TK,
                  s.tile_m, tiles, meta);
}

cudaError_t launch_tiles_and_gather(const Shape& s, const uint16_t* x, const int32_t* perm_slot,
                                    const int32_t* offsets, uint16_t* xp, TileEntry* tiles,
                                    Meta* meta, bool tiles_built, cudaStream_t st) {
  if (!tiles_built) {
    const cudaError_t e = launch_tiles(s, offsets, tiles, meta, st);
    if (e != cudaSuccess) return e;
  }
  const long long rows_per_blk = kThreads / 32;
  const long long grid = (s.TK + rows_per_blk - 1) / rows_per_blk;
  return launch_k(gather_kernel, dim3((unsigned)grid), dim3(kThreads), 0, st, x, perm_slot,
                  offsets, s.E, s.k, s.d, s.TK, xp);
}

}  // namespace moe
