// Grouped GEMM over variable-length expert segments on the 5th-generation tensor cores.
//
//   gate/up pass (MODE 0):  H[p, n] = silu(sum_k A[p,k] W_gate[e][k,n]) * (sum_k A[p,k] W_up[e][k,n])
//   down pass    (MODE 1):  Y[row(p), n] = gate(p) * sum_k H[p,k] W_down[e][k,n]
// On the fp16 down path (HF16, with an fp16 copy of W_down so both down operands share the
// type) H and Y are stored in fp16: 11 significant bits, but a range of +-65504, so the
// epilogues record MOE_DEVFAULT_FP16_RANGE when a value of a stored row would be clamped. On the
// bf16 down path H is bf16 and Y fp32, with fp32's range.
//
// Expert SwiGLU: "GPT-4 Has 1.8 Trillion Parameters. It Uses 2% of Them Per Token", §3.3, and
// "大模型MoE稀疏激活原理与工程实践", §3.2 (uniform d -> d_ff -> d experts). Running every
// expert's rows as one batched tensor-core matmul is the "expert fusion" of the same page's §4.2;
// the gate-scaled unpermuting epilogue replaces the separate gather/scatter/weighted-sum steps that
// "AI架构演进从稀疏MoE到条件记忆的工程实践" fuses into one kernel.
//
// Design (one CTA per SM, persistent):
//   warp 0  TMA producer: A tile [128 rows x 64 k] (K-major, 128-byte swizzle) and NCH weight
//           chunks [64 k x 64 n] (N-major, 128-byte swizzle) per stage, straight from the
//           row-major [E, K, N] weight tensors (no repack).
//   warp 1  MMA issuer: tcgen05.mma kind::f16, M=128, N=64*NCH, K=16 per instruction, fp32
//           accumulators in TMEM, two accumulator buffers so the epilogue of tile i overlaps the
//           main loop of tile i+1.
//   warp 2  TMEM allocator.
//   warps 4-7 epilogue: tcgen05.ld 32 columns at a time, fused SiLU*up (MODE 0) or gate scale and
//           scatter to slot order (MODE 1), 16-byte stores.
// Work units: (row tile of the device-written tile list) x (column tile), ordered expert by
// expert; inside an expert, in blocks of kNBlock column tiles, every row tile of the expert for
// the block's columns. CTAs running at the same time then share each weight tile (across the
// expert's row tiles) and each row tile (across the block's columns) through L2, so both are read
// from DRAM about once. The host never reads the tile
// count. Every mbarrier wait is bounded (MOE_DEVFAULT_PIPELINE_TIMEOUT on expiry).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kChunkN = 64;
constexpr int kABytes = kBM * kBK * 2;             // 16 KB
constexpr int kChunkBytes = kBK * kChunkN * 2;     // 8 KB
constexpr int kThreads = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per wait
constexpr int kNBlock = 8;                          // column tiles per expert block

template <int NCH>
struct Cfg {
  static constexpr int BN = NCH * kChunkN;                  // MMA N
  static constexpr int kStageBytes = kABytes + NCH * kChunkBytes;
  static constexpr int kStages = (200 * 1024 / kStageBytes) > 8 ? 8 : (200 * 1024 / kStageBytes);
  static constexpr int kTmemCols = 2 * BN;                  // two accumulators
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
};

struct GemmArgs {
  const TileEntry* tiles;
  const Meta* meta;
  int n_ntiles;       // column tiles
  int k_blocks;       // K / 64
  int E;              // routed experts; tile.expert >= E is shared expert (expert - E)
  void* out;          // H (MODE 0) or Y (MODE 1: fp16 on the fp16 down path, else fp32)
  long long out_ld;   // elements per output row
  const int32_t* perm_slot;  // MODE 1
  const float* topk_w;       // MODE 1 (NULL: gate 1)
  int* status;
};

// Work unit w -> (row tile, column tile) in the expert-major blocked order described above.
__device__ __forceinline__ void map_unit(long long w, int n_nt, const TileEntry* tiles,
                                         TileEntry& te, int& nt) {
  const TileEntry first = tiles[w / n_nt];  // some row tile of the unit's expert
  const long long u = w - (long long)n_nt * first.g0;
  const long long blk = (long long)first.gn * kNBlock;
  const int nb = (int)(u / blk);
  const int nbs = min(kNBlock, n_nt - nb * kNBlock);
  const int rr = (int)(u - (long long)nb * blk);
  te = tiles[first.g0 + rr / nbs];
  nt = nb * kNBlock + rr % nbs;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// fp16x2, round to nearest even, saturating to +-65504 (no infinities from large activations)
__device__ __forceinline__ uint32_t pack_f16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Magnitude bits of a float with the sign cleared: they order as |v| does, and NaN orders above
// infinity. A value whose bits reach kF16Clamp (65520.0f) would round past the largest finite
// fp16 (65504), so the saturating conversion clamps it (or it is not finite at all).
__device__ __forceinline__ uint32_t mag_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }
constexpr uint32_t kF16Clamp = 0x477FF000u;

// The epilogue of one work unit for one accumulator row (one thread): the unit's BN accumulator
// columns from TMEM at taddr, written to row `orow` of the output from column nt * (BN / 2)
// (MODE 0) or nt * BN (MODE 1).
//   MODE 0: H = silu(G) * U, G the first BN/2 columns and U the rest; fp16 (HF16) or bf16.
//   MODE 1: Y = gate * acc; fp16 (HF16) or fp32 (the bf16 down path: no range limit).
// Returns the largest magnitude bits (mag_bits) among values converted to fp16 by a valid row
// (0 when nothing went to fp16), so the caller can report a clamp.
template <int MODE, int BN, bool HF16>
__device__ __forceinline__ uint32_t epilogue_row(uint32_t taddr, void* out, long long out_ld,
                                                 long long orow, int nt, float gate,
                                                 bool valid) {
  uint32_t mx = 0u;
  if (MODE == 0) {
    uint16_t* dst = static_cast<uint16_t*>(out) + orow * out_ld + (long long)nt * (BN / 2);
#pragma unroll 1
    for (int c = 0; c < BN / 2 / 32; ++c) {
      uint32_t g[32], u[32];
      ptx::tmem_ld_32x32b_x32(taddr + c * 32, g);
      ptx::tmem_ld_32x32b_x32(taddr + BN / 2 + c * 32, u);
      ptx::tmem_wait_ld();
      uint32_t hv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
        const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
        const float h0 = g0 / (1.0f + __expf(-g0)) * u0;
        const float h1 = g1 / (1.0f + __expf(-g1)) * u1;
        if (HF16) mx = max(mx, max(mag_bits(h0), mag_bits(h1)));
        hv[i] = HF16 ? pack_f16x2_sat(h0, h1) : pack_bf16x2(h0, h1);
      }
      if (valid) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          d4[i] = make_uint4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
      }
    }
  } else if (HF16) {
    uint16_t* dst = static_cast<uint16_t*>(out) + orow * out_ld + (long long)nt * BN;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t v[32];
      ptx::tmem_ld_32x32b_x32(taddr + c * 32, v);
      ptx::tmem_wait_ld();
      uint32_t yv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float y0 = gate * __uint_as_float(v[2 * i]);
        const float y1 = gate * __uint_as_float(v[2 * i + 1]);
        mx = max(mx, max(mag_bits(y0), mag_bits(y1)));
        yv[i] = pack_f16x2_sat(y0, y1);
      }
      if (valid) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          d4[i] = make_uint4(yv[4 * i], yv[4 * i + 1], yv[4 * i + 2], yv[4 * i + 3]);
      }
    }
  } else {
    float* dst = static_cast<float*>(out) + orow * out_ld + (long long)nt * BN;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t v[32];
      ptx::tmem_ld_32x32b_x32(taddr + c * 32, v);
      ptx::tmem_wait_ld();
      if (valid) {
        float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          d4[i] = make_float4(gate * __uint_as_float(v[4 * i]), gate * __uint_as_float(v[4 * i + 1]),
                              gate * __uint_as_float(v[4 * i + 2]),
                              gate * __uint_as_float(v[4 * i + 3]));
      }
    }
  }
  return valid ? mx : 0u;
}

// After an epilogue warp's last unit: one vote, and one atomic per warp that clamped a value.
__device__ __forceinline__ void report_f16_clamp(uint32_t mx, int lane, int* status) {
  if (__any_sync(0xffffffffu, mx >= kF16Clamp) && lane == 0)
    atomicOr(status, MOE_DEVFAULT_FP16_RANGE);
}

template <int MODE, int NCH, bool HF16>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA_routed,
                        const __grid_constant__ CUtensorMap tmA_shared,
                        const __grid_constant__ CUtensorMap tmB0_routed,
                        const __grid_constant__ CUtensorMap tmB1_routed,
                        const __grid_constant__ CUtensorMap tmB0_shared,
                        const __grid_constant__ CUtensorMap tmB1_shared, const GemmArgs a) {
  using C = Cfg<NCH>;
  constexpr int BN = C::BN;
  constexpr int STAGES = C::kStages;
  // gate/up multiplies bf16 x bf16; down multiplies H x W_down in fp16 (HF16) or bf16
  constexpr uint32_t IDESC =
      ptx::idesc_f16kind_f32(kBM, BN, 0, 1, (MODE == 1 && HF16) ? 0u : 1u);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + STAGES * C::kStageBytes;
  // barrier addresses
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t mma_done_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + STAGES * C::kStageBytes +
                                                    8 * (2 * STAGES + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull_bar(b), 1);
      ptx::mbar_init(tempty_bar(b), 4);
    }
    ptx::mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbarrier_init();
    ptx::prefetch_tmap(&tmA_routed);
    ptx::prefetch_tmap(&tmB0_routed);
    if (MODE == 0) ptx::prefetch_tmap(&tmB1_routed);
  }
  if (warp == 2) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();  // everything above touched only shared memory, TMEM and parameters

  const int n_mt = a.meta->n_tiles;
  const long long total = (long long)n_mt * a.n_ntiles;

  if (warp == 0) {
    if (lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, last_parity = 0;  // per stage: issued at least once / its parity
    bool ok = true;
    for (long long w = blockIdx.x; w < total && ok; w += gridDim.x) {
      TileEntry te;
      int nt;
      map_unit(w, a.n_ntiles, a.tiles, te, nt);
      const bool shared = te.expert >= a.E;
      const int ex = shared ? te.expert - a.E : te.expert;
      const CUtensorMap* tA = shared ? &tmA_shared : &tmA_routed;
      const CUtensorMap* tB0 = shared ? &tmB0_shared : &tmB0_routed;
      const CUtensorMap* tB1 = shared ? &tmB1_shared : &tmB1_routed;
      const int arow = (MODE == 0) ? te.arow0 : te.row0;
      for (int kb = 0; kb < a.k_blocks; ++kb) {
        if (!ptx::mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, a.status,
                                    MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const uint32_t sA = base + stage * C::kStageBytes;
        const uint32_t sB = sA + kABytes;
        const uint32_t fb = full_bar(stage);
        ptx::mbar_arrive_expect_tx(fb, C::kStageBytes);
        ptx::tma_load_2d(sA, tA, fb, kb * kBK, arow);
        // one copy per weight matrix: its 64-column chunks are the map's third dimension
        if (MODE == 0) {
          // chunks [0, NCH/2): gate columns; [NCH/2, NCH): up columns of the same n range
          ptx::tma_load_4d(sB, tB0, fb, 0, kb * kBK, nt * (NCH / 2), ex);
          ptx::tma_load_4d(sB + (NCH / 2) * kChunkBytes, tB1, fb, 0, kb * kBK, nt * (NCH / 2),
                           ex);
        } else {
          ptx::tma_load_4d(sB, tB0, fb, 0, kb * kBK, nt * NCH, ex);
        }
        issued_mask |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // never leave while a copy into this CTA's shared memory may still be in flight
    for (int s = 0; s < STAGES; ++s)
      if (issued_mask & (1u << s)) {
        volatile int no_abort = 0;
        ptx::mbar_wait_bounded(full_bar(s), (last_parity >> s) & 1u, &no_abort, a.status,
                               MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs / 4);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (long long w = blockIdx.x; w < total && ok; w += gridDim.x) {
      if (!ptx::mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, a.status,
                                  MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs))
        break;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
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
          // A: K-major, 128 B rows, 8-row groups 1024 B apart; K step of 16 = +32 B in the row.
          const uint64_t adesc = ptx::smem_desc_sw128(sA + kk * 32, 16, 1024);
          // B: N-major, 64-column chunks 8 KB apart (LBO), 8-row k groups 1024 B apart (SBO);
          // K step of 16 rows = +2048 B.
          const uint64_t bdesc = ptx::smem_desc_sw128(sB + kk * 2048, kChunkBytes, 1024);
          ptx::umma_f16(d_tmem, adesc, bdesc, IDESC, (kb | kk) != 0 ? 1u : 0u);
        }
        ptx::umma_commit(empty_bar(stage));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      ptx::umma_commit(tfull_bar(acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // all MMAs issued by this thread have finished before TMEM is released
    ptx::umma_commit(mma_done_bar);
    volatile int no_abort = 0;
    ptx::mbar_wait_bounded(mma_done_bar, 0, &no_abort, a.status, MOE_DEVFAULT_PIPELINE_TIMEOUT,
                           kWaitLimitNs / 4);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp - 4;  // TMEM lanes [32q, 32q + 32)
    const int row_in_tile = 32 * q + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t clamp = 0u;  // largest magnitude this thread converted to fp16 (mag_bits)
    for (long long w = blockIdx.x; w < total; w += gridDim.x) {
      TileEntry te;
      int nt;
      map_unit(w, a.n_ntiles, a.tiles, te, nt);
      const bool valid = row_in_tile < te.rows;
      const long long p = (long long)te.row0 + row_in_tile;
      // MODE 1: the row's slot and gate are loaded before waiting for the accumulator
      long long orow = p;
      float gate = 1.0f;
      if (MODE == 1 && valid && te.expert < a.E) {
        const int slot = a.perm_slot[p];
        orow = slot;
        if (a.topk_w != nullptr) gate = a.topk_w[slot];
      }
      if (!ptx::mbar_wait_bounded_warp(tfull_bar(acc), acc_phase, abort_flag, a.status,
                                       MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs))
        break;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);
      clamp = max(clamp, epilogue_row<MODE, BN, HF16>(taddr, a.out, a.out_ld,
                                                       MODE == 0 ? p : orow, nt, gate, valid));
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(tempty_bar(acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    report_f16_clamp(clamp, lane, a.status);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------------------ CTA pairs
// The same grouped GEMM on pairs of CTAs (a cluster of two) sharing one tcgen05 MMA of M = 256:
// a work unit is a 256-row tile of one expert x a 256-column tile; CTA rank r stages rows
// [128 r, 128 r + 128) of A and half of the weight columns (gate/up: rank 0 the gate chunks,
// rank 1 the up chunks; down: chunks 2 r, 2 r + 1), so each CTA's stage is 32 KB instead of 48
// and seven stages fit. Rank 0's thread issues the MMAs (reading both CTAs' shared memory) and
// commits to both CTAs' barriers; each CTA's epilogue reads its own 128 TMEM lanes (all 256
// columns) exactly as in the single-CTA kernel, and both release the accumulator on rank 0.
struct Cfg2 {
  static constexpr int BN = 256;            // MMA N over the pair
  static constexpr int kHalfChunks = 2;     // 64-column weight chunks staged per CTA
  static constexpr int kStageBytes = kABytes + kHalfChunks * kChunkBytes;  // 32 KB
  static constexpr int kStages = 7;  // 224 KB: the most that fits beside the barriers
  static constexpr int kTmemCols = 2 * BN;  // two accumulators
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
};

template <int MODE, bool HF16>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm2_kernel(const __grid_constant__ CUtensorMap tmA_routed,
                         const __grid_constant__ CUtensorMap tmA_shared,
                         const __grid_constant__ CUtensorMap tmB0_routed,
                         const __grid_constant__ CUtensorMap tmB1_routed,
                         const __grid_constant__ CUtensorMap tmB0_shared,
                         const __grid_constant__ CUtensorMap tmB1_shared, const GemmArgs a) {
  using C = Cfg2;
  constexpr int BN = C::BN;
  constexpr int STAGES = C::kStages;
  constexpr uint32_t IDESC =
      ptx::idesc_f16kind_f32(2 * kBM, BN, 0, 1, (MODE == 1 && HF16) ? 0u : 1u);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + STAGES * C::kStageBytes;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t mma_done_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + STAGES * C::kStageBytes +
                                                    8 * (2 * STAGES + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_rank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);   // rank 0's: one arrival + both CTAs' bytes
      ptx::mbar_init(empty_bar(s), 1);  // one commit from rank 0's MMA thread
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull_bar(b), 1);
      ptx::mbar_init(tempty_bar(b), 8);  // rank 0's: four epilogue warps of each CTA
    }
    ptx::mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbarrier_init();
    ptx::prefetch_tmap(&tmA_routed);
    ptx::prefetch_tmap(&tmB0_routed);
    if (MODE == 0) ptx::prefetch_tmap(&tmB1_routed);
  }
  if (warp == 2) {
    ptx::tmem_alloc_cg2(ptx::smem_u32(tmem_slot), C::kTmemCols);
    ptx::tmem_relinquish_cg2();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  ptx::cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA arrival
  griddep_wait();       // everything above touched only shared memory, TMEM and parameters

  const int n_mt = a.meta->n_tiles;
  const long long total = (long long)n_mt * a.n_ntiles;
  const long long pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer (both)
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (long long w = pair; w < total && ok; w += n_pairs) {
        TileEntry te;
        int nt;
        map_unit(w, a.n_ntiles, a.tiles, te, nt);
        const bool shared = te.expert >= a.E;
        const int ex = shared ? te.expert - a.E : te.expert;
        const CUtensorMap* tA = shared ? &tmA_shared : &tmA_routed;
        const CUtensorMap* tB =
            MODE == 0 ? (rank == 0 ? (shared ? &tmB0_shared : &tmB0_routed)
                                   : (shared ? &tmB1_shared : &tmB1_routed))
                      : (shared ? &tmB0_shared : &tmB0_routed);
        const int arow = ((MODE == 0) ? te.arow0 : te.row0) + kBM * (int)rank;
        const int chunk0 = MODE == 0 ? nt * C::kHalfChunks : nt * 2 * C::kHalfChunks +
                                                                 C::kHalfChunks * (int)rank;
        for (int kb = 0; kb < a.k_blocks; ++kb) {
          if (!ptx::mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, a.status,
                                      MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t sA = base + stage * C::kStageBytes;
          const uint32_t sB = sA + kABytes;
          // completion is counted on rank 0's full barrier, which expects both CTAs' bytes
          const uint32_t fb = leader ? full_bar(stage) : ptx::mapa_shared(full_bar(stage), 0);
          if (leader) ptx::mbar_arrive_expect_tx(fb, 2 * C::kStageBytes);
          ptx::tma_load_2d_cg2(sA, tA, fb, kb * kBK, arow);
          ptx::tma_load_4d_cg2(sB, tB, fb, 0, kb * kBK, chunk0, ex);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------------- MMA issuer (rank 0)
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (long long w = pair; w < total && ok; w += n_pairs) {
        if (!ptx::mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, a.status,
                                    MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs))
          break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
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
            ptx::umma_f16_cg2(d_tmem, adesc, bdesc, IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::umma_commit_cg2(empty_bar(stage), 0x3);  // frees the stage in both CTAs
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::umma_commit_cg2(tfull_bar(acc), 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // all MMAs issued by this thread have finished before TMEM is released
      ptx::umma_commit_cg2(mma_done_bar, 0x1);
      volatile int no_abort = 0;
      ptx::mbar_wait_bounded(mma_done_bar, 0, &no_abort, a.status,
                             MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs / 4);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue (both)
    const int q = warp - 4;  // TMEM lanes [32q, 32q + 32) of this CTA
    const int row_in_tile = kBM * (int)rank + 32 * q + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t clamp = 0u;  // largest magnitude this thread converted to fp16 (mag_bits)
    for (long long w = pair; w < total; w += n_pairs) {
      TileEntry te;
      int nt;
      map_unit(w, a.n_ntiles, a.tiles, te, nt);
      const bool valid = row_in_tile < te.rows;
      const long long p = (long long)te.row0 + row_in_tile;
      long long orow = p;
      float gate = 1.0f;
      if (MODE == 1 && valid && te.expert < a.E) {
        const int slot = a.perm_slot[p];
        orow = slot;
        if (a.topk_w != nullptr) gate = a.topk_w[slot];
      }
      if (!ptx::mbar_wait_bounded_warp(tfull_bar(acc), acc_phase, abort_flag, a.status,
                                       MOE_DEVFAULT_PIPELINE_TIMEOUT, kWaitLimitNs))
        break;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);
      clamp = max(clamp, epilogue_row<MODE, BN, HF16>(taddr, a.out, a.out_ld,
                                                       MODE == 0 ? p : orow, nt, gate, valid));
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          ptx::mbar_arrive(tempty_bar(acc));
        else
          ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar(acc), 0));
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    report_f16_clamp(clamp, lane, a.status);
  }

  // every copy into either CTA has landed and every MMA has finished once rank 0's MMA thread
  // passed its final wait; neither CTA leaves (nor frees TMEM) before both get here
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_cg2(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_impl() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

bool make_map_a(CUtensorMap* m, const void* ptr, long long rows, long long K,
                CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  return make_tmap_2d(m, ptr, rows, K, kBK, kBM, dt);
}

// Weights [n_exp, K, N] seen as [n_exp][N/64 chunks][K][64]: dims (64 columns, K, chunk,
// expert), box (64, 64, chunks per copy, 1), so one copy lands `chunks` 8 KB chunks back to back.
bool make_map_b(CUtensorMap* m, const void* ptr, long long n_exp, long long K, long long N,
                int chunks, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn_impl();
  if (fn == nullptr || N % kChunkN != 0) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)kChunkN, (cuuint64_t)K, (cuuint64_t)(N / kChunkN),
                              (cuuint64_t)n_exp};
  const cuuint64_t strides[3] = {(cuuint64_t)N * 2, (cuuint64_t)kChunkN * 2,
                                 (cuuint64_t)K * N * 2};
  const cuuint32_t box[4] = {(cuuint32_t)kChunkN, (cuuint32_t)kBK, (cuuint32_t)chunks, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, dt, 4, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int NCH, bool HF16>
cudaError_t launch_one(const CUtensorMap (&maps)[6], const GemmArgs& args, cudaStream_t st) {
  using C = Cfg<NCH>;
  auto kern = grouped_gemm_kernel<MODE, NCH, HF16>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  return launch_k(kern, dim3(num_sms()), dim3(kThreads), C::kSmemBytes, st, maps[0], maps[1],
                  maps[2], maps[3], maps[4], maps[5], args);
}

template <int MODE, bool HF16>
cudaError_t launch_two(const CUtensorMap (&maps)[6], const GemmArgs& args, cudaStream_t st) {
  using C = Cfg2;
  auto kern = grouped_gemm2_kernel<MODE, HF16>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms() / 2 * 2);  // persistent: one CTA pair per two SMs
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5],
                            args);
}

template <bool HF16>
cudaError_t launch_pair(const Shape& s, const FfnPtrs& p, cudaStream_t st, cudaEvent_t ev_mid) {
  const long long rows = s.rows;
  const bool has_shared = s.S > 0;
  constexpr CUtensorMapDataType kHType =
      HF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint16_t* Wd = HF16 ? p.W_down_f16 : p.W_down;
  const uint16_t* Wsd = HF16 ? p.Wsh_down_f16 : p.Wsh_down;
  // ---- gate/up: A = gathered rows (routed) or x (shared); B = W_gate / W_up
  CUtensorMap m0[6];
  const int gu_chunks = s.f % 128 == 0 ? 2 : 1;  // chunks per matrix and copy (NCH / 2)
  bool ok = make_map_a(&m0[0], p.xp, s.TK, s.d) && make_map_a(&m0[1], p.x, s.T, s.d) &&
            make_map_b(&m0[2], p.W_gate, s.E, s.d, s.f, gu_chunks) &&
            make_map_b(&m0[3], p.W_up, s.E, s.d, s.f, gu_chunks);
  if (has_shared)
    ok = ok && make_map_b(&m0[4], p.Wsh_gate, s.S, s.d, s.f, gu_chunks) &&
         make_map_b(&m0[5], p.Wsh_up, s.S, s.d, s.f, gu_chunks);
  else {
    m0[4] = m0[2];
    m0[5] = m0[3];
  }
  if (!ok) return cudaErrorInvalidValue;
  GemmArgs g{};
  g.tiles = p.tiles;
  g.meta = p.meta;
  g.E = s.E;
  g.status = p.status;
  g.k_blocks = s.d / kBK;
  g.out = p.h;
  g.out_ld = s.f;
  const bool pairs = s.tile_m == 2 * kBM;  // 256-row tiles: the CTA-pair kernels
  cudaError_t err;
  if (pairs) {
    g.n_ntiles = s.f / 128;
    err = launch_two<0, HF16>(m0, g, st);
  } else if (s.f % 128 == 0) {
    g.n_ntiles = s.f / 128;
    err = launch_one<0, 4, HF16>(m0, g, st);
  } else {
    g.n_ntiles = s.f / 64;
    err = launch_one<0, 2, HF16>(m0, g, st);
  }
  if (err != cudaSuccess) return err;
  if (ev_mid != nullptr && (err = cudaEventRecord(ev_mid, st)) != cudaSuccess) return err;

  // ---- down: A = H rows; B = W_down; epilogue scales by the gate and writes slot order (fp32)
  CUtensorMap m1[6];
  // chunks per copy: a CTA of a pair stages half of the down pass's four
  const int dn_chunks = pairs ? 2 : (s.d % 256 == 0 ? 4 : (s.d % 128 == 0 ? 2 : 1));
  ok = make_map_a(&m1[0], p.h, rows, s.f, kHType) &&
       make_map_b(&m1[2], Wd, s.E, s.f, s.d, dn_chunks, kHType);
  if (has_shared)
    ok = ok && make_map_b(&m1[4], Wsd, s.S, s.f, s.d, dn_chunks, kHType);
  else
    m1[4] = m1[2];
  if (!ok) return cudaErrorInvalidValue;
  m1[1] = m1[0];
  m1[3] = m1[2];
  m1[5] = m1[4];
  GemmArgs g1 = g;
  g1.k_blocks = s.f / kBK;
  g1.out = p.y;
  g1.out_ld = s.d;
  g1.perm_slot = p.perm_slot;
  g1.topk_w = p.topk_w;
  if (pairs) {
    g1.n_ntiles = s.d / 256;
    return launch_two<1, HF16>(m1, g1, st);
  } else if (s.d % 256 == 0) {
    g1.n_ntiles = s.d / 256;
    return launch_one<1, 4, HF16>(m1, g1, st);
  } else if (s.d % 128 == 0) {
    g1.n_ntiles = s.d / 128;
    return launch_one<1, 2, HF16>(m1, g1, st);
  }
  g1.n_ntiles = s.d / 64;
  return launch_one<1, 1, HF16>(m1, g1, st);
}

}  // namespace

bool make_tmap_2d(CUtensorMap* m, const void* ptr, long long rows, long long cols, int box_cols,
                  int box_rows, CUtensorMapDataType dt) {
  auto fn = encode_fn_impl();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_3d(CUtensorMap* m, const void* ptr, long long n, long long rows, long long cols,
                  int box_cols, int box_rows, CUtensorMapDataType dt) {
  auto fn = encode_fn_impl();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)n};
  const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)rows * cols * 2};
  const cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_grouped_ffn(const Shape& s, const FfnPtrs& p, cudaStream_t st,
                               cudaEvent_t ev_mid) {
  if (encode_fn_impl() == nullptr) return cudaErrorNotSupported;
  if (p.W_down_f16 != nullptr) return launch_pair<true>(s, p, st, ev_mid);
  return launch_pair<false>(s, p, st, ev_mid);
}

}  // namespace moe
