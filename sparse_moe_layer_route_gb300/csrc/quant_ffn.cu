// Weight-only group-wise quantized experts ("大模型MoE稀疏激活原理与工程实践", §4.2 量化与混合精度:
// expert weights to INT4 with one scale and zero-point per 128 weights, the router kept in
// higher precision).
//
// quantize_kernel     one thread per (matrix, group of 128 input rows, output column): min/max,
//                     fp16 scale, zero-point and codes, all in float64; codes are written in the
//                     fragment order of include/moe.h (moe_qmatrix).
// act_prep_kernel     x16 = fp16(x) once per token, with each 128-column group's sum; the
//                     gate/up pass reads its rows by token (no gathered copy).
// qffn_kernel<B, M>   the expert FFN on the codes, one warp per (8-row tile, 16 or 32 output
//                     columns): M = 0 gate/up with the SwiGLU epilogue into H (fp16), M = 1 down
//                     with the gate scale into the slot-ordered fp16 rows Y (the same buffers and
//                     layouts as the bf16 grouped GEMM, so dispatch and combine are shared).
//
// Why this shape. At decode sizes an expert sees one or two rows, so the layer is bound by the
// bytes of the weights it touches; the kernel streams each code once with 16-byte coalesced
// loads (a warp reads 512 contiguous bytes per load) and the arithmetic per code has to stay
// below the memory time. A code becomes an exact fp16 integer in one instruction: a byte, or a
// nibble, placed into the mantissa of 1024.0 gives 1024 + q (a nibble that sits 4 bits up gives
// 1024 + 16 q, and the rows stored that way take a scale 16 times smaller). These feed mma.sync
// m16n8k16 as the A operand straight from registers (weights as the M side, up to 8 tokens as
// N); every product is exact and the sums are fp32. Per 128-row group the constant is removed
// once, (1024 + z) * sum(b), and the group's fp32 scale applied; sum(b) comes precomputed with
// x16 (gate/up), or in the down pass from one more MMA against an all-ones fragment (8-bit) or
// fp32 adds of the lane's own H values (4-bit). The result is the dequantized weights'
// (q - z) * s dot product up to the fp32 rounding of the offset (about 1e-4 of it, far below the
// fp16 rows' rounding). x16 and H are stored in fragment order (frag_pos), so a lane reads its B
// operands of a group in four 16-byte loads. The
// zero-point subtraction thus leaves the per-code path, which at 4 bits was the limit (the
// kernel issue-bound below the memory rate). tcgen05 measured slower for this shape: with A in
// shared memory the dequantized tile costs 2 more bytes written and read per weight, more
// shared-memory traffic than the SM has at the HBM rate of 1-byte codes; with A in TMEM (codes
// dequantized in registers, tcgen05.st, an M = 128 N = 16 MMA per 16-deep step) the stores ran at
// about 48 B per clock per SM and each N = 16 MMA took 60-90 cycles to issue, so the 4-bit decode
// layer took 0.97 ms against this kernel's 0.52 ms. Register operands skip both.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "internal.h"

namespace moe {
namespace {

constexpr int kGroup = 128;
constexpr int kQThreads = 128;  // 4 warps per CTA, each taking work units on its own

// ------------------------------------------------------------------------------ quantization
template <int BITS>
__global__ void __launch_bounds__(256) quantize_kernel(const uint16_t* __restrict__ W,
                                                       uint8_t* __restrict__ q,
                                                       uint16_t* __restrict__ scale,
                                                       uint8_t* __restrict__ zero, int n_mat,
                                                       int K, int N) {
  const long long groups = (long long)n_mat * (K / kGroup);
  const long long total = groups * N;
  const double top = (double)((1 << BITS) - 1);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int n = (int)(i % N);
    const long long mg = i / N;  // matrix * K/128 + group
    const int m = (int)(mg / (K / kGroup));
    const int grp = (int)(mg % (K / kGroup));
    const uint16_t* col = W + ((size_t)m * K + (size_t)grp * kGroup) * N + n;
    double lo = INFINITY, hi = -INFINITY;
    for (int r = 0; r < kGroup; ++r) {
      const double w = (double)__uint_as_float((uint32_t)col[(size_t)r * N] << 16);
      lo = fmin(lo, w);
      hi = fmax(hi, w);
    }
    __half sh = __double2half((hi - lo) / top);
    double s = (double)__half2float(sh);
    if (!(s > 0.0) || isinf(s)) {  // no range (or under/overflow): fp16(max |w|), else 1
      sh = __double2half(fmax(fabs(lo), fabs(hi)));
      s = (double)__half2float(sh);
      if (!(s > 0.0) || isinf(s)) {
        sh = __float2half(1.0f);
        s = 1.0;
      }
    }
    const double z = fmin(fmax(rint(-lo / s), 0.0), top);
    scale[mg * N + n] = __half_as_ushort(sh);
    zero[mg * N + n] = (uint8_t)z;
    // fragment-order position of (n, k): tile nt, lane, slot j in the step (see moe_qmatrix)
    const int nt = n / 16, rr = n % 16;
    for (int r = 0; r < kGroup; ++r) {
      const double w = (double)__uint_as_float((uint32_t)col[(size_t)r * N] << 16);
      const int code = (int)fmin(fmax(rint(w / s) + z, 0.0), top);
      const int k = grp * kGroup + r;
      const int st = k / 16, kk = k % 16;
      const int lane = (rr % 8) * 4 + (kk % 8) / 2;
      const int j = (kk % 2) + 2 * (rr / 8) + 4 * (kk / 8);
      const size_t tile = (size_t)m * (N / 16) + nt;
      if (BITS == 8) {
        const size_t off = (tile * (K / 32) + st / 2) * 512 + lane * 16 + (st % 2) * 8 + j;
        q[off] = (uint8_t)code;
      } else {
        const size_t off = (tile * (K / 64) + st / 4) * 512 + lane * 16 + (st % 4) * 4;
        atomicOr(reinterpret_cast<unsigned int*>(q + off),
                 (unsigned int)code << (16 * (j % 2) + 4 * (j / 2)));
      }
    }
  }
}

// ------------------------------------------------------------------------------ FFN
// bf16 pair -> fp16 pair (activations of the gate/up pass)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const __half2 h = __floats2half2_rn(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}

struct QMat {
  const uint8_t* q;
  const uint16_t* s;
  const uint8_t* z;
};

struct QArgs {
  QMat routed[2], shared[2];  // M = 0: gate, up; M = 1: down (index 0)
  const uint16_t* src;        // M = 0: x16 [T, K] fp16, read by token; M = 1: H [rows, K] fp16
  const float* bsum;          // M = 0: sbx [T, K / 128], the group sums of x16
  uint16_t* out;              // M = 0: H [rows, N] fp16; M = 1: Y [rows, N] fp16
  const TileEntry* tiles;     // 8-row tiles of every expert's rows (device-written)
  Meta* meta;                 // tile count and the work counters
  const int32_t* perm_slot;   // slot of each expert-ordered row
  const float* topk_w;        // M = 1 (NULL: gate 1)
  float* tail_acc;            // partial accumulators of split tail units (see qffn_kernel)
  int* tail_ticket;           // pieces finished per split tail unit (zero between launches)
  int tail_cap;               // pieces tail_acc holds
  int* status;                // MOE_DEVFAULT_FP16_RANGE when an fp16 output value is clamped
  int E, K, N, top_k;
};

// The activations the passes read as MMA B operands (x16, H) are kept in fragment order inside
// every 128-column group: column 16 s + j of the group (step s, j < 16) sits at
//   32 p + 4 s + 2 w + e,   p = (j % 8) / 2, w = j / 8, e = j % 2,
// so the 32 values lane c of a token's quad needs for the group's eight steps (k = 16 s + 2c,
// 2c + 1, 2c + 8, 2c + 9) are 64 contiguous bytes, four 16-byte loads.
__host__ __device__ constexpr int frag_pos(int col) {
  return (col & ~127) + ((col & 7) >> 1) * 32 + ((col & 127) >> 4) * 4 + ((col >> 3) & 1) * 2 +
         (col & 1);
}

// x16[t, :] = fp16(x[t, :]) (round to nearest, as the MMA operand takes it) and
// sbx[t, g] = the fp32 sum of x16[t, 128 g : 128 g + 128]: each lane adds its 8 values in column
// order, then 16 lanes combine by a fixed tree. One warp per (token, 256 columns): two groups.
__global__ void __launch_bounds__(256) act_prep_kernel(const uint16_t* __restrict__ x, int T,
                                                       int K, uint16_t* __restrict__ x16,
                                                       float* __restrict__ sbx,
                                                       int* __restrict__ tickets, int n_tickets) {
  griddep_wait();
  // the FFN passes' tail tickets start at zero (each pass leaves them zero, but a fresh
  // workspace holds anything)
  for (int i = blockIdx.x * 256 + threadIdx.x; i < n_tickets; i += gridDim.x * 256) tickets[i] = 0;
  const int lane = threadIdx.x & 31;
  const int chunks = K / 8, groups = K / kGroup;
  const int passes = (chunks + 31) / 32;
  const long long items = (long long)T * passes;
  for (long long w = blockIdx.x * 8LL + (threadIdx.x >> 5); w < items; w += gridDim.x * 8LL) {
    const long long t = w / passes;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * K);
    uint4* dst = reinterpret_cast<uint4*>(x16 + t * K);
    const int c = (int)(w % passes) * 32 + lane;  // lanes 0-15: one group, 16-31: the next
    float sum = 0.f;
    if (c < chunks) {
      const uint4 v = src[c];
      const uint4 h = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y),
                                 bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
      const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
      // pair p of the chunk (columns 8 c + 2p, + 1) to its fragment-order place
      uint32_t* drow = reinterpret_cast<uint32_t*>(dst);
#pragma unroll
      for (int p = 0; p < 4; ++p) drow[frag_pos(8 * c + 2 * p) / 2] = hw[p];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[i]));
        sum += f.x;
        sum += f.y;
      }
    }
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if ((lane & 15) == 0 && c < chunks) sbx[t * groups + c / 16] = sum;
  }
}

// A fragment of one 16x16 step from its 8 codes, as fp16 integers 1024 + q.
// 8-bit: lo = codes j0..j3, hi = codes j4..j7 (one byte each).
__device__ __forceinline__ void a_frag8(uint32_t lo, uint32_t hi, uint32_t (&a)[4]) {
  a[0] = __byte_perm(lo, 0x64646464u, 0x4140);  // (j0, j1) row g
  a[1] = __byte_perm(lo, 0x64646464u, 0x4342);  // (j2, j3) row g + 8
  a[2] = __byte_perm(hi, 0x64646464u, 0x4140);  // (j4, j5) row g
  a[3] = __byte_perm(hi, 0x64646464u, 0x4342);  // (j6, j7) row g + 8
}

// 4-bit: one word; slot j at bit 16 * (j % 2) + 4 * (j / 2). Rows g + 8 (slots 2, 3, 6, 7) sit
// at bits 4-7 of their byte and stay there: 1024 + 16 q, undone by their scale (1/16).
__device__ __forceinline__ void a_frag4(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t w8 = w >> 8;
  a[0] = (w & 0x000F000Fu) | 0x64006400u;   // row g:     1024 + q
  a[1] = (w & 0x00F000F0u) | 0x64006400u;   // row g + 8: 1024 + 16 q
  a[2] = (w8 & 0x000F000Fu) | 0x64006400u;  // row g
  a[3] = (w8 & 0x00F000F0u) | 0x64006400u;  // row g + 8
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}


__device__ __forceinline__ uint16_t f16_sat(float v) {
  return __half_as_ushort(__float2half_rn(fminf(fmaxf(v, -65504.f), 65504.f)));
}

// Magnitude bits of a float with the sign cleared (they order as |v|; NaN above infinity). From
// kF16Clamp (65520.0f) on, a value is past the largest finite fp16 and f16_sat clamps it.
__device__ __forceinline__ uint32_t mag_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }
constexpr uint32_t kF16Clamp = 0x477FF000u;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kStages = 3;  // 128-row groups of codes in flight per warp (shared-memory ring)

// Codes of one 128-row group of one unit into ring stage `stage`: NM matrices x TL 16-column
// tiles x NL 512-byte blocks, each lane copying its own 16 bytes of every block (and later
// reading only those).
template <int NM, int TL, int NL>
__device__ __forceinline__ void issue_group(uint32_t ring, int stage, const QMat* mats,
                                            size_t tile0, int grp, int KP, int lane) {
#pragma unroll
  for (int m = 0; m < NM; ++m)
#pragma unroll
    for (int t = 0; t < TL; ++t)
#pragma unroll
      for (int l = 0; l < NL; ++l)
        cp_async16(ring + (uint32_t)(((((stage * NM + m) * TL + t) * NL + l) * 32 + lane) * 16),
                   mats[m].q + ((tile0 + t) * KP + (size_t)grp * NL + l) * 512 + lane * 16);
}

// Per group, for this lane's two rows n, n + 8 of every tile and every matrix of the unit: the
// scale (fp32) and the constant the MMA's A values carry, 1024 + z; for 4-bit rows n + 8, whose
// values are 1024 + 16 q, the scale / 16 and 1024 + 16 z (both exact).
template <int NM, int TL>
struct GroupQ {
  float sc[NM][TL][2];
  float off[NM][TL][2];
};

template <int BITS, int NM, int TL>
__device__ __forceinline__ void load_group_q(GroupQ<NM, TL>& q, const QMat* mats, int ex_ix,
                                             int grp, int groups, int N, int n, bool ok) {
#pragma unroll
  for (int m = 0; m < NM; ++m)
#pragma unroll
    for (int t = 0; t < TL; ++t)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const size_t ix = ((size_t)ex_ix * groups + (ok ? grp : 0)) * N + n + 16 * t + 8 * h;
        const float sc = __half2float(__ushort_as_half(mats[m].s[ix]));
        const float z = (float)mats[m].z[ix];
        const bool up = BITS == 4 && h == 1;
        q.sc[m][t][h] = up ? sc * 0.0625f : sc;
        q.off[m][t][h] = up ? 1024.f + 16.f * z : 1024.f + z;
      }
}

// The group's activation sum per token 2c + j (this lane's accumulator columns): M = 0 takes it
// from sb_in (precomputed by act_prep_kernel); M = 1 forms it from the B fragments themselves, at
// 8 bits with one more MMA per step against an all-ones A fragment, at 4 bits (where the MMAs per
// code byte double) by fp32 adds of the lane's H values and three shuffles (measured: 4-bit down
// 192.5 -> 188.4 us on the decode shape, while the adds cost the 8-bit pass 12 us).
template <int BITS, int MODE, int NM, int TL, int NL>
__device__ __forceinline__ void compute_group(const uint4 (&code)[NM][TL][NL],
                                              const uint32_t (&bq)[8][2],
                                              const float (&sb_in)[2], const GroupQ<NM, TL>& q,
                                              float (&acc)[NM][TL][4]) {
  float cg[NM][TL][4];
#pragma unroll
  for (int m = 0; m < NM; ++m)
#pragma unroll
    for (int t = 0; t < TL; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) cg[m][t][i] = 0.f;
  constexpr bool kAddSums = MODE == 1 && BITS == 4;
  float sb[4] = {sb_in[0], sb_in[1], 0.f, 0.f};
  if (MODE == 1) sb[0] = sb[1] = 0.f;
  const uint32_t ones[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};  // fp16 1.0
  // 4-bit M = 1: this lane's share of token g's group sum (k = 2c, 2c + 1, 2c + 8, 2c + 9 of
  // every step)
  float part = 0.f;
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    const uint32_t b0 = bq[st][0], b1 = bq[st][1];
    if (kAddSums) {
      const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&b0));
      const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&b1));
      part += (f0.x + f0.y) + (f1.x + f1.y);
    } else if (MODE == 1) {
      mma16816(sb, ones, b0, b1);
    }
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int t = 0; t < TL; ++t) {
        uint32_t af[4];
        if (BITS == 8) {
          const uint4 v = code[m][t][st / 2];
          const uint32_t lo = (st & 1) ? v.z : v.x, hi = (st & 1) ? v.w : v.y;
          a_frag8(lo, hi, af);
        } else {
          const uint4 v = code[m][t][st / 4];
          const int qq = st & 3;
          a_frag4(qq == 0 ? v.x : qq == 1 ? v.y : qq == 2 ? v.z : v.w, af);
        }
        mma16816(cg[m][t], af, b0, b1);
      }
  }
  if (kAddSums) {
    // the four lanes of token g add their shares; each lane then takes tokens 2c and 2c + 1
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    const int c = threadIdx.x & 3;
    sb[0] = __shfl_sync(0xffffffffu, part, 8 * c);
    sb[1] = __shfl_sync(0xffffffffu, part, 8 * c + 4);
  }
  // element i: row n + 8 (i / 2) of the tile, token 2c + i % 2
#pragma unroll
  for (int m = 0; m < NM; ++m)
#pragma unroll
    for (int t = 0; t < TL; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int h = i >> 1;
        acc[m][t][i] = fmaf(q.sc[m][t][h], fmaf(-q.off[m][t][h], sb[i & 1], cg[m][t][i]),
                            acc[m][t][i]);
      }
}

// 16-column tiles per work unit: 4-bit groups carry half the bytes of 8-bit ones, so a 4-bit
// unit takes two tiles (gate/up, two matrices) or four (down) to give each group at least the same
// code bytes, and its B fragments serve more MMAs (4-bit down with four tiles: 157.7 -> 147.5 us
// on the decode shape; the 8-bit down pass with two measured slower).
template <int BITS, int MODE>
__host__ __device__ constexpr int tiles_per_unit() {
  return BITS == 8 ? 1 : (MODE == 0 ? 2 : 4);
}

template <int NM, int TL, int NL>
__host__ __device__ constexpr int ring_bytes_per_warp() {
  return kStages * NM * TL * NL * 512;
}

// Work unit = (8-row tile, 16 * TL output columns), taken from a device counter so that units of
// every length balance across warps. Units with the same column strip run side by side (unit u
// -> tile u % n_tiles, strip u / n_tiles), so the tiles of one expert share its codes in L2.
// Each warp keeps kStages groups of codes in flight through its shared-memory ring (cp.async,
// 16 bytes per lane per block); the activations of the next group are loaded into registers
// while the current one is computed.
// Register budgets (minimum CTAs per SM): 4-bit gate/up 1, so it keeps its ~160 registers
// (three CTAs per SM, measured faster than 128 registers at four); 8-bit gate/up 4, which its
// 48 KB ring allows anyway; the down passes the compiler's default (0: none given).
template <int BITS, int MODE>
__global__ void __launch_bounds__(kQThreads, MODE == 0 ? (BITS == 8 ? 4 : 1) : 0)
    qffn_kernel(const QArgs a) {
  constexpr int NM = MODE == 0 ? 2 : 1;  // matrices per unit (gate and up, or down)
  constexpr int NL = BITS == 8 ? 4 : 2;  // 512-byte code blocks per group, matrix and tile
  constexpr int TL = tiles_per_unit<BITS, MODE>();
  constexpr int RB = ring_bytes_per_warp<NM, TL, NL>();
  extern __shared__ __align__(16) uint8_t qsmem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const uint32_t ring = (uint32_t)__cvta_generic_to_shared(qsmem) + (uint32_t)(warp * RB);
  const uint4* ring4 = reinterpret_cast<const uint4*>(qsmem + warp * RB);
  griddep_wait();
  const int n_tiles = a.meta->n_tiles;
  const int strips = a.N / (16 * TL);
  const int units = n_tiles * strips;  // < 2^31: tiles of 8 rows x column strips
  const int KP = a.K / (16 * (BITS == 8 ? 2 : 4));
  const int groups = a.K / kGroup;
  int* counter = &a.meta->work[MODE];
  // Tail split. Units have equal length, so with W warps the last, partial round leaves most
  // warps idle. The first `full` units run whole; each of the `tail` remaining ones is cut into
  // S pieces over group ranges. S (the same on every warp) minimises the tail's time: rounds of
  // pieces x piece length, a piece costing its groups plus about kPieceCost groups of start-up
  // and reduction. Each piece stores its partial accumulators; the last piece of a unit to
  // finish (ticket) adds all of them in piece order and runs the epilogue.
  constexpr int kPieceCost = 3;
  const int W = gridDim.x * (kQThreads / 32);
  const int full = units / W * W, tail = units - full;
  int S = 1;
  // (the down pass's units span only d_ff / 128 groups, too few for pieces to pay: measured)
  if (MODE == 0 && tail > 0) {
    long long best = (long long)((tail + W - 1) / W) * (groups + kPieceCost);  // x S = 1
    for (int s2 = 2; s2 <= 16 && s2 <= groups && tail * s2 <= a.tail_cap; ++s2) {
      const long long r = (tail * s2 + W - 1) / W;
      // r (groups / s2 + kPieceCost) < best / S, in integers
      if (r * (groups + kPieceCost * s2) * S < best * s2) {
        best = r * (groups + kPieceCost * s2);
        S = s2;
      }
    }
  }
  const int work = full + tail * S;
  constexpr int F = NM * TL * 4;  // accumulators per lane
  uint32_t clamp = 0u;             // largest magnitude this lane stored in fp16 (mag_bits)
  while (true) {
    int v = 0;
    if (lane == 0) v = atomicAdd(counter, 1);
    v = __shfl_sync(0xffffffffu, v, 0);
    if (v >= work) break;
    int u = v;
    int gA = 0, gB = groups, piece = -1;
    if (MODE == 0 && S > 1 && v >= full) {
      piece = (v - full) % S;
      u = full + (v - full) / S;
      gA = piece * groups / S;
      gB = (piece + 1) * groups / S;
    }
    const TileEntry te = a.tiles[u % n_tiles];
    const int strip = u / n_tiles;
    const bool shared = te.expert >= a.E;
    const int ex_ix = shared ? te.expert - a.E : te.expert;
    const QMat* mats = shared ? a.shared : a.routed;
    const size_t tile0 = (size_t)ex_ix * (a.N / 16) + (size_t)strip * TL;
    // start the ring: groups gA .. gA + kStages - 2 (stage = (group - gA) % kStages)
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
      if (gA + s < gB) issue_group<NM, TL, NL>(ring, s, mats, tile0, gA + s, KP, lane);
      cp_async_commit();
    }
    // Row r of the tile reads, in M = 0, x16 row (shared) arow0 + r or (routed) the token of
    // slot perm_slot[row0 + r]; in M = 1, H row row0 + r. This lane's B fragments come from row
    // g; its accumulator columns are rows 2c and 2c + 1, whose activation sums it needs.
    auto src_row = [&](int r) -> long long {
      if (MODE == 1) return te.row0 + r;
      return shared ? te.arow0 + r : a.perm_slot[te.row0 + r] / a.top_k;
    };
    const int tok = g;
    const bool tok_ok = tok < te.rows;
    const uint32_t* brow =
        reinterpret_cast<const uint32_t*>(a.src + src_row(tok_ok ? tok : 0) * a.K);
    // M = 0: the group sums of the two x16 rows, sbx[row][grp]
    const float* bsum_j[2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
      bsum_j[j] = MODE == 0 && 2 * c + j < te.rows ? a.bsum + src_row(2 * c + j) * groups
                                                    : nullptr;
    auto load_sums = [&](int grp, float (&sb)[2]) {
#pragma unroll
      for (int j = 0; j < 2; ++j)
        sb[j] = bsum_j[j] != nullptr && grp < gB ? bsum_j[j][grp] : 0.f;
    };
    const int n = strip * 16 * TL + g;  // this lane's rows of tile t: n + 16 t and n + 16 t + 8
    float acc[NM][TL][4];
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int t = 0; t < TL; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[m][t][i] = 0.f;
    // the group's B fragments: 64 contiguous bytes per lane in the fragment-order layout
    auto load_b = [&](int grp, bool ok, uint32_t (&b)[8][2]) {
      const uint4* p4 = reinterpret_cast<const uint4*>(brow + grp * 64 + c * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = ok ? p4[q] : make_uint4(0u, 0u, 0u, 0u);
        b[2 * q][0] = v.x;
        b[2 * q][1] = v.y;
        b[2 * q + 1][0] = v.z;
        b[2 * q + 1][1] = v.w;
      }
    };
    uint32_t bq[8][2];
    load_b(gA, tok_ok, bq);
    GroupQ<NM, TL> gq;
    load_group_q<BITS, NM, TL>(gq, mats, ex_ix, gA, groups, a.N, n, true);
    float sb[2];
    load_sums(gA, sb);
    for (int grp = gA; grp < gB; ++grp) {
      const int ahead = grp + kStages - 1;
      if (ahead < gB)
        issue_group<NM, TL, NL>(ring, (ahead - gA) % kStages, mats, tile0, ahead, KP, lane);
      cp_async_commit();
      cp_async_wait<kStages - 1>();  // this lane's copies of group grp have landed
      uint4 code[NM][TL][NL];
      const int stage = (grp - gA) % kStages;
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int t = 0; t < TL; ++t)
#pragma unroll
          for (int l = 0; l < NL; ++l)
            code[m][t][l] = ring4[(((stage * NM + m) * TL + t) * NL + l) * 32 + lane];
      // the next group's activations, scales and zero-points, loaded during this group's MMAs
      uint32_t bn[8][2];
      load_b(grp + 1, tok_ok && grp + 1 < gB, bn);
      GroupQ<NM, TL> gn;
      load_group_q<BITS, NM, TL>(gn, mats, ex_ix, grp + 1, groups, a.N, n, grp + 1 < gB);
      float sbn[2];
      load_sums(grp + 1, sbn);
      compute_group<BITS, MODE, NM, TL, NL>(code, bq, sb, gq, acc);
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        bq[st][0] = bn[st][0];
        bq[st][1] = bn[st][1];
      }
      gq = gn;
      sb[0] = sbn[0];
      sb[1] = sbn[1];
    }
    cp_async_wait<0>();
    if (MODE == 0 && piece >= 0) {
      // a piece of a split tail unit: park the partials; the unit's last piece adds them
      const int tu = u - full;
      float* mine = a.tail_acc + (size_t)(tu * S + piece) * F * 32;
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int t = 0; t < TL; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i) mine[((m * TL + t) * 4 + i) * 32 + lane] = acc[m][t][i];
      __threadfence();
      __syncwarp();
      int done = 0;
      if (lane == 0) done = atomicAdd(a.tail_ticket + tu, 1);
      done = __shfl_sync(0xffffffffu, done, 0);
      if (done != S - 1) continue;
      __threadfence();  // the other pieces' partials, published before their tickets
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int t = 0; t < TL; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float* p0 = a.tail_acc + (size_t)tu * S * F * 32 +
                              ((m * TL + t) * 4 + i) * 32 + lane;
            float sum = __ldcg(p0);
            for (int q = 1; q < S; ++q) sum += __ldcg(p0 + q * F * 32);
            acc[m][t][i] = sum;
          }
      if (lane == 0) a.tail_ticket[tu] = 0;  // ready for the next launch
    }
    // epilogue: element i of tile t is (column n + 16 t + 8 (i / 2), token 2 c + i % 2)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 2 * c + (i & 1);
      if (t >= te.rows) continue;
      long long orow = te.row0 + t;
      float gate = 1.f;
      if (MODE == 1 && !shared) {
        const int slot = a.perm_slot[te.row0 + t];
        orow = slot;
        if (a.topk_w != nullptr) gate = a.topk_w[slot];
      }
#pragma unroll
      for (int t = 0; t < TL; ++t) {
        const int col = n + 16 * t + 8 * (i >> 1);
        float v;
        if (MODE == 0) {
          const float gv = acc[0][t][i], uv = acc[NM - 1][t][i];
          v = gv / (1.0f + __expf(-gv)) * uv;
        } else {
          v = gate * acc[0][t][i];
        }
        clamp = max(clamp, mag_bits(v));
        // H (M = 0) in fragment order for the down pass; Y (M = 1) in plain column order
        a.out[orow * a.N + (MODE == 0 ? frag_pos(col) : col)] = f16_sat(v);
      }
    }
  }
  if (__any_sync(0xffffffffu, clamp >= kF16Clamp) && lane == 0)
    atomicOr(a.status, MOE_DEVFAULT_FP16_RANGE);
}

}  // namespace

cudaError_t launch_quantize(int bits, int n_mat, int K, int N, const uint16_t* W, uint8_t* q,
                            uint16_t* scale, uint8_t* zero, cudaStream_t st) {
  const size_t code_bytes = (size_t)n_mat * K * N * bits / 8;
  if (bits == 4) {  // nibbles are OR-ed into zeroed words
    const cudaError_t e = cudaMemsetAsync(q, 0, code_bytes, st);
    if (e != cudaSuccess) return e;
  }
  const long long total = (long long)n_mat * (K / kGroup) * N;
  const int grid = (int)std::min<long long>((total + 255) / 256, 8LL * num_sms());
  if (bits == 8)
    quantize_kernel<8><<<grid, 256, 0, st>>>(W, q, scale, zero, n_mat, K, N);
  else
    quantize_kernel<4><<<grid, 256, 0, st>>>(W, q, scale, zero, n_mat, K, N);
  return cudaGetLastError();
}

int quant_tail_cap() { return 64 * num_sms(); }  // warps an SM can hold, over the GPU

cudaError_t launch_quant_act(const Shape& s, const QFfnPtrs& p, cudaStream_t st) {
  const long long items = (long long)s.T * ((s.d / 8 + 31) / 32);  // warps of work
  const int grid = (int)std::min<long long>((items + 7) / 8, 8LL * num_sms());
  return launch_k(act_prep_kernel, dim3(grid), dim3(256), 0, st, p.x, s.T, s.d, p.x16, p.sbx,
                  p.tail_ticket, 2 * p.tail_cap);
}

cudaError_t launch_quant_ffn(const Shape& s, int bits, const QFfnPtrs& p, cudaStream_t st,
                             cudaEvent_t ev_mid) {
  QArgs a{};
  a.E = s.E;
  a.tiles = p.tiles;
  a.meta = p.meta;
  a.perm_slot = p.perm_slot;
  a.topk_w = p.topk_w;
  a.top_k = s.k;
  a.tail_acc = p.tail_acc;
  a.tail_cap = p.tail_cap;
  a.status = p.status;
  a.tail_ticket = p.tail_ticket;  // gate/up; the down pass uses the next tail_cap
  const int sms = num_sms();
  // persistent: as many CTAs as fit (work units come from the counters in Meta)
  auto smem_of = [&](int mode) {
    const int rb =
        bits == 8 ? (mode == 0 ? ring_bytes_per_warp<2, tiles_per_unit<8, 0>(), 4>()
                               : ring_bytes_per_warp<1, tiles_per_unit<8, 1>(), 4>())
                  : (mode == 0 ? ring_bytes_per_warp<2, tiles_per_unit<4, 0>(), 2>()
                               : ring_bytes_per_warp<1, tiles_per_unit<4, 1>(), 2>());
    return (size_t)(kQThreads / 32) * rb;
  };
  auto grid_of = [&](void (*k)(const QArgs), size_t smem) {
    int per_sm = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kQThreads, smem) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    return dim3(per_sm * sms);
  };
  // ---- gate/up: K = d, N = d_ff
  a.routed[0] = {p.qw->gate.q, p.qw->gate.scale, p.qw->gate.zero};
  a.routed[1] = {p.qw->up.q, p.qw->up.scale, p.qw->up.zero};
  a.shared[0] = {p.qw->sh_gate.q, p.qw->sh_gate.scale, p.qw->sh_gate.zero};
  a.shared[1] = {p.qw->sh_up.q, p.qw->sh_up.scale, p.qw->sh_up.zero};
  a.src = p.x16;
  a.bsum = p.sbx;
  a.out = p.h;
  a.K = s.d;
  a.N = s.f;
  cudaError_t err;
  const size_t sm0 = smem_of(0), sm1 = smem_of(1);
  if (bits == 8)
    err = launch_k(qffn_kernel<8, 0>, grid_of(qffn_kernel<8, 0>, sm0), dim3(kQThreads), sm0, st,
                   a);
  else
    err = launch_k(qffn_kernel<4, 0>, grid_of(qffn_kernel<4, 0>, sm0), dim3(kQThreads), sm0, st,
                   a);
  if (err != cudaSuccess) return err;
  if (ev_mid != nullptr && (err = cudaEventRecord(ev_mid, st)) != cudaSuccess) return err;
  // ---- down: K = d_ff, N = d
  a.routed[0] = {p.qw->down.q, p.qw->down.scale, p.qw->down.zero};
  a.routed[1] = a.routed[0];
  a.shared[0] = {p.qw->sh_down.q, p.qw->sh_down.scale, p.qw->sh_down.zero};
  a.shared[1] = a.shared[0];
  a.src = p.h;
  a.bsum = nullptr;
  a.tail_ticket = p.tail_ticket + p.tail_cap;
  a.out = p.y;
  a.K = s.f;
  a.N = s.d;
  if (bits == 8)
    return launch_k(qffn_kernel<8, 1>, grid_of(qffn_kernel<8, 1>, sm1), dim3(kQThreads), sm1, st,
                    a);
  return launch_k(qffn_kernel<4, 1>, grid_of(qffn_kernel<4, 1>, sm1), dim3(kQThreads), sm1, st,
                  a);
}

}  // namespace moe
