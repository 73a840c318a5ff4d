// Internal launch interface between the C-ABI layer (moe_api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <utility>

#include "../../include/moe.h"

namespace moe {

constexpr int kTileM = 128;        // rows per grouped-GEMM tile (one UMMA M=128 accumulator)
constexpr int kQTileM = 8;         // rows per tile of the quantized expert path (MMA N = 8)
constexpr int kPermuteBlock = 256; // slots per dispatch block

struct Shape {
  int T, d, E, k, f, S, mode;
  int G, Gk;      // group-limited routing: groups, groups kept (G = 0: off)
  bool reroute;   // Level-2 overflow re-route (only with a capacity limit)
  float tau;
  int C;          // capacity, or INT32_MAX for no limit
  long long TK;   // T * k
  long long rows; // rows of the expert-ordered buffers: T * k + S * T
  int n_pblk;     // dispatch blocks = ceil(T*k / kPermuteBlock)
  int tile_m;     // rows per row tile: kTileM (bf16 GEMM) or kQTileM (quantized experts)
  int max_tiles;  // upper bound on row tiles
};

// One grouped-GEMM row tile: rows [row0, row0 + rows) of the expert-ordered buffers belong to
// `expert` (E + s for shared expert s); the A operand of the gate/up GEMM starts at row `arow0`
// of its source (the gathered rows for routed experts, x itself for shared ones). The expert's
// row tiles are entries [g0, g0 + gn) of the list (the GEMMs' work order is expert-major).
struct TileEntry {
  int expert;
  int row0;
  int rows;
  int arow0;
  int g0;
  int gn;
};

// Meta block inside the workspace (device ints); moe_workspace_init zeroes it.
struct Meta {
  int n_tiles;        // row tiles written by the dispatch scan
  int n_kept;         // N = kept routed slots
  int refine_count;   // near-tie tokens listed by the router (reset by the router GEMM)
  int dispatch_ticket; // dispatch histogram CTAs finished (reset by the last one)
  int reroute_rounds; // proposal rounds of the last overflow re-route (diagnostic)
  int work[2];        // next work unit of the quantized gate/up and down passes
  int reroute_exact;  // first windows listed for the re-route's exact pass (zero between calls)
  unsigned check_arrive, check_gen;  // grid barrier of moe_check_bounded_waits (arrivals zero)
  int pad[54];
};
static_assert(sizeof(Meta) == 256, "moe_workspace_init clears the status word and this block");

// Offsets of every buffer carved from the caller's workspace (bytes, 256-aligned).
struct WsLayout {
  size_t status, meta, topk_idx, topk_w, counts, offsets, perm_slot, slot_pos;
  size_t blk_hist, blk_base, tiles, wg_t, rpart, rrec, xp, h, y, x_stage,
      u_stage, out_stage;
  size_t x16, sbx, tail_acc, tail_ticket;  // quantized experts only
  // overflow re-route (zero-sized unless enabled)
  size_t sfull, maxl, pref, rr_tok, rr_exp, rr_bits, rr_ctl;
  size_t total;
};

Shape make_shape(const moe_config& c);
WsLayout ws_layout(const Shape& s);

// ---- launchers (all asynchronous on `st`; return cudaGetLastError()) ----
// Router scratch carved from the workspace.
constexpr int kRouterMaxCand = 16;
// One near-tie record, 128 bytes: [0] token, [1] candidate count (n > 0) or -1 (every expert),
// [2, 2 + n) the candidate experts in index order (n <= kRouterMaxCand).
constexpr int kRouterRecInts = 32;
struct RouterScratch {
  uint16_t* wg_t;    // E x d bf16: W_g transposed for this call when the caller has none
  float* part;       // [splits, T, round_up(E, 64)] fp32 partial logits
  int32_t* rrec;     // [T][kRouterRecInts] near-tie records, appended by the selection
  int* rcount;       // their number (cleared by the router GEMM at the start of each call)
  float* sfull;      // [T, E] selection scores kept for the overflow re-route, or nullptr
  float* maxl;       // [T] largest |logit| per token (with sfull)
};
// K slices of the router GEMM for T tokens and hidden size d.
int router_splits(int T, int d);
// W_g_t: W_g transposed ([E, d], from moe_prepare_router), or nullptr to transpose into
// rs.wg_t first.
cudaError_t launch_router(const Shape& s, const uint16_t* x, const uint16_t* W_g,
                          const uint16_t* W_g_t, const float* bias, const float* u,
                          int32_t* topk_idx, float* topk_w, const RouterScratch& rs, int* status,
                          cudaStream_t st);
// W_g_t[e, j] = W_g[j, e] for W_g [d, E].
cudaError_t launch_router_transpose(int d, int E, const uint16_t* W_g, uint16_t* W_g_t,
                                    cudaStream_t st);

// Level-2 overflow re-route (reroute.cu). Per-token and per-expert state lives in the workspace;
// the preceding router call left the selection scores (sfull), the row scales (maxl) and the
// transposed router weights (WgT) there, and the preceding dispatch left counts and slot_pos.
struct RerouteArgs {
  const uint16_t* x;       // [T, d] bf16
  const uint16_t* WgT;     // [E, d] bf16
  const float* bias;       // [E] (BIAS_SELECT)
  const float* u;          // [T, E] (GUMBEL)
  const float* sfull;      // [T, E] tensor-core selection scores
  const float* maxl;       // [T] largest |logit| per token
  int32_t* topk_idx;       // [T, k] in/out: dropped slots get their new expert
  float* topk_w;           // [T, k] out for re-routed tokens: softmax over the final experts
  const int32_t* counts;   // [E] Level-1 counts (before the capacity clamp)
  const int32_t* slot_pos; // [T * k] Level-1 positions (-1: dropped)
  uint8_t* pref;           // [T, PS] preference lists (expert ids < 256), PS = E rounded up to 16
  int32_t *plen, *dem, *ptr, *held;  // [T] each: list length, dropped slots, next position, kept
  int32_t *rlen, *ext_list;          // [T] each: exactly ordered prefix, tokens needing more
  int32_t* ex_list;        // [T] tokens whose first window waits for reroute_exact_kernel
  int32_t* ex_count;       // their number (zero between calls)
  int32_t *room, *cut, *touched;     // [E] each
  uint32_t* bits;          // [E, W] proposals held by each expert, bit t of word t / 32
  int32_t* rejected;       // [1024] turn-aways per round
  int32_t* extended;       // [1024] tokens listed for their next exact window, per round
  int32_t* ctl;            // [2] grid barrier: arrivals, generation
  int32_t* rounds_out;     // proposal rounds of the last call
  int* status;
  int T, d, E, k, mode, C, W, PS;
  float tau;
};
cudaError_t launch_reroute(const RerouteArgs& a, cudaStream_t st);
// moe_check_bounded_waits: both bounded waits against conditions that never come true.
cudaError_t launch_wait_check(uint64_t limit_ns, int* status, int32_t* expired,
                              unsigned* arrive, unsigned* gen, cudaStream_t st);

// Dispatch: histogram (its last CTA also scans, and builds the row-tile list into tiles/meta
// unless tiles is nullptr), then the stable scatter. *ticket is zero before and after.
cudaError_t launch_permute(const Shape& s, const int32_t* topk_idx, int32_t* counts,
                           int32_t* offsets, int32_t* perm_slot, int32_t* slot_pos,
                           int32_t* blk_hist, int32_t* blk_base, int* ticket, int* status,
                           TileEntry* tiles, Meta* meta, cudaStream_t st);

// moe_permute_noalloc: the same kernels with their scratch in a static device array.
cudaError_t launch_permute_noalloc(const Shape& s, const int32_t* topk_idx, int32_t* counts,
                                   int32_t* offsets, int32_t* perm_slot, int32_t* slot_pos,
                                   int* fault_bits, cudaStream_t st);

// Builds the row-tile list from offsets (routed) plus the shared experts' identity segments.
cudaError_t launch_tiles(const Shape& s, const int32_t* offsets, TileEntry* tiles, Meta* meta,
                         cudaStream_t st);
// launch_tiles (unless the dispatch already built the list, tiles_built), then gathers x rows
// into expert order
// (xp[p] = x[perm_slot[p] / k] for p < offsets[E]).
cudaError_t launch_tiles_and_gather(const Shape& s, const uint16_t* x, const int32_t* perm_slot,
                                    const int32_t* offsets, uint16_t* xp, TileEntry* tiles,
                                    Meta* meta, bool tiles_built, cudaStream_t st);

struct FfnPtrs {
  const uint16_t* x;
  const uint16_t* xp;
  const int32_t* perm_slot;
  const float* topk_w;
  const uint16_t *W_gate, *W_up, *W_down;
  const uint16_t *Wsh_gate, *Wsh_up, *Wsh_down;
  const uint16_t *W_down_f16, *Wsh_down_f16;  // fp16 down path when W_down_f16 != nullptr
  uint16_t* h;                                // H: fp16 on the fp16 down path, else bf16
  void* y;  // slot-ordered expert outputs: fp16 on the fp16 down path, fp32 on the bf16 one
  const TileEntry* tiles;
  const Meta* meta;
  int* status;
};
// ev_mid (optional): recorded on st between the gate/up and the down GEMM.
cudaError_t launch_grouped_ffn(const Shape& s, const FfnPtrs& p, cudaStream_t st,
                               cudaEvent_t ev_mid = nullptr);

// Weight-only quantized experts (quant_ffn.cu).
cudaError_t launch_quantize(int bits, int n_mat, int K, int N, const uint16_t* W, uint8_t* q,
                            uint16_t* scale, uint8_t* zero, cudaStream_t st);
struct QFfnPtrs {
  const uint16_t* x;          // [T, d] bf16
  uint16_t* x16;              // [T, d] fp16 copy of x (launch_quant_act)
  float* sbx;                 // [T, d / 128] sums of x16 over each 128-column group
  float* tail_acc;            // [tail_cap][16][32] partials of split tail units
  int* tail_ticket;           // [2][tail_cap]: per pass, pieces finished per tail unit
  int tail_cap;               // quant_tail_cap()
  uint16_t* h;                // H [rows, f] fp16
  uint16_t* y;                // Y [rows, d] fp16, slot order
  const int32_t* perm_slot;   // [T*k]
  const float* topk_w;        // [T*k] or nullptr
  const TileEntry* tiles;     // kQTileM-row tiles (launch_tiles_and_gather)
  Meta* meta;
  const moe_qweights* qw;
  int* status;                // device status word (MOE_DEVFAULT_FP16_RANGE)
};
// Pieces of split tail units the quantized passes can hold (at most one per resident warp).
int quant_tail_cap();
// The quantized passes' activations: x16 = fp16(x) and its 128-column group sums sbx; also
// zeroes the passes' tail tickets.
cudaError_t launch_quant_act(const Shape& s, const QFfnPtrs& p, cudaStream_t st);
// ev_mid (optional): recorded on st between the gate/up and the down pass.
cudaError_t launch_quant_ffn(const Shape& s, int bits, const QFfnPtrs& p, cudaStream_t st,
                             cudaEvent_t ev_mid = nullptr);

// y_f32: the slot rows are fp32 (bf16 down path), else fp16.
cudaError_t launch_combine(const Shape& s, const void* y, bool y_f32, const int32_t* slot_pos,
                           uint16_t* out, cudaStream_t st);

// fault (optional): MOE_DEVFAULT_FP16_RANGE is OR-ed in when a weight had to be clamped.
cudaError_t launch_pack_f16(const uint16_t* src, uint16_t* dst, size_t n, int* fault,
                            cudaStream_t st);

cudaError_t launch_bias_update(int E, const int32_t* counts, float* bias, float decay, float rate,
                               cudaStream_t st);

int num_sms();

// Device side of programmatic dependent launch: wait until the preceding kernel in the stream
// has completed and its memory is visible. Every kernel of the layer calls this before it reads
// or writes global memory (setup that touches only shared memory, TMEM and parameters may come
// first), so launching it early (launch_k) is safe whatever precedes it.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel on the stream (launched with programmatic stream serialization) start
// once every CTA of this one has passed this point or exited.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kernel` with programmatic stream serialization: it may begin while the previous
// kernel on the stream drains (its griddep_wait() provides the ordering).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Tensor maps (cuTensorMapEncodeTiled through the runtime's driver entry point), 128-byte swizzle.
// 2-D over a row-major [rows, cols] 16-bit matrix with a box of box_cols (inner) x box_rows.
bool make_tmap_2d(CUtensorMap* m, const void* ptr, long long rows, long long cols, int box_cols,
                  int box_rows, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
// 3-D over a row-major [n, rows, cols] 16-bit tensor with a box of box_cols x box_rows x 1.
bool make_tmap_3d(CUtensorMap* m, const void* ptr, long long n, long long rows, long long cols,
                  int box_cols, int box_rows,
                  CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);

}  // namespace moe
