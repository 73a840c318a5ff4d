/*
 * moe.h -- C ABI of a sparse Mixture-of-Experts FFN layer forward pass on one GB300 (sm_103a).
 *
 * The layer (forward only, per token t of x[T, d]):
 *   1. router logits   logits[t, e] = sum_j x[t, j] * W_g[j, e]          (fp32 accumulation)
 *   2. selection score s[t, e] = logits                     (MOE_ROUTE_PLAIN)
 *                                logits + expert_bias[e]    (MOE_ROUTE_BIAS_SELECT)
 *                                (logits - log(-log u)) / tau   (MOE_ROUTE_GUMBEL)
 *   3. top-k           the k largest s, ordered by s descending, ties to the lower index
 *                      (optionally only among the experts of the best expert groups)
 *   4. gates           softmax over the k selected logits (PLAIN, BIAS_SELECT) or over the k
 *                      selected scores s (GUMBEL)
 *   5. dispatch        per-expert segments, tokens in ascending order; with a capacity C an
 *                      expert keeps its first C slots (token order) and drops the rest (gate 0)
 *   6.-8. experts      y = (silu(x W_gate[e]) * (x W_up[e])) W_down[e]   (SwiGLU)
 *   9. shared experts  z_s = SwiGLU_s(x) for every token, gate 1
 *  10. combine         out[t] = sum over kept j of gate[t,j] * y(t,j) + sum_s z_s[t]
 *
 * Sources (titles of the pages that define the method):
 *   router, top-k, softmax over top-k, weighted sum of experts:
 *       "大模型MoE稀疏激活原理与工程实践", §3.1 路由器 (Router code) and §3.2 专家.
 *   bias-adjusted (aux-loss-free) selection:
 *       "AI架构演进从稀疏MoE到条件记忆的工程实践", gating-network code (expert bias added to the
 *       scores that top-k ranks) and its layered-architecture figure (routing, dispatch,
 *       compute, aggregation layers).
 *   Gumbel top-k with temperature:
 *       "GPT-4 Has 1.8 Trillion Parameters. It Uses 2% of Them Per Token", §3.1 门控网络.
 *   expert capacity and overflow:
 *       "参数规模与稀疏激活的真相拆解", §3.2 专家容量 (Level 1 hard limit).
 *   SwiGLU experts: "GPT-4 ... 2% ...", §3.3; shared experts: "V4" rework page, §2.2.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are caller-owned DEVICE memory unless the name ends in _host.
 *     The library allocates nothing on the device and keeps no per-call global state; every
 *     scratch buffer lives in the caller's workspace `ws` (see moe_workspace_size).
 *   - Tensor pointers are 16-byte aligned (TMA tiles, the gather and the exact dot products move
 *     16-byte pieces); an x that is not returns MOE_ERR_INVALID_ARG from every entry point that
 *     takes x.
 *   - Row-major layouts. bf16 tensors are passed as uint16_t bit patterns.
 *     x [T, d]; W_g [d, E]; W_gate, W_up [E, d, d_ff]; W_down [E, d_ff, d];
 *     shared expert weights [S, d, d_ff] / [S, d_ff, d]; expert_bias fp32 [E];
 *     gumbel_u fp32 [T, E] with values in (0, 1).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream) and
 *     returns before it completes. Argument errors are detected on the host and returned
 *     synchronously (nothing is enqueued then). Errors detected by the kernels (an expert index
 *     outside [0, E), a pipeline wait that timed out) are recorded in a status word inside `ws`
 *     and read with moe_device_status.
 *   - Supported sizes: T >= 0; 1 <= E <= 256; 1 <= top_k <= min(E, 8); 0 <= n_shared <= 4;
 *     d and d_ff multiples of 64; T * (top_k + n_shared) < 2^31. Anything else returns
 *     MOE_ERR_UNSUPPORTED (a negative T returns MOE_ERR_INVALID_ARG).
 *   - An empty batch (T = 0) is valid everywhere and launches no kernel. The configuration is
 *     still validated; tensor pointers and the workspace are not examined (an empty tensor may
 *     pass NULL). Only the per-expert dispatch outputs are non-empty: moe_permute and
 *     moe_permute_noalloc (which require counts and offsets) and moe_layer_forward(_profiled)
 *     (for the members of route_out that are given) clear counts [E] and offsets [E + 1] with
 *     cudaMemsetAsync on the stream; moe_permute_noalloc also clears fault_bits if given;
 *     moe_layer_forward_profiled records its seven events back to back.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* NULL pointer where one is required, negative T or non-positive
                                other size, bad mode */
  MOE_ERR_UNSUPPORTED = 2,   /* sizes outside the supported range above */
  MOE_ERR_WORKSPACE = 3,     /* ws is NULL, misaligned (needs 256 B) or smaller than required */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed (launch, tensor-map encode) */
  MOE_ERR_DEVICE_FAULT = 5   /* a kernel recorded a fault in the status word */
} moe_status;

typedef enum {
  MOE_ROUTE_PLAIN = 0,       /* select and gate on the logits */
  MOE_ROUTE_BIAS_SELECT = 1, /* select on logits + expert_bias, gate on the logits */
  MOE_ROUTE_GUMBEL = 2       /* select and gate on (logits - log(-log u)) / tau */
} moe_route_mode;

/* Bits of the device status word (moe_device_status). */
#define MOE_DEVFAULT_BAD_EXPERT_INDEX 0x1 /* a top-k index outside [0, E) reached dispatch   */
#define MOE_DEVFAULT_PIPELINE_TIMEOUT 0x2 /* a GEMM pipeline wait exceeded its bound          */
#define MOE_DEVFAULT_BAD_TILE 0x4         /* the grouped GEMM met an inconsistent tile list   */
#define MOE_DEVFAULT_FP16_RANGE 0x8       /* a value stored in fp16 (H or a slot row on the fp16
                                             down path or the quantized path, or a weight
                                             re-encoded by moe_pack_f16) was past +-65504 (or
                                             not finite) and was clamped: that output is not
                                             exact; use the bf16 down path for such data   */

/* Element type of the slot-ordered expert outputs y_slot (written by moe_grouped_ffn, read by
 * moe_combine). */
typedef enum {
  MOE_Y_F16 = 0, /* fp16 rows: the fp16 down path (W_down_f16 given) and quantized experts */
  MOE_Y_F32 = 1  /* fp32 rows: the bf16 down path (W_down_f16 NULL) */
} moe_y_type;

typedef struct {
  int32_t T;                 /* tokens */
  int32_t d;                 /* hidden size */
  int32_t E;                 /* routed experts */
  int32_t top_k;             /* experts per token */
  int32_t d_ff;              /* expert intermediate size */
  int32_t n_shared;          /* always-on shared experts (0..4) */
  int32_t mode;              /* moe_route_mode */
  float tau;                 /* Gumbel temperature (> 0); ignored otherwise */
  float capacity_factor;     /* <= 0: no capacity limit; else C = ceil(cf * T * top_k / E) */
  int32_t capacity_override; /* > 0: use this capacity C instead of the factor */
  /* Group-limited (two-level) routing, "大模型MoE稀疏激活原理与工程实践" (routing outlook: first pick
   * one of 8 groups, then 2 experts inside it): experts form n_groups consecutive groups of
   * E / n_groups; a group scores its largest selection score; the topk_groups best groups (ties to
   * the lower group index) are kept and top-k picks among their experts. n_groups = 0: off.
   * Requires E % n_groups == 0, n_groups <= 64, 1 <= topk_groups <= n_groups and
   * top_k <= topk_groups * E / n_groups. */
  int32_t n_groups;
  int32_t topk_groups;
  /* Level-2 capacity protection, "参数规模与稀疏激活的真相拆解" §3.2 专家容量 (overflow tokens are
   * not dropped; a fallback router picks the next-best expert that is not full). 1: after the
   * Level-1 dispatch, the dropped slots, in slot order, each take the best-scoring expert that
   * still has room and that their token does not already use (ties to the lower index); a slot
   * with no such expert stays dropped. The re-routed experts replace the dropped ones in topk_idx
   * and a re-routed token's gates become the softmax over its final experts. 0: Level 1 only.
   * Needs a capacity limit to have an effect; not supported together with n_groups > 0. */
  int32_t overflow_reroute;
  /* Expert weight format: 0 = bf16 (moe_weights.W_gate/W_up/W_down and the shared ones); 4 or
   * 8 = weight-only group-wise quantized experts (moe_weights.quant, written by
   * moe_quantize_weights), "大模型MoE稀疏激活原理与工程实践" §4.2 量化与混合精度 (expert weights to
   * INT4, one scale and zero-point per 128 weights; the router stays in higher precision).
   * Quantized experts need d and d_ff multiples of 128. Activations stay bf16/fp16 and every
   * product accumulates in fp32; the path streams each touched expert's codes once and is
   * built for decode-sized batches (a few rows per expert), where the layer is bound by weight
   * bytes. */
  int32_t weight_bits;
} moe_config;

/* One group-wise quantized weight matrix set: n_mat matrices of K x N (K = input dimension).
 * For every matrix m, group g (input rows [128 g, 128 g + 128)) and output column n:
 *   scale[(m * K/128 + g) * N + n]  fp16, zero[(m * K/128 + g) * N + n]  uint8,
 *   code q in [0, 2^bits - 1], weight = (q - zero) * scale.
 * Codes are stored in the order the tensor-core fragments consume them: 16-column tiles
 * nt = n / 16, and inside a tile 16-row steps st = k / 16 for 32 lanes. With r = n % 16,
 * kk = k % 16: lane = (r % 8) * 4 + (kk % 8) / 2 and the element's slot in the lane's step is
 *   j = (kk % 2) + 2 * (r / 8) + 4 * (kk / 8)           (j = 0..7).
 *   8-bit: byte ((m * N/16 + nt) * K/32 + st / 2) * 512 + lane * 16 + (st % 2) * 8 + j;
 *   4-bit: 32-bit word at byte ((m * N/16 + nt) * K/64 + st / 4) * 512 + lane * 16 + (st % 4) * 4,
 *          nibble at bit 16 * (j % 2) + 4 * (j / 2).
 * Total code bytes: n_mat * K * N * bits / 8. */
typedef struct {
  const uint8_t* q;
  const uint16_t* scale;
  const uint8_t* zero;
} moe_qmatrix;

typedef struct {
  moe_qmatrix gate, up, down;          /* routed experts: [E, d, d_ff], [E, d, d_ff], [E, d_ff, d] */
  moe_qmatrix sh_gate, sh_up, sh_down; /* shared experts (n_shared > 0): [S, ...] likewise */
} moe_qweights;

typedef struct {
  const uint16_t* W_g;        /* [d, E] bf16 */
  const float* expert_bias;   /* [E] fp32; required for BIAS_SELECT, ignored otherwise */
  const uint16_t* W_gate;     /* [E, d, d_ff] bf16 */
  const uint16_t* W_up;       /* [E, d, d_ff] bf16 */
  const uint16_t* W_down;     /* [E, d_ff, d] bf16 */
  const uint16_t* Wsh_gate;   /* [S, d, d_ff] bf16, NULL when n_shared == 0 */
  const uint16_t* Wsh_up;     /* [S, d, d_ff] bf16 */
  const uint16_t* Wsh_down;   /* [S, d_ff, d] bf16 */
  /* Optional fp16 re-encodings of W_down / Wsh_down written once by moe_pack_f16. When given,
   * the down GEMM runs fp16 x fp16 and carries the SwiGLU activations H and the gate-scaled
   * expert outputs in fp16 (11-bit significand) instead of bf16 H (8-bit) and fp32 outputs,
   * which keeps the layer output within bf16 rounding of the exact result and halves the
   * combine's reads. fp16's range ends at 65504: a value past it is clamped and reported as
   * MOE_DEVFAULT_FP16_RANGE. NULL selects the bf16 down path (no packed copy needed), whose H
   * and outputs have fp32's range: choose it when activations may reach that magnitude (for
   * instance outlier features of a trained model), or after that fault was reported. */
  const uint16_t* W_down_f16;   /* [E, d_ff, d] fp16 or NULL */
  const uint16_t* Wsh_down_f16; /* [S, d_ff, d] fp16 or NULL (required when W_down_f16 is set
                                 * and n_shared > 0) */
  /* Quantized experts, used instead of the bf16 ones when moe_config.weight_bits is 4 or 8
   * (the bf16 expert pointers may then be NULL). */
  const moe_qweights* quant;
  /* Optional W_g transposed, [E, d] bf16, written once by moe_prepare_router (16-byte aligned).
   * NULL: every call transposes W_g into the workspace first (one extra kernel per call). */
  const uint16_t* W_g_t;
} moe_weights;

/* Optional copies of the routing results written by moe_layer_forward (any member may be
 * NULL; each non-NULL member receives the same content the stand-alone entry point writes). */
typedef struct {
  int32_t* topk_idx;   /* [T, k] */
  float* topk_w;       /* [T, k] */
  int32_t* counts;     /* [E] */
  int32_t* offsets;    /* [E + 1] */
  int32_t* perm_slot;  /* [T * k] */
  int32_t* slot_pos;   /* [T * k] */
} moe_route_out;

/* Bytes of workspace every entry point below needs for this config (an upper bound that is
 * the same for all of them; 512 for an empty batch, T = 0, which only moe_workspace_init and
 * moe_device_status use). Host only; no CUDA call. */
moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Clears the device status word and the counter block at the start of ws (a 512-byte
 * cudaMemsetAsync on stream). Call once after allocating a workspace; moe_device_status clears
 * the status word again after reading it. The counters in that block are left zero by every
 * call that completes; every other workspace buffer is written before it is read within a
 * call. */
moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/* One-time weight preparation for the router: W_g_t[e, j] = W_g[j, e] (W_g [d, E] bf16 ->
 * W_g_t [E, d] bf16), each expert's router weights contiguous. The router's tensor-core GEMM
 * reads it as its operand and the exact dot products of near-tie tokens read it row by row.
 * Requires 1 <= E <= 256 and d a multiple of 64 (else MOE_ERR_UNSUPPORTED); W_g_t 16-byte
 * aligned. Asynchronous on stream. */
moe_status moe_prepare_router(int32_t d, int32_t E, const uint16_t* W_g, uint16_t* W_g_t,
                              moe_stream_t stream);

/* Steps 1-4. Router: logits in fp32 (per-K-slice partial sums pass through the workspace; the
 * full logits exist only in the selection kernel's registers), selection score, top-k, gates.
 *   x [T, d] bf16, W_g [d, E] bf16, W_g_t [E, d] bf16 from moe_prepare_router (NULL: W_g is
 *   transposed into the workspace by this call), expert_bias [E] fp32 (BIAS_SELECT; else may be
 *   NULL), gumbel_u [T, E] fp32 (GUMBEL; else may be NULL).
 *   Writes topk_idx [T, k] int32 (descending score, ties to the lower index) and
 *   topk_w [T, k] fp32 (gates, summing to 1 per token). */
moe_status moe_route(const moe_config* cfg, const uint16_t* x, const uint16_t* W_g,
                     const uint16_t* W_g_t, const float* expert_bias, const float* gumbel_u,
                     int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                     moe_stream_t stream);

/* Step 5. Dispatch ("参数规模与稀疏激活的真相拆解", §3.2 for the capacity rule).
 *   topk_idx [T, k] int32 in [0, E) (an index outside it sets MOE_DEVFAULT_BAD_EXPERT_INDEX and
 *   that slot is dropped). Slot index = t * k + j.
 *   Writes counts [E] (slots per expert before the capacity limit), offsets [E + 1]
 *   (exclusive scan of min(counts, C); offsets[E] = kept slots N), perm_slot [T * k]
 *   (position -> slot, tokens ascending inside each expert's segment, -1 at positions >= N)
 *   and slot_pos [T * k] (slot -> position, -1 for a dropped slot). Bit-exact and
 *   deterministic. */
moe_status moe_permute(const moe_config* cfg, const int32_t* topk_idx, int32_t* counts,
                       int32_t* offsets, int32_t* perm_slot, int32_t* slot_pos, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/* Level-2 overflow re-route (cfg->overflow_reroute = 1; see moe_config). Must follow moe_route and
 * moe_permute on the same workspace and config: it reads the selection scores that moe_route kept
 * in the workspace, and the Level-1 counts [E] and slot_pos [T * k] that moe_permute wrote.
 *   x [T, d] bf16, W_g_t and expert_bias / gumbel_u as given to moe_route (the exact
 *   re-ordering of experts whose tensor-core scores are too close to call recomputes their
 *   logits; with W_g_t NULL it reads the transposed copy moe_route left in the workspace).
 *   topk_idx [T, k] is updated in place (dropped slots get their new expert), topk_w [T, k] is
 *   rewritten for the re-routed tokens. Run moe_permute again on the updated topk_idx for the
 *   final dispatch. Returns MOE_ERR_INVALID_ARG when cfg->overflow_reroute is 0, and does nothing
 *   when the config has no capacity limit. The proposal rounds run as one cooperative kernel whose
 *   grid barriers wait at most 2 s each (MOE_DEVFAULT_PIPELINE_TIMEOUT on expiry). */
moe_status moe_overflow_reroute(const moe_config* cfg, const uint16_t* x, const uint16_t* W_g_t,
                                const float* expert_bias, const float* gumbel_u,
                                int32_t* topk_idx, float* topk_w, const int32_t* counts,
                                const int32_t* slot_pos, void* ws, size_t ws_bytes,
                                moe_stream_t stream);

/* Largest T * top_k that moe_permute_noalloc accepts (its scratch is a fixed-size array). */
#define MOE_NOALLOC_MAX_SLOTS 262144

/* Dispatch (the same computation and outputs as moe_permute) for callers that cannot allocate
 * device memory at all: a plugin handed only its input and output buffers by a host application
 * that owns every allocation, or a latency-critical loop where cudaMalloc/cudaFree (which may
 * synchronise the device) are not allowed. No counterpart in the source pages: this is a
 * deployment convenience, not a step of the method.
 *   Takes no workspace and allocates nothing (no cudaMalloc, cudaFree or allocating library
 *   call). Its scratch (per-block expert histograms and their running sums, 512 KB) is a
 *   file-scope static __device__ array that every GPU loading this library holds until the
 *   process exits. Each call made outside stream capture looks up that array's device address
 *   (cudaGetSymbolAddress) with the current device, so a device reset in between is harmless; a
 *   call made while the stream is capturing uses the address found by the last call outside
 *   capture on that device. So make one call outside capture before capturing (and again after
 *   any device reset). All calls share the one array, so calls whose executions overlap on the
 *   GPU (different streams, or several host threads) race and must be serialised by the
 *   caller.
 *   fault_bits: optional device int32 the call clears and then ORs MOE_DEVFAULT_* bits into
 *   (NULL: faults are not reported; a bad index still only drops its slot).
 *   Returns MOE_ERR_UNSUPPORTED when T * top_k > MOE_NOALLOC_MAX_SLOTS (or the config is
 *   otherwise unsupported); nothing is enqueued then. */
moe_status moe_permute_noalloc(const moe_config* cfg, const int32_t* topk_idx, int32_t* counts,
                               int32_t* offsets, int32_t* perm_slot, int32_t* slot_pos,
                               int32_t* fault_bits, moe_stream_t stream);

/* Steps 6-9. Gathers x rows into expert order, runs the gate/up grouped GEMM with the fused
 * SiLU*up epilogue and the down grouped GEMM with the fused gate-scale + unpermute epilogue on
 * the tensor cores, and the shared experts over all T tokens.
 *   perm_slot, offsets as written by moe_permute; topk_w [T, k] (NULL: every gate is 1).
 *   Shared weights may be NULL when cfg->n_shared == 0. W_down_f16 / Wsh_down_f16: optional
 *   fp16 re-encodings from moe_pack_f16 (see moe_weights); NULL selects the bf16 down path.
 *   Writes y_slot [T * k + S * T, d]: row t*k + j = gate[t,j] * y(t,j) for every kept slot
 *   (rows of dropped slots are not written); row T*k + s*T + t = z_s[t]. The rows are fp16
 *   (MOE_Y_F16, round to nearest, saturating at +-65504 with MOE_DEVFAULT_FP16_RANGE recorded)
 *   on the fp16 down path and fp32 (MOE_Y_F32) on the bf16 down path. fp16 keeps 11
 *   significant bits per term, so the fixed-order sum in moe_combine stays within bf16
 *   rounding of the exact layer output. */
moe_status moe_grouped_ffn(const moe_config* cfg, const uint16_t* x, const int32_t* perm_slot,
                           const int32_t* offsets, const float* topk_w, const uint16_t* W_gate,
                           const uint16_t* W_up, const uint16_t* W_down,
                           const uint16_t* Wsh_gate, const uint16_t* Wsh_up,
                           const uint16_t* Wsh_down, const uint16_t* W_down_f16,
                           const uint16_t* Wsh_down_f16, void* y_slot, void* ws,
                           size_t ws_bytes, moe_stream_t stream);

/* Step 10. out[t] = sum_{j=0..k-1, slot_pos[t*k+j] >= 0} y_slot[t*k+j]
 *                   + sum_{s=0..S-1} y_slot[T*k + s*T + t],
 * summed in fp32 in exactly that order and rounded once to bf16. y_slot holds rows of y_type
 * (moe_y_type, as moe_grouped_ffn wrote them: MOE_Y_F16 or MOE_Y_F32; anything else returns
 * MOE_ERR_INVALID_ARG), out [T, d] bf16. */
moe_status moe_combine(const moe_config* cfg, const void* y_slot, int32_t y_type,
                       const int32_t* slot_pos, uint16_t* out, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* One-time weight preparation (not part of the layer's per-call work): dst[i] = src[i]
 * re-encoded from bf16 to fp16, round to nearest even, saturating at +-65504. Exact for every
 * bf16 value whose magnitude lies in [2^-14, 65504]; smaller magnitudes become fp16 subnormals
 * (absolute error <= 2^-25). n elements; src and dst device pointers, 16-byte aligned.
 * fault_bits: optional device int32 into which the call ORs MOE_DEVFAULT_FP16_RANGE when a
 * weight had to be clamped (|w| >= 65536 or not finite); the caller clears it beforehand.
 * Weights like that need the bf16 down path. */
moe_status moe_pack_f16(const uint16_t* src_bf16, uint16_t* dst_f16, size_t n,
                        int32_t* fault_bits, moe_stream_t stream);

/* One-time weight preparation: group-wise quantization of n_mat bf16 matrices W [n_mat, K, N]
 * (row-major, K = input dimension, K % 128 == 0, N % 32 == 0) to bits = 4 or 8, in the layout
 * of moe_qmatrix. For each group of 128 weights w along K of one column: s = fp16((max - min) /
 * (2^bits - 1)) (a zero or non-finite s becomes fp16(max |w|), or 1 for an all-zero group),
 * z = clamp(rint(-min / s), 0, 2^bits - 1), q = clamp(rint(w / s) + z, 0, 2^bits - 1); every
 * division in float64, rint to nearest even. q_out needs n_mat*K*N*bits/8 bytes, scale_out and
 * zero_out n_mat*K/128*N entries each. Asynchronous on stream. */
moe_status moe_quantize_weights(int32_t bits, int32_t n_mat, int32_t K, int32_t N,
                                const uint16_t* W, uint8_t* q_out, uint16_t* scale_out,
                                uint8_t* zero_out, moe_stream_t stream);

/* Steps 7-9 with quantized experts (cfg->weight_bits = 4 or 8): the same contract as
 * moe_grouped_ffn (x, perm_slot, offsets, topk_w, fp16 y_slot rows [T*k + S*T, d]) with the
 * expert weights taken from qw. */
moe_status moe_grouped_ffn_quantized(const moe_config* cfg, const uint16_t* x,
                                     const int32_t* perm_slot, const int32_t* offsets,
                                     const float* topk_w, const moe_qweights* qw,
                                     uint16_t* y_slot, void* ws, size_t ws_bytes,
                                     moe_stream_t stream);

/* Steps 1-10 on device buffers: route -> permute -> grouped FFN -> combine, all enqueued on
 * stream with no host synchronisation. gumbel_u is required for GUMBEL. route_out may be NULL.
 * With cfg->overflow_reroute the dispatch is Level 1, the re-route, then the final dispatch;
 * route_out then holds the final experts, gates and dispatch. */
moe_status moe_layer_forward(const moe_config* cfg, const moe_weights* w, const uint16_t* x,
                             const float* gumbel_u, uint16_t* out, moe_route_out* route_out,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* The same layer with the per-call tensors in HOST memory (pinned memory recommended):
 * copies x_host [T, d] (and gumbel_u_host [T, E] for GUMBEL) to staging buffers inside ws,
 * runs moe_layer_forward, and copies out back to out_host [T, d], all enqueued on stream.
 * Weights stay on the device. The caller must synchronise the stream before reading out_host. */
moe_status moe_layer_forward_host(const moe_config* cfg, const moe_weights* w,
                                  const uint16_t* x_host, const float* gumbel_u_host,
                                  uint16_t* out_host, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* moe_layer_forward that also records CUDA events (cudaEvent_t handles created by the caller)
 * on stream at the boundaries of its phases, for per-kernel timing:
 *   events[0] before the router, [1] after the router, [2] after dispatch (histogram, scan,
 *   scatter), [3] after the tile list + row gather, [4] after the gate/up GEMM, [5] after the
 *   down GEMM, [6] after the combine.  n_events must be 7. Same results as moe_layer_forward. */
moe_status moe_layer_forward_profiled(const moe_config* cfg, const moe_weights* w,
                                      const uint16_t* x, const float* gumbel_u, uint16_t* out,
                                      moe_route_out* route_out, void* ws, size_t ws_bytes,
                                      moe_stream_t stream, void* const* events, int n_events);

/* Aux-loss-free expert-bias update, the step that follows a forward pass with bias-adjusted
 * selection ("AI架构演进从稀疏MoE到条件记忆的工程实践", gating-network code, its no_grad block):
 *   load[e] = counts[e] (selections of expert e over all top-k picks, before any capacity limit,
 *   as written by moe_permute or moe_layer_forward's route_out), then
 *   expert_bias[e] <- decay * expert_bias[e] - rate * load[e] / (mean(load) + 1e-8),
 * in place on the device (mean and ratio in fp64). The page uses decay 0.99 and rate 0.01.
 * counts [E] int32, expert_bias [E] fp32. Enqueued on stream. */
moe_status moe_bias_update(int32_t E, const int32_t* counts, float* expert_bias, float decay,
                           float rate, moe_stream_t stream);

/* Failure-detection check of this device: runs the library's two kinds of bounded device wait,
 * each against a condition that never comes true, with a wait limit of limit_ns (100 us .. 2 s;
 * the layer's own waits use 2 s). One is the mbarrier wait of the tensor-core pipelines (a
 * barrier no one arrives on), the other the grid barrier of the overflow re-route's proposal
 * rounds (one of its two CTAs skips its arrival). Each must give up after about limit_ns, record
 * MOE_DEVFAULT_PIPELINE_TIMEOUT in the status word of ws and return, leaving nothing in flight
 * and the context usable. expired: device int32[2], set to 1 for each wait that gave up (0 would
 * mean a wait saw its condition come true). ws: a workspace initialised by moe_workspace_init
 * (its first 512 bytes are used). No counterpart in the source pages, whose overflow circuit
 * breaker ("参数规模与稀疏激活的真相拆解", §3.2) is the analogue on the serving side. Read the
 * result with moe_device_status, which then returns MOE_ERR_DEVICE_FAULT with that bit. */
moe_status moe_check_bounded_waits(int64_t limit_ns, int32_t* expired, void* ws, size_t ws_bytes,
                                   moe_stream_t stream);

/* Synchronises stream, reads the device status word of ws into *fault_bits (MOE_DEVFAULT_*),
 * clears it, and returns MOE_ERR_DEVICE_FAULT if any bit was set, MOE_ERR_CUDA if the stream
 * reported an error, else MOE_OK. */
moe_status moe_device_status(void* ws, moe_stream_t stream, int32_t* fault_bits);

/* Static English description of a status code. */
const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
