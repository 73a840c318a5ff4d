// C ABI of the sparse-MoE layer (declarations and argument contracts: include/moe.h).
// Host-side validation, workspace carving and launch sequencing. No device allocation.
#include <cuda_runtime.h>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "internal.h"

namespace moe {

namespace {
constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// ceil(cf * T * k / E) exactly: cf = m * 2^ex with an integer m (24-bit mantissa of the fp32).
long long exact_capacity(float cf, long long TK, int E) {
  int ex = 0;
  const float fr = std::frexp(cf, &ex);          // cf = fr * 2^ex, fr in [0.5, 1)
  const long long m = (long long)std::ldexp(fr, 24);  // exact: fr has a 24-bit mantissa
  const int sh = ex - 24;                         // cf = m * 2^sh
  // value = m * TK * 2^sh / E
  unsigned __int128 num = (unsigned __int128)m * (unsigned long long)TK;
  unsigned __int128 den = (unsigned __int128)E;
  if (sh >= 0) {
    if (sh > 60) return LLONG_MAX;
    num <<= sh;
  } else {
    if (-sh > 100) return 1;
    den <<= -sh;
  }
  const unsigned __int128 q = (num + den - 1) / den;
  if (q > (unsigned __int128)LLONG_MAX) return LLONG_MAX;
  return (long long)q;
}
}  // namespace

Shape make_shape(const moe_config& c) {
  Shape s;
  s.T = c.T;
  s.d = c.d;
  s.E = c.E;
  s.k = c.top_k;
  s.f = c.d_ff;
  s.S = c.n_shared;
  s.mode = c.mode;
  s.G = c.n_groups;
  s.Gk = c.topk_groups;
  s.tau = c.tau;
  s.TK = (long long)c.T * c.top_k;
  s.rows = s.TK + (long long)c.n_shared * c.T;
  long long C = INT_MAX;
  if (c.capacity_override > 0)
    C = c.capacity_override;
  else if (c.capacity_factor > 0.f)
    C = exact_capacity(c.capacity_factor, s.TK, c.E);
  if (C > INT_MAX) C = INT_MAX;
  if (C < 1) C = 1;
  s.C = (int)C;
  s.reroute = c.overflow_reroute != 0 && s.C != INT_MAX;
  s.n_pblk = (int)((s.TK + kPermuteBlock - 1) / kPermuteBlock);
  // Row tiles: 8 rows for quantized experts; 256 rows (CTA-pair GEMMs) when the expert segments
  // are long enough for the pair's M = 256 MMA to pay for its padding (about T*k/E >= 320
  // rows per expert) and the shape fits its 256-column tiles; else 128.
  const bool pairs = c.weight_bits == 0 && c.d_ff % 128 == 0 && c.d % 256 == 0 &&
                     (long long)c.T * c.top_k >= 320LL * c.E;
  s.tile_m = c.weight_bits != 0 ? kQTileM : (pairs ? 2 * kTileM : kTileM);
  s.max_tiles = (int)((s.TK + s.tile_m - 1) / s.tile_m + s.E +
                      (long long)s.S * ((s.T + s.tile_m - 1) / s.tile_m));
  return s;
}

WsLayout ws_layout(const Shape& s) {
  WsLayout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.status = take(sizeof(int));
  L.meta = take(sizeof(Meta));
  L.topk_idx = take(sizeof(int32_t) * s.TK);
  L.topk_w = take(sizeof(float) * s.TK);
  L.counts = take(sizeof(int32_t) * s.E);
  L.offsets = take(sizeof(int32_t) * (s.E + 1));
  L.perm_slot = take(sizeof(int32_t) * s.TK);
  L.slot_pos = take(sizeof(int32_t) * s.TK);
  L.blk_hist = take(sizeof(int32_t) * (size_t)s.n_pblk * s.E);
  L.blk_base = take(sizeof(int32_t) * (size_t)s.n_pblk * s.E);
  L.tiles = take(sizeof(TileEntry) * (size_t)s.max_tiles);
  L.wg_t = take(2ull * s.d * s.E);
  L.rpart = take(4ull * router_splits(s.T, s.d) * s.T * ((s.E + 63) / 64 * 64));
  L.rrec = take(sizeof(int32_t) * (size_t)s.T * kRouterRecInts);
  const bool quant = s.tile_m == kQTileM;
  L.xp = take(quant ? 0 : 2ull * s.TK * s.d);  // the quantized passes read x16 by token
  L.x16 = take(quant ? 2ull * s.T * s.d : 0);
  L.sbx = take(quant ? 4ull * s.T * (s.d / 128) : 0);
  L.tail_acc = take(quant ? 4ull * quant_tail_cap() * 16 * 32 : 0);
  L.tail_ticket = take(quant ? 4ull * 2 * quant_tail_cap() : 0);
  L.h = take(2ull * s.rows * s.f);
  L.y = take(4ull * s.rows * s.d);  // fp32 rows on the bf16 down path, fp16 otherwise
  L.x_stage = take(2ull * s.T * s.d);
  L.u_stage = take(s.mode == MOE_ROUTE_GUMBEL ? 4ull * s.T * s.E : 0);
  L.out_stage = take(2ull * s.T * s.d);
  const bool rr = s.reroute;
  const size_t W = ((size_t)s.T + 31) / 32;
  L.sfull = take(rr ? 4ull * s.T * s.E : 0);
  L.maxl = take(rr ? 4ull * s.T : 0);
  L.pref = take(rr ? (size_t)s.T * ((s.E + 15) / 16 * 16) : 0);
  L.rr_tok = take(rr ? 4ull * 7 * s.T : 0);     // plen, dem, ptr, held, rlen, ext_list, ex_list
  L.rr_exp = take(rr ? 4ull * 3 * s.E : 0);     // room, cut, touched
  L.rr_bits = take(rr ? 4ull * s.E * W : 0);
  L.rr_ctl = take(rr ? 4ull * (2 * 1024 + 2) : 0);  // per-round counters, barrier
  L.total = o;
  return L;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

}  // namespace moe

using namespace moe;

namespace {

moe_status check_cfg(const moe_config* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d < 1 || c->E < 1 || c->top_k < 1 || c->d_ff < 1 || c->n_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->mode < MOE_ROUTE_PLAIN || c->mode > MOE_ROUTE_GUMBEL) return MOE_ERR_INVALID_ARG;
  if (c->mode == MOE_ROUTE_GUMBEL && !(c->tau > 0.f && std::isfinite(c->tau)))
    return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(c->capacity_factor)) return MOE_ERR_INVALID_ARG;
  if (c->E > 256 || c->top_k > 8 || c->top_k > c->E || c->n_shared > 4) return MOE_ERR_UNSUPPORTED;
  if (c->d % 64 != 0 || c->d_ff % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (c->n_groups < 0) return MOE_ERR_INVALID_ARG;
  if (c->n_groups > 0) {
    if (c->n_groups > 64 || c->E % c->n_groups != 0) return MOE_ERR_UNSUPPORTED;
    if (c->topk_groups < 1 || c->topk_groups > c->n_groups) return MOE_ERR_INVALID_ARG;
    if ((long long)c->top_k > (long long)c->topk_groups * (c->E / c->n_groups))
      return MOE_ERR_INVALID_ARG;
  }
  if (c->weight_bits != 0 && c->weight_bits != 4 && c->weight_bits != 8) return MOE_ERR_INVALID_ARG;
  if (c->weight_bits != 0 && (c->d % 128 != 0 || c->d_ff % 128 != 0)) return MOE_ERR_UNSUPPORTED;
  if (c->overflow_reroute != 0 && c->overflow_reroute != 1) return MOE_ERR_INVALID_ARG;
  if (c->overflow_reroute && c->n_groups > 0) return MOE_ERR_UNSUPPORTED;
  const long long rows = (long long)c->T * (c->top_k + c->n_shared);
  if (rows >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status check_ws(const moe_config* c, void* ws, size_t ws_bytes) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % 256) != 0) return MOE_ERR_WORKSPACE;
  if (ws_bytes < ws_layout(make_shape(*c)).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// An empty batch (T = 0) launches no kernel and reads no tensor. The dispatch's per-expert
// outputs are its only non-empty results: every expert receives nothing, so counts [E] and
// offsets [E + 1] are cleared (each only if given).
moe_status clear_dispatch(int E, int32_t* counts, int32_t* offsets, cudaStream_t st) {
  if (counts && cudaMemsetAsync(counts, 0, 4ull * E, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (offsets && cudaMemsetAsync(offsets, 0, 4ull * (E + 1), st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status route_impl(const Shape& s, const WsLayout& L, void* ws, const uint16_t* x,
                      const uint16_t* W_g, const uint16_t* W_g_t, const float* bias,
                      const float* u, int32_t* idx, float* w, cudaStream_t st) {
  RouterScratch rs;
  rs.wg_t = at<uint16_t>(ws, L.wg_t);
  rs.part = at<float>(ws, L.rpart);
  rs.rrec = at<int32_t>(ws, L.rrec);
  Meta* meta = at<Meta>(ws, L.meta);
  rs.rcount = &meta->refine_count;
  rs.sfull = s.reroute ? at<float>(ws, L.sfull) : nullptr;
  rs.maxl = s.reroute ? at<float>(ws, L.maxl) : nullptr;
  return cuda_status(
      launch_router(s, x, W_g, W_g_t, bias, u, idx, w, rs, at<int>(ws, L.status), st));
}

// with_tiles: the FFN follows, so the dispatch also builds its row-tile list
moe_status permute_impl(const Shape& s, const WsLayout& L, void* ws, const int32_t* idx,
                        int32_t* counts, int32_t* offsets, int32_t* perm_slot, int32_t* slot_pos,
                        cudaStream_t st, bool with_tiles = false) {
  Meta* meta = at<Meta>(ws, L.meta);
  return cuda_status(launch_permute(s, idx, counts, offsets, perm_slot, slot_pos,
                                    at<int32_t>(ws, L.blk_hist), at<int32_t>(ws, L.blk_base),
                                    &meta->dispatch_ticket, at<int>(ws, L.status),
                                    with_tiles ? at<TileEntry>(ws, L.tiles) : nullptr,
                                    with_tiles ? meta : nullptr, st));
}

// W_g_t: the prepared transpose given to the router, or nullptr when the router made its own in
// the workspace
moe_status reroute_impl(const Shape& s, const WsLayout& L, void* ws, const uint16_t* x,
                        const uint16_t* W_g_t, const float* bias, const float* u, int32_t* idx,
                        float* w, const int32_t* counts, const int32_t* slot_pos,
                        cudaStream_t st) {
  RerouteArgs a;
  a.x = x;
  a.WgT = W_g_t != nullptr ? W_g_t : at<uint16_t>(ws, L.wg_t);
  a.bias = bias;
  a.u = u;
  a.sfull = at<float>(ws, L.sfull);
  a.maxl = at<float>(ws, L.maxl);
  a.topk_idx = idx;
  a.topk_w = w;
  a.counts = counts;
  a.slot_pos = slot_pos;
  a.pref = at<uint8_t>(ws, L.pref);
  int32_t* tok = at<int32_t>(ws, L.rr_tok);
  a.plen = tok;
  a.dem = tok + s.T;
  a.ptr = tok + 2 * (size_t)s.T;
  a.held = tok + 3 * (size_t)s.T;
  a.rlen = tok + 4 * (size_t)s.T;
  a.ext_list = tok + 5 * (size_t)s.T;
  a.ex_list = tok + 6 * (size_t)s.T;
  a.ex_count = &at<Meta>(ws, L.meta)->reroute_exact;
  int32_t* ex = at<int32_t>(ws, L.rr_exp);
  a.room = ex;
  a.cut = ex + s.E;
  a.touched = ex + 2 * s.E;
  a.bits = at<uint32_t>(ws, L.rr_bits);
  a.rejected = at<int32_t>(ws, L.rr_ctl);
  a.extended = a.rejected + 1024;
  a.ctl = a.rejected + 2048;
  a.rounds_out = &at<Meta>(ws, L.meta)->reroute_rounds;
  a.status = at<int>(ws, L.status);
  a.T = s.T;
  a.d = s.d;
  a.E = s.E;
  a.k = s.k;
  a.mode = s.mode;
  a.C = s.C;
  a.W = (s.T + 31) / 32;
  a.PS = (s.E + 15) / 16 * 16;
  a.tau = s.tau;
  return cuda_status(launch_reroute(a, st));
}

moe_status ffn_impl(const Shape& s, const WsLayout& L, void* ws, const uint16_t* x,
                    const int32_t* perm_slot, const int32_t* offsets, const float* topk_w,
                    const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd,
                    const uint16_t* Wsg, const uint16_t* Wsu, const uint16_t* Wsd,
                    const uint16_t* Wd16, const uint16_t* Wsd16, void* y,
                    cudaStream_t st, bool tiles_built = false, cudaEvent_t ev_gathered = nullptr,
                    cudaEvent_t ev_gate_up = nullptr) {
  cudaError_t e = launch_tiles_and_gather(s, x, perm_slot, offsets, at<uint16_t>(ws, L.xp),
                                          at<TileEntry>(ws, L.tiles), at<Meta>(ws, L.meta),
                                          tiles_built, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (ev_gathered != nullptr && cudaEventRecord(ev_gathered, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  FfnPtrs p;
  p.x = x;
  p.xp = at<uint16_t>(ws, L.xp);
  p.perm_slot = perm_slot;
  p.topk_w = topk_w;
  p.W_gate = Wg;
  p.W_up = Wu;
  p.W_down = Wd;
  p.Wsh_gate = Wsg;
  p.Wsh_up = Wsu;
  p.Wsh_down = Wsd;
  p.W_down_f16 = Wd16;
  p.Wsh_down_f16 = Wsd16;
  p.h = at<uint16_t>(ws, L.h);
  p.y = y;
  p.tiles = at<TileEntry>(ws, L.tiles);
  p.meta = at<Meta>(ws, L.meta);
  p.status = at<int>(ws, L.status);
  return cuda_status(launch_grouped_ffn(s, p, st, ev_gate_up));
}

bool qmat_ok(const moe_qmatrix& m) { return m.q && m.scale && m.zero; }

bool qweights_ok(const moe_config* c, const moe_qweights* q) {
  if (q == nullptr || !qmat_ok(q->gate) || !qmat_ok(q->up) || !qmat_ok(q->down)) return false;
  if (c->n_shared > 0 && (!qmat_ok(q->sh_gate) || !qmat_ok(q->sh_up) || !qmat_ok(q->sh_down)))
    return false;
  return true;
}

moe_status qffn_impl(const Shape& s, int bits, const WsLayout& L, void* ws, const uint16_t* x,
                     const int32_t* perm_slot, const int32_t* offsets, const float* topk_w,
                     const moe_qweights* qw, void* y, cudaStream_t st,
                     bool tiles_built = false, cudaEvent_t ev_gathered = nullptr,
                     cudaEvent_t ev_gate_up = nullptr) {
  if (!tiles_built &&
      launch_tiles(s, offsets, at<TileEntry>(ws, L.tiles), at<Meta>(ws, L.meta), st) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  QFfnPtrs p;
  p.x = x;
  p.x16 = at<uint16_t>(ws, L.x16);
  p.sbx = at<float>(ws, L.sbx);
  p.tail_acc = at<float>(ws, L.tail_acc);
  p.tail_ticket = at<int>(ws, L.tail_ticket);
  p.tail_cap = quant_tail_cap();
  if (launch_quant_act(s, p, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (ev_gathered != nullptr && cudaEventRecord(ev_gathered, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  p.h = at<uint16_t>(ws, L.h);
  p.y = static_cast<uint16_t*>(y);
  p.perm_slot = perm_slot;
  p.topk_w = topk_w;
  p.tiles = at<TileEntry>(ws, L.tiles);
  p.meta = at<Meta>(ws, L.meta);
  p.qw = qw;
  p.status = at<int>(ws, L.status);
  return cuda_status(launch_quant_ffn(s, bits, p, st, ev_gate_up));
}

moe_status layer_impl(const moe_config* cfg, const moe_weights* w, const uint16_t* x,
                      const float* gumbel_u, uint16_t* out, moe_route_out* ro, void* ws,
                      size_t ws_bytes, cudaStream_t st, cudaEvent_t const* ev) {
  moe_status r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (cfg->T == 0) {
    // the phase events are still recorded, back to back, so that every elapsed time is defined
    for (int i = 0; ev != nullptr && i < 7; ++i)
      if (cudaEventRecord(ev[i], st) != cudaSuccess) return MOE_ERR_CUDA;
    return ro ? clear_dispatch(cfg->E, ro->counts, ro->offsets, st) : MOE_OK;
  }
  if (!w || !x || !out || !w->W_g) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(w->W_g_t) % 16 != 0) return MOE_ERR_INVALID_ARG;
  const bool quant = cfg->weight_bits != 0;
  if (quant) {
    if (!qweights_ok(cfg, w->quant)) return MOE_ERR_INVALID_ARG;
  } else {
    if (!w->W_gate || !w->W_up || !w->W_down) return MOE_ERR_INVALID_ARG;
    if (cfg->n_shared > 0 && (!w->Wsh_gate || !w->Wsh_up || !w->Wsh_down))
      return MOE_ERR_INVALID_ARG;
    if (w->W_down_f16 && cfg->n_shared > 0 && !w->Wsh_down_f16) return MOE_ERR_INVALID_ARG;
  }
  if (cfg->mode == MOE_ROUTE_BIAS_SELECT && !w->expert_bias) return MOE_ERR_INVALID_ARG;
  if (cfg->mode == MOE_ROUTE_GUMBEL && !gumbel_u) return MOE_ERR_INVALID_ARG;
  if ((r = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return r;
  const Shape s = make_shape(*cfg);
  const WsLayout L = ws_layout(s);
  auto mark = [&](int i) { return ev == nullptr || cudaEventRecord(ev[i], st) == cudaSuccess; };
  int32_t* idx = (ro && ro->topk_idx) ? ro->topk_idx : at<int32_t>(ws, L.topk_idx);
  float* gw = (ro && ro->topk_w) ? ro->topk_w : at<float>(ws, L.topk_w);
  int32_t* counts = (ro && ro->counts) ? ro->counts : at<int32_t>(ws, L.counts);
  int32_t* offsets = (ro && ro->offsets) ? ro->offsets : at<int32_t>(ws, L.offsets);
  int32_t* perm_slot = (ro && ro->perm_slot) ? ro->perm_slot : at<int32_t>(ws, L.perm_slot);
  int32_t* slot_pos = (ro && ro->slot_pos) ? ro->slot_pos : at<int32_t>(ws, L.slot_pos);
  if (!mark(0)) return MOE_ERR_CUDA;
  if ((r = route_impl(s, L, ws, x, w->W_g, w->W_g_t, w->expert_bias, gumbel_u, idx, gw, st)) !=
      MOE_OK)
    return r;
  if (!mark(1)) return MOE_ERR_CUDA;
  // the last dispatch also builds the FFN's row-tile list
  if ((r = permute_impl(s, L, ws, idx, counts, offsets, perm_slot, slot_pos, st,
                        !s.reroute)) != MOE_OK)
    return r;
  if (s.reroute) {
    // Level 2: dropped slots move to the best expert with room, then the final dispatch
    if ((r = reroute_impl(s, L, ws, x, w->W_g_t, w->expert_bias, gumbel_u, idx, gw, counts,
                          slot_pos, st)) != MOE_OK)
      return r;
    if ((r = permute_impl(s, L, ws, idx, counts, offsets, perm_slot, slot_pos, st, true)) !=
        MOE_OK)
      return r;
  }
  if (!mark(2)) return MOE_ERR_CUDA;
  void* y = at<void>(ws, L.y);
  // slot rows in fp32 on the bf16 down path (full range), else fp16
  const bool y_f32 = !quant && w->W_down_f16 == nullptr;
  if (quant)
    r = qffn_impl(s, cfg->weight_bits, L, ws, x, perm_slot, offsets, gw, w->quant, y, st, true,
                  ev ? ev[3] : nullptr, ev ? ev[4] : nullptr);
  else
    r = ffn_impl(s, L, ws, x, perm_slot, offsets, gw, w->W_gate, w->W_up, w->W_down,
                 w->Wsh_gate, w->Wsh_up, w->Wsh_down, w->W_down_f16, w->Wsh_down_f16, y, st,
                 true, ev ? ev[3] : nullptr, ev ? ev[4] : nullptr);
  if (r != MOE_OK) return r;
  if (!mark(5)) return MOE_ERR_CUDA;
  if ((r = cuda_status(launch_combine(s, y, y_f32, slot_pos, out, st))) != MOE_OK) return r;
  return mark(6) ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

extern "C" {

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  moe_status r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  // an empty batch needs only the status word and the meta block that moe_workspace_init clears
  *bytes = cfg->T == 0 ? 512 : ws_layout(make_shape(*cfg)).total;
  return MOE_OK;
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
  // the status word (first 256 bytes) and the meta block with the router's near-tie list
  // counters (next 256 bytes)
  if (ws == nullptr || ws_bytes < 512 || (reinterpret_cast<uintptr_t>(ws) % 256) != 0)
    return MOE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, 512, (cudaStream_t)stream));
}

moe_status moe_prepare_router(int32_t d, int32_t E, const uint16_t* W_g, uint16_t* W_g_t,
                              moe_stream_t stream) {
  if (d < 1 || E < 1 || !W_g || !W_g_t) return MOE_ERR_INVALID_ARG;
  if (E > 256 || d % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(W_g_t) % 16 != 0) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_router_transpose(d, E, W_g, W_g_t, (cudaStream_t)stream));
}

moe_status moe_route(const moe_config* cfg, const uint16_t* x, const uint16_t* W_g,
                     const uint16_t* W_g_t, const float* expert_bias, const float* gumbel_u,
                     int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                     moe_stream_t stream) {
  moe_status r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !W_g || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(W_g_t) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (cfg->mode == MOE_ROUTE_BIAS_SELECT && !expert_bias) return MOE_ERR_INVALID_ARG;
  if (cfg->mode == MOE_ROUTE_GUMBEL && !gumbel_u) return MOE_ERR_INVALID_ARG;
  if ((r = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return r;
  const Shape s = make_shape(*cfg);
  const WsLayout L = ws_layout(s);
  return route_impl(s, L, ws, x, W_g, W_g_t, expert_bias, gumbel_u, topk_idx, topk_w,
                    (cudaStream_t)stream);
}

moe_status moe_permute(const moe_config* cfg, const int32_t* topk_idx, int32_t* counts,
                       int32_t* offsets, int32_t* perm_slot, int32_t* slot_pos, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
  moe_status r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (cfg->T == 0) {
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    return clear_dispatch(cfg->E, counts, offsets, (cudaStream_t)stream);
  }
  if (!topk_idx || !counts || !offsets || !perm_slot || !slot_pos) return MOE_ERR_INVALID_ARG;
  if ((r = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return r;
  const Shape s = make_shape(*cfg);
  const WsLayout L = ws_layout(s);
  return permute_impl(s, L, ws, topk_idx, counts, offsets, perm_slot, slot_pos,
                      (cudaStream_t)stream);
}

moe_status moe_overflow_reroute(const moe_config* cfg, const uint16_t* x, const uint16_t* W_g_t,
                                const float* expert_bias, const float* gumbel_u,
                                int32_t* topk_idx, float* topk_w, const int32_t* counts,
                                const int32_t* slot_pos, void* ws, size_t ws_bytes,
                                moe_stream_t stream) {
  moe_status r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (cfg->overflow_reroute == 0) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !topk_idx || !topk_w || !counts || !slot_pos) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(W_g_t) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (cfg->mode == MOE_ROUTE_BIAS_SELECT && !expert_bias) return MOE_ERR_INVALID_ARG;
  if (cfg->mode == MOE_ROUTE_GUMBEL && !gumbel_u) return MOE_ERR_INVALID_ARG;
  if ((r = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return r;
  const Shape s = make_shape(*cfg);
  if (!s.reroute) return MOE_OK;  // no capacity limit: nothing can overflow
  const WsLayout L = ws_layout(s);
  return reroute_impl(s, L, ws, x, W_g_t, expert_bias, gumbel_u, topk_idx, topk_w, counts,
                      slot_pos, (cudaStream_t)stream);
}

moe_status moe_quantize_weights(int32_t bits, int32_t n_mat, int32_t K, int32_t N,
                                const uint16_t* W, uint8_t* q_out, uint16_t* scale_out,
                                uint8_t* zero_out, moe_stream_t stream) {
  if (bits != 4 && bits != 8) return MOE_ERR_INVALID_ARG;
  if (n_mat < 1 || K < 1 || N < 1 || !W || !q_out || !scale_out || !zero_out)
    return MOE_ERR_INVALID_ARG;
  if (K % 128 != 0 || N % 32 != 0) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_quantize(bits, n_mat, K, N, W, q_out, scale_out, zero_out,
                                     (cudaStream_t)stream));
}

moe_status moe_grouped_ffn_quantized(const moe_config* cfg, const uint16_t* x,
                                     const int32_t* perm_slot, const int32_t* offsets,
                                     const float* topk_w, const moe_qweights* qw,
                                     uint16_t* y_slot, void* ws, size_t ws_bytes,
                                     moe_stream_t stream) {
  moe_status r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (cfg->weight_bits == 0) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !perm_slot || !offsets || !y_slot || !qweights_ok(cfg, qw)) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if ((r = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return r;
  const Shape s = make_shape(*cfg);
  const WsLayout L = ws_layout(s);
  return qffn_impl(s, cfg->weight_bits, L, ws, x, perm_slot, offsets, topk_w, qw, y_slot,
                   (cudaStream_t)stream);
}

moe_status moe_permute_noalloc(const moe_config* cfg, const int32_t* topk_idx, int32_t* counts,
                               int32_t* offsets, int32_t* perm_slot, int32_t* slot_pos,
                               int32_t* fault_bits, moe_stream_t stream) {
  moe_status r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (cfg->T == 0) {
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (fault_bits && cudaMemsetAsync(fault_bits, 0, 4, (cudaStream_t)stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    return clear_dispatch(cfg->E, counts, offsets, (cudaStream_t)stream);
  }
  if (!topk_idx || !counts || !offsets || !perm_slot || !slot_pos) return MOE_ERR_INVALID_ARG;
  const Shape s = make_shape(*cfg);
  if (s.TK > MOE_NOALLOC_MAX_SLOTS) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_permute_noalloc(s, topk_idx, counts, offsets, perm_slot, slot_pos,
                                            fault_bits, (cudaStream_t)stream));
}

moe_status moe_grouped_ffn(const moe_config* cfg, const uint16_t* x, const int32_t* perm_slot,
                           const int32_t* offsets, const float* topk_w, const uint16_t* W_gate,
                           const uint16_t* W_up, const uint16_t* W_down,
                           const uint16_t* Wsh_gate, const uint16_t* Wsh_up,
                           const uint16_t* Wsh_down, const uint16_t* W_down_f16,
                           const uint16_t* Wsh_down_f16, void* y_slot, void* ws,
                           size_t ws_bytes, moe_stream_t stream) {
  moe_status r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (cfg->weight_bits != 0) return MOE_ERR_INVALID_ARG;  // see moe_grouped_ffn_quantized
  if (cfg->T == 0) return MOE_OK;
  if (!x || !perm_slot || !offsets || !W_gate || !W_up || !W_down || !y_slot)
    return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (cfg->n_shared > 0 && (!Wsh_gate || !Wsh_up || !Wsh_down)) return MOE_ERR_INVALID_ARG;
  if (W_down_f16 && cfg->n_shared > 0 && !Wsh_down_f16) return MOE_ERR_INVALID_ARG;
  if ((r = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return r;
  const Shape s = make_shape(*cfg);
  const WsLayout L = ws_layout(s);
  return ffn_impl(s, L, ws, x, perm_slot, offsets, topk_w, W_gate, W_up, W_down, Wsh_gate,
                  Wsh_up, Wsh_down, W_down_f16, Wsh_down_f16, y_slot, (cudaStream_t)stream);
}

moe_status moe_combine(const moe_config* cfg, const void* y_slot, int32_t y_type,
                       const int32_t* slot_pos, uint16_t* out, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  moe_status r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (y_type != MOE_Y_F16 && y_type != MOE_Y_F32) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (!y_slot || !slot_pos || !out) return MOE_ERR_INVALID_ARG;
  if ((r = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return r;
  const Shape s = make_shape(*cfg);
  return cuda_status(
      launch_combine(s, y_slot, y_type == MOE_Y_F32, slot_pos, out, (cudaStream_t)stream));
}

moe_status moe_layer_forward(const moe_config* cfg, const moe_weights* w, const uint16_t* x,
                             const float* gumbel_u, uint16_t* out, moe_route_out* ro, void* ws,
                             size_t ws_bytes, moe_stream_t stream) {
  return layer_impl(cfg, w, x, gumbel_u, out, ro, ws, ws_bytes, (cudaStream_t)stream, nullptr);
}

moe_status moe_layer_forward_profiled(const moe_config* cfg, const moe_weights* w,
                                      const uint16_t* x, const float* gumbel_u, uint16_t* out,
                                      moe_route_out* ro, void* ws, size_t ws_bytes,
                                      moe_stream_t stream, void* const* events, int n_events) {
  if (events == nullptr || n_events != 7) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 7; ++i)
    if (events[i] == nullptr) return MOE_ERR_INVALID_ARG;
  return layer_impl(cfg, w, x, gumbel_u, out, ro, ws, ws_bytes, (cudaStream_t)stream,
                    reinterpret_cast<cudaEvent_t const*>(events));
}

moe_status moe_layer_forward_host(const moe_config* cfg, const moe_weights* w,
                                  const uint16_t* x_host, const float* gumbel_u_host,
                                  uint16_t* out_host, void* ws, size_t ws_bytes,
                                  moe_stream_t stream) {
  moe_status r = check_cfg(cfg);
  if (r != MOE_OK) return r;
  if (cfg->T == 0) return MOE_OK;
  if (!x_host || !out_host) return MOE_ERR_INVALID_ARG;
  if (cfg->mode == MOE_ROUTE_GUMBEL && !gumbel_u_host) return MOE_ERR_INVALID_ARG;
  if ((r = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return r;
  const Shape s = make_shape(*cfg);
  const WsLayout L = ws_layout(s);
  cudaStream_t st = (cudaStream_t)stream;
  uint16_t* xd = at<uint16_t>(ws, L.x_stage);
  float* ud = cfg->mode == MOE_ROUTE_GUMBEL ? at<float>(ws, L.u_stage) : nullptr;
  uint16_t* od = at<uint16_t>(ws, L.out_stage);
  if (cudaMemcpyAsync(xd, x_host, 2ull * s.T * s.d, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (ud && cudaMemcpyAsync(ud, gumbel_u_host, 4ull * s.T * s.E, cudaMemcpyHostToDevice, st) !=
                cudaSuccess)
    return MOE_ERR_CUDA;
  if ((r = moe_layer_forward(cfg, w, xd, ud, od, nullptr, ws, ws_bytes, stream)) != MOE_OK)
    return r;
  return cuda_status(
      cudaMemcpyAsync(out_host, od, 2ull * s.T * s.d, cudaMemcpyDeviceToHost, st));
}

moe_status moe_pack_f16(const uint16_t* src_bf16, uint16_t* dst_f16, size_t n,
                        int32_t* fault_bits, moe_stream_t stream) {
  if (!src_bf16 || !dst_f16 || n == 0) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src_bf16) | reinterpret_cast<uintptr_t>(dst_f16)) % 16 != 0)
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_pack_f16(src_bf16, dst_f16, n, fault_bits, (cudaStream_t)stream));
}

moe_status moe_bias_update(int32_t E, const int32_t* counts, float* expert_bias, float decay,
                           float rate, moe_stream_t stream) {
  if (E < 1 || !counts || !expert_bias) return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(decay) || !std::isfinite(rate)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_bias_update(E, counts, expert_bias, decay, rate, (cudaStream_t)stream));
}

moe_status moe_check_bounded_waits(int64_t limit_ns, int32_t* expired, void* ws,
                                   size_t ws_bytes, moe_stream_t stream) {
  if (ws == nullptr || ws_bytes < 512 || (reinterpret_cast<uintptr_t>(ws) % 256) != 0)
    return MOE_ERR_WORKSPACE;
  if (expired == nullptr || limit_ns < 100000 || limit_ns > 2000000000) return MOE_ERR_INVALID_ARG;
  Meta* meta = reinterpret_cast<Meta*>(static_cast<char*>(ws) + 256);  // ws_layout's meta block
  return cuda_status(launch_wait_check((uint64_t)limit_ns, static_cast<int*>(ws), expired,
                                       &meta->check_arrive, &meta->check_gen,
                                       (cudaStream_t)stream));
}

moe_status moe_device_status(void* ws, moe_stream_t stream, int32_t* fault_bits) {
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0 && cudaMemset(ws, 0, sizeof(v)) != cudaSuccess) return MOE_ERR_CUDA;
  if (fault_bits) *fault_bits = v;
  return v != 0 ? MOE_ERR_DEVICE_FAULT : MOE_OK;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or option";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA runtime or driver call failed";
    case MOE_ERR_DEVICE_FAULT: return "a kernel recorded a device-side fault";
  }
  return "unknown status";
}

}  // extern "C"
