"""Python binding of libmoe_gb300.so (the C ABI in include/moe.h).

Argument marshalling only: every function forwards torch tensors' device pointers and the
current CUDA stream to the entry point of the same name; all computation runs in the library's
CUDA kernels. There is no fallback: if the library is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_FAULT"}
ROUTE_PLAIN, ROUTE_BIAS_SELECT, ROUTE_GUMBEL = 0, 1, 2
DEVFAULT_BAD_EXPERT_INDEX, DEVFAULT_PIPELINE_TIMEOUT, DEVFAULT_BAD_TILE = 0x1, 0x2, 0x4
DEVFAULT_FP16_RANGE = 0x8
Y_F16, Y_F32 = 0, 1

EXPORTS = ("moe_workspace_size", "moe_workspace_init", "moe_prepare_router", "moe_route",
           "moe_permute", "moe_permute_noalloc", "moe_overflow_reroute", "moe_grouped_ffn",
           "moe_grouped_ffn_quantized", "moe_quantize_weights", "moe_combine",
           "moe_layer_forward", "moe_layer_forward_profiled", "moe_layer_forward_host",
           "moe_pack_f16", "moe_bias_update", "moe_check_bounded_waits", "moe_device_status",
           "moe_status_string")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("mode", ctypes.c_int32), ("tau", ctypes.c_float),
                ("capacity_factor", ctypes.c_float), ("capacity_override", ctypes.c_int32),
                ("n_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32),
                ("overflow_reroute", ctypes.c_int32), ("weight_bits", ctypes.c_int32)]

    @classmethod
    def make(cls, T, d, E, top_k, d_ff, n_shared=0, mode=ROUTE_PLAIN, tau=1.0,
             capacity_factor=0.0, capacity_override=0, n_groups=0, topk_groups=0,
             overflow_reroute=0, weight_bits=0):
        return cls(T, d, E, top_k, d_ff, n_shared, mode, tau, capacity_factor, capacity_override,
                   n_groups, topk_groups, int(bool(overflow_reroute)), weight_bits)

    @classmethod
    def from_layer(cls, c):
        """From any object with T, d, E, k, f, S, mode, tau, capacity_factor (and optionally
        n_groups, topk_groups, reroute, weight_bits) attributes."""
        return cls.make(c.T, c.d, c.E, c.k, c.f, c.S, c.mode, c.tau, c.capacity_factor,
                        n_groups=getattr(c, "n_groups", 0),
                        topk_groups=getattr(c, "topk_groups", 0),
                        overflow_reroute=getattr(c, "reroute", False),
                        weight_bits=getattr(c, "weight_bits", 0))


class MoeQMatrix(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("zero", ctypes.c_void_p)]


class MoeQWeights(ctypes.Structure):
    _fields_ = [(n, MoeQMatrix) for n in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("W_g", "expert_bias", "W_gate", "W_up", "W_down", "Wsh_gate", "Wsh_up",
                 "Wsh_down", "W_down_f16", "Wsh_down_f16")] + \
        [("quant", ctypes.POINTER(MoeQWeights)), ("W_g_t", ctypes.c_void_p)]


class MoeRouteOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("topk_idx", "topk_w", "counts", "offsets", "perm_slot", "slot_pos")]


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m sparse_moe_layer_route_gb300._build`")
        L = ctypes.CDLL(LIB_PATH)
        P, S, I = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        cfgp = ctypes.POINTER(MoeConfig)
        L.moe_workspace_size.argtypes = [cfgp, ctypes.POINTER(ctypes.c_size_t)]
        L.moe_workspace_init.argtypes = [P, S, P]
        L.moe_prepare_router.argtypes = [ctypes.c_int32, ctypes.c_int32, P, P, P]
        L.moe_route.argtypes = [cfgp, P, P, P, P, P, P, P, P, S, P]
        L.moe_permute.argtypes = [cfgp, P, P, P, P, P, P, S, P]
        L.moe_permute_noalloc.argtypes = [cfgp, P, P, P, P, P, P, P]
        L.moe_overflow_reroute.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, S, P]
        i32 = ctypes.c_int32
        L.moe_quantize_weights.argtypes = [i32, i32, i32, i32, P, P, P, P, P]
        L.moe_grouped_ffn_quantized.argtypes = [cfgp, P, P, P, P, ctypes.POINTER(MoeQWeights),
                                                P, P, S, P]
        L.moe_grouped_ffn.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, P, P, P, P, P, S, P]
        L.moe_combine.argtypes = [cfgp, P, ctypes.c_int32, P, P, P, S, P]
        L.moe_layer_forward.argtypes = [cfgp, ctypes.POINTER(MoeWeights), P, P, P,
                                        ctypes.POINTER(MoeRouteOut), P, S, P]
        L.moe_layer_forward_profiled.argtypes = [cfgp, ctypes.POINTER(MoeWeights), P, P, P,
                                                 ctypes.POINTER(MoeRouteOut), P, S, P,
                                                 ctypes.POINTER(ctypes.c_void_p), I]
        L.moe_layer_forward_host.argtypes = [cfgp, ctypes.POINTER(MoeWeights), P, P, P, P, S, P]
        L.moe_pack_f16.argtypes = [P, P, S, P, P]
        L.moe_bias_update.argtypes = [ctypes.c_int32, P, P, ctypes.c_float, ctypes.c_float, P]
        L.moe_device_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
        L.moe_check_bounded_waits.argtypes = [ctypes.c_int64, P, P, S, P]
        L.moe_status_string.argtypes = [I]
        L.moe_status_string.restype = ctypes.c_char_p
        for name in EXPORTS:
            if name != "moe_status_string":
                getattr(L, name).restype = I
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(status, where):
    if status != MOE_OK:
        raise MoeError(status, where)


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def alloc_workspace(cfg: MoeConfig, device="cuda"):
    """A workspace tensor of the right size (torch allocates; 256-byte aligned) with its status
    word cleared."""
    import torch
    ws = torch.empty(workspace_size(cfg), dtype=torch.uint8, device=device)
    workspace_init(ws)
    return ws


def workspace_init(ws, stream=None):
    _check(lib().moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "moe_workspace_init")


def prepare_router(W_g, W_g_t=None, stream=None):
    """W_g [d, E] bf16 transposed into W_g_t [E, d] (a new tensor unless given); one-time."""
    import torch
    d, E = W_g.shape
    if W_g_t is None:
        W_g_t = torch.empty((E, d), dtype=W_g.dtype, device=W_g.device)
    _check(lib().moe_prepare_router(d, E, _ptr(W_g), _ptr(W_g_t), _stream(stream)),
           "moe_prepare_router")
    return W_g_t


def route(cfg, x, W_g, expert_bias, gumbel_u, topk_idx, topk_w, ws, stream=None, W_g_t=None):
    _check(lib().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(W_g), _ptr(W_g_t), _ptr(expert_bias),
                           _ptr(gumbel_u), _ptr(topk_idx), _ptr(topk_w), _ptr(ws), ws.numel(),
                           _stream(stream)), "moe_route")


def permute(cfg, topk_idx, counts, offsets, perm_slot, slot_pos, ws, stream=None):
    _check(lib().moe_permute(ctypes.byref(cfg), _ptr(topk_idx), _ptr(counts), _ptr(offsets),
                             _ptr(perm_slot), _ptr(slot_pos), _ptr(ws), ws.numel(),
                             _stream(stream)), "moe_permute")


NOALLOC_MAX_SLOTS = 262144


def permute_noalloc(cfg, topk_idx, counts, offsets, perm_slot, slot_pos, fault_bits=None,
                    stream=None):
    """moe_permute without a workspace, for callers that cannot allocate device memory: the
    library's own static device array holds the scratch (shared by every call; calls that
    overlap on the GPU race). fault_bits: optional int32 device tensor of one element."""
    _check(lib().moe_permute_noalloc(ctypes.byref(cfg), _ptr(topk_idx), _ptr(counts),
                                     _ptr(offsets), _ptr(perm_slot), _ptr(slot_pos),
                                     _ptr(fault_bits), _stream(stream)), "moe_permute_noalloc")


def overflow_reroute(cfg, x, expert_bias, gumbel_u, topk_idx, topk_w, counts, slot_pos, ws,
                     stream=None, W_g_t=None):
    _check(lib().moe_overflow_reroute(ctypes.byref(cfg), _ptr(x), _ptr(W_g_t), _ptr(expert_bias),
                                      _ptr(gumbel_u), _ptr(topk_idx), _ptr(topk_w), _ptr(counts),
                                      _ptr(slot_pos), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_overflow_reroute")


def grouped_ffn(cfg, x, perm_slot, offsets, topk_w, W_gate, W_up, W_down, Wsh_gate, Wsh_up,
                Wsh_down, y_slot, ws, stream=None, W_down_f16=None, Wsh_down_f16=None):
    """y_slot [T*k + S*T, d]: float16 on the fp16 down path (W_down_f16 given), float32 on the
    bf16 down path."""
    _check(lib().moe_grouped_ffn(ctypes.byref(cfg), _ptr(x), _ptr(perm_slot), _ptr(offsets),
                                 _ptr(topk_w), _ptr(W_gate), _ptr(W_up), _ptr(W_down),
                                 _ptr(Wsh_gate), _ptr(Wsh_up), _ptr(Wsh_down),
                                 _ptr(W_down_f16), _ptr(Wsh_down_f16), _ptr(y_slot),
                                 _ptr(ws), ws.numel(), _stream(stream)), "moe_grouped_ffn")


QUANT_GROUP = 128


def quantize_weights(W, bits, stream=None):
    """Group-wise quantization of bf16 weights W [n, K, N] (or [K, N]) on W's device; returns
    a dict with q (uint8, fragment order), scale (fp16 [n, K/128, N]) and zero (uint8, same)."""
    import torch
    shp = tuple(W.shape)
    n_mat = 1 if len(shp) == 2 else shp[0]
    K, N = shp[-2], shp[-1]
    dev = W.device
    q = torch.empty(n_mat * K * N * bits // 8, dtype=torch.uint8, device=dev)
    sc = torch.empty((n_mat, K // QUANT_GROUP, N), dtype=torch.float16, device=dev)
    z = torch.empty((n_mat, K // QUANT_GROUP, N), dtype=torch.uint8, device=dev)
    _check(lib().moe_quantize_weights(bits, n_mat, K, N, _ptr(W), _ptr(q), _ptr(sc), _ptr(z),
                                      _stream(stream)), "moe_quantize_weights")
    return {"q": q, "scale": sc, "zero": z, "bits": bits, "shape": (n_mat, K, N)}


def make_qweights(gate, up, down, sh_gate=None, sh_up=None, sh_down=None) -> MoeQWeights:
    """From quantize_weights() results (keep those tensors alive while the struct is used)."""
    def m(d):
        return MoeQMatrix(None, None, None) if d is None else \
            MoeQMatrix(_ptr(d["q"]), _ptr(d["scale"]), _ptr(d["zero"]))
    return MoeQWeights(m(gate), m(up), m(down), m(sh_gate), m(sh_up), m(sh_down))


def grouped_ffn_quantized(cfg, x, perm_slot, offsets, topk_w, qweights: MoeQWeights, y_slot,
                          ws, stream=None):
    _check(lib().moe_grouped_ffn_quantized(ctypes.byref(cfg), _ptr(x), _ptr(perm_slot),
                                           _ptr(offsets), _ptr(topk_w), ctypes.byref(qweights),
                                           _ptr(y_slot), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_grouped_ffn_quantized")


def pack_f16(src_bf16, dst_f16, stream=None, fault_bits=None):
    """dst (int16/float16 tensor) = fp16 re-encoding of the bf16 tensor src (same shape).
    fault_bits: optional int32 device tensor into which DEVFAULT_FP16_RANGE is OR-ed when a
    weight had to be clamped."""
    assert src_bf16.numel() == dst_f16.numel()
    _check(lib().moe_pack_f16(_ptr(src_bf16), _ptr(dst_f16), src_bf16.numel(), _ptr(fault_bits),
                              _stream(stream)), "moe_pack_f16")


def packed_f16(src_bf16, stream=None, fault_bits=None):
    """A new float16 tensor holding the fp16 re-encoding of src (torch allocates)."""
    import torch
    dst = torch.empty(src_bf16.shape, dtype=torch.float16, device=src_bf16.device)
    pack_f16(src_bf16, dst, stream, fault_bits)
    return dst


def combine(cfg, y_slot, slot_pos, out, ws, stream=None):
    """y_slot: float16 or float32 slot rows (its dtype selects MOE_Y_F16 / MOE_Y_F32)."""
    import torch
    y_type = Y_F32 if y_slot.dtype == torch.float32 else Y_F16
    _check(lib().moe_combine(ctypes.byref(cfg), _ptr(y_slot), y_type, _ptr(slot_pos), _ptr(out),
                             _ptr(ws), ws.numel(), _stream(stream)), "moe_combine")


def make_weights(W_g, expert_bias, W_gate, W_up, W_down, Wsh_gate=None, Wsh_up=None,
                 Wsh_down=None, W_down_f16=None, Wsh_down_f16=None,
                 quant: MoeQWeights | None = None, W_g_t=None) -> MoeWeights:
    w = MoeWeights(*[_ptr(t) for t in (W_g, expert_bias, W_gate, W_up, W_down, Wsh_gate,
                                        Wsh_up, Wsh_down, W_down_f16, Wsh_down_f16)])
    w.W_g_t = _ptr(W_g_t)
    if quant is not None:
        w.quant = ctypes.pointer(quant)
        w._quant_ref = quant          # keep the struct alive with the weights
    return w


def make_route_out(topk_idx=None, topk_w=None, counts=None, offsets=None, perm_slot=None,
                   slot_pos=None) -> MoeRouteOut:
    return MoeRouteOut(*[_ptr(t) for t in (topk_idx, topk_w, counts, offsets, perm_slot,
                                           slot_pos)])


def layer_forward(cfg, weights: MoeWeights, x, gumbel_u, out, route_out: MoeRouteOut | None,
                  ws, stream=None):
    _check(lib().moe_layer_forward(ctypes.byref(cfg), ctypes.byref(weights), _ptr(x),
                                   _ptr(gumbel_u), _ptr(out),
                                   ctypes.byref(route_out) if route_out is not None else None,
                                   _ptr(ws), ws.numel(), _stream(stream)), "moe_layer_forward")


PROFILE_PHASES = ("router", "dispatch", "tiles_gather", "gate_up_gemm", "down_gemm", "combine")


def layer_forward_profiled(cfg, weights: MoeWeights, x, gumbel_u, out, route_out, ws, events,
                           stream=None):
    """layer_forward recording the 7 torch.cuda.Event objects in `events` at the phase
    boundaries (PROFILE_PHASES lie between consecutive events)."""
    for e in events:
        if not e.cuda_event:      # torch creates the CUDA event on its first record
            e.record()
    arr = (ctypes.c_void_p * 7)(*[e.cuda_event for e in events])
    _check(lib().moe_layer_forward_profiled(
        ctypes.byref(cfg), ctypes.byref(weights), _ptr(x), _ptr(gumbel_u), _ptr(out),
        ctypes.byref(route_out) if route_out is not None else None, _ptr(ws), ws.numel(),
        _stream(stream), arr, 7), "moe_layer_forward_profiled")


def layer_forward_host(cfg, weights: MoeWeights, x_host, gumbel_u_host, out_host, ws,
                       stream=None):
    _check(lib().moe_layer_forward_host(ctypes.byref(cfg), ctypes.byref(weights), _ptr(x_host),
                                        _ptr(gumbel_u_host), _ptr(out_host), _ptr(ws),
                                        ws.numel(), _stream(stream)), "moe_layer_forward_host")


def bias_update(counts, expert_bias, decay=0.99, rate=0.01, stream=None):
    """In place: expert_bias <- decay*expert_bias - rate*counts/(mean(counts)+1e-8)."""
    _check(lib().moe_bias_update(expert_bias.numel(), _ptr(counts), _ptr(expert_bias), decay, rate,
                                 _stream(stream)), "moe_bias_update")


def check_bounded_waits(limit_ns, expired, ws, stream=None):
    """Both bounded device waits against conditions that never come true (limit_ns each);
    expired: int32 device tensor of 2. Read the result with device_status()."""
    _check(lib().moe_check_bounded_waits(int(limit_ns), _ptr(expired), _ptr(ws), ws.numel(),
                                         _stream(stream)), "moe_check_bounded_waits")


def device_status(ws, stream=None) -> int:
    """Synchronises, returns the device fault bits (and clears them)."""
    bits = ctypes.c_int32(0)
    st = lib().moe_device_status(_ptr(ws), _stream(stream), ctypes.byref(bits))
    if st not in (MOE_OK, 5):
        raise MoeError(st, "moe_device_status")
    return bits.value
