"""The C-ABI library builds, loads and exports every entry point include/moe.h declares; its
host-side logic (workspace sizing, argument validation, status strings) runs without a GPU."""
import ctypes
import os
import re

import pytest

import sparse_moe_layer_route_gb300 as M
from sparse_moe_layer_route_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return M.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(M.EXPORTS)


def test_workspace_size_and_layout(lib):
    cfg = M.MoeConfig.make(16384, 7168, 128, 2, 2048, mode=M.ROUTE_BIAS_SELECT,
                           capacity_factor=1.25)
    n = M.workspace_size(cfg)
    TK = 16384 * 2
    # at least the gathered rows, H and the slot-ordered outputs
    assert n >= 2 * TK * 7168 + 2 * TK * 2048 + 2 * TK * 7168
    assert n < 4 * 1024 ** 3
    small = M.MoeConfig.make(128, 256, 8, 2, 512)
    assert 0 < M.workspace_size(small) < n


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), 1), (dict(T=0), 0), (dict(T=0, E=300), 2), (dict(E=0), 1), (dict(top_k=0), 1), (dict(mode=3), 1),
    (dict(mode=2, tau=0.0), 1), (dict(E=300), 2), (dict(top_k=9, E=16), 2),
    (dict(top_k=5, E=4), 2), (dict(d=100), 2), (dict(d_ff=96), 2), (dict(n_shared=5), 2),
    (dict(overflow_reroute=2), 1), (dict(overflow_reroute=1, n_groups=4, topk_groups=2), 2),
    (dict(n_groups=3), 2), (dict(n_groups=4, topk_groups=0), 1),
    (dict(n_groups=4, topk_groups=1, top_k=3), 1),
    (dict(weight_bits=5), 1), (dict(weight_bits=8, d=192), 2), (dict(weight_bits=4), 0),
])
def test_bad_configs_rejected(lib, kw, status):
    base = dict(T=64, d=128, E=8, top_k=2, d_ff=128, n_shared=0, mode=0, tau=1.0,
                capacity_factor=0.0, capacity_override=0)
    base.update(kw)
    cfg = M.MoeConfig(**base)
    n = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == status


def test_entry_points_validate_before_any_launch(lib):
    cfg = M.MoeConfig.make(64, 128, 8, 2, 128)
    need = M.workspace_size(cfg)
    fake = 0x10000000  # never dereferenced: every call below must fail validation first
    # missing tensors
    assert lib.moe_route(ctypes.byref(cfg), None, fake, None, None, None, fake, fake, fake, need,
                         None) == 1
    # bias mode without a bias
    bcfg = M.MoeConfig.make(64, 128, 8, 2, 128, mode=M.ROUTE_BIAS_SELECT)
    assert lib.moe_route(ctypes.byref(bcfg), fake, fake, None, None, None, fake, fake, fake, need,
                         None) == 1
    # workspace: NULL, misaligned, too small
    assert lib.moe_route(ctypes.byref(cfg), fake, fake, None, None, None, fake, fake, None, need,
                         None) == 3
    assert lib.moe_route(ctypes.byref(cfg), fake, fake, None, None, None, fake, fake, fake + 8, need,
                         None) == 3
    assert lib.moe_permute(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake, need - 1,
                           None) == 3
    # shared experts requested without their weights
    scfg = M.MoeConfig.make(64, 128, 8, 2, 128, n_shared=1)
    assert lib.moe_grouped_ffn(ctypes.byref(scfg), fake, fake, fake, fake, fake, fake, fake,
                               None, None, None, None, None, fake, fake,
                               M.workspace_size(scfg), None) == 1
    # the fp16 down path with shared experts needs the shared fp16 copy too
    assert lib.moe_grouped_ffn(ctypes.byref(scfg), fake, fake, fake, fake, fake, fake, fake,
                               fake, fake, fake, fake, None, fake, fake,
                               M.workspace_size(scfg), None) == 1
    # rows of x move in 16-byte pieces: a misaligned x is refused before any launch
    assert lib.moe_grouped_ffn(ctypes.byref(cfg), fake + 2, fake, fake, fake, fake, fake, fake,
                               None, None, None, None, None, fake, fake, need, None) == 1
    wf = M.MoeWeights()
    wf.W_g = wf.W_gate = wf.W_up = wf.W_down = fake
    assert lib.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(wf), fake + 8, None, fake, None,
                                 fake, need, None) == 1
    # the router's and the re-route's exact dot products and the quantized passes' activation
    # prep read x in 16-byte pieces too
    assert lib.moe_route(ctypes.byref(cfg), fake + 2, fake, None, None, None, fake, fake, fake, need,
                         None) == 1
    rcfg = M.MoeConfig.make(64, 128, 8, 2, 128, capacity_factor=1.0, overflow_reroute=1)
    assert lib.moe_overflow_reroute(ctypes.byref(rcfg), fake + 4, None, None, None, fake, fake, fake,
                                    fake, fake, M.workspace_size(rcfg), None) == 1
    qcfg = M.MoeConfig.make(64, 128, 8, 2, 128, weight_bits=8)
    qm = M.MoeQMatrix(q=fake, scale=fake, zero=fake)
    qw = M.MoeQWeights(gate=qm, up=qm, down=qm)
    assert lib.moe_grouped_ffn_quantized(ctypes.byref(qcfg), fake + 6, fake, fake, None,
                                         ctypes.byref(qw), fake, fake, M.workspace_size(qcfg),
                                         None) == 1
    # router preparation: NULL / misaligned transpose, unsupported sizes
    assert lib.moe_prepare_router(128, 8, None, fake, None) == 1
    assert lib.moe_prepare_router(128, 8, fake, fake + 2, None) == 1
    assert lib.moe_prepare_router(96, 8, fake, fake, None) == 2
    assert lib.moe_prepare_router(128, 257, fake, fake, None) == 2
    assert lib.moe_route(ctypes.byref(cfg), fake, fake, fake + 8, None, None, fake, fake, fake, need,
                         None) == 1
    wt = M.MoeWeights()
    wt.W_g = wt.W_gate = wt.W_up = wt.W_down = fake
    wt.W_g_t = fake + 4
    assert lib.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(wt), fake, None, fake, None,
                                 fake, need, None) == 1
    # pack: NULL / misaligned pointers
    assert lib.moe_pack_f16(None, fake, 16, None, None) == 1
    assert lib.moe_pack_f16(fake + 2, fake, 16, None, None) == 1
    # combine: the slot rows' type must be one of the two
    assert lib.moe_combine(ctypes.byref(cfg), fake, 2, fake, fake, fake, need, None) == 1
    assert lib.moe_combine(ctypes.byref(cfg), fake, -1, fake, fake, fake, need, None) == 1
    w = M.MoeWeights()
    assert lib.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(w), fake, None, fake, None,
                                 fake, need, None) == 1
    assert lib.moe_workspace_init(None, 0, None) == 3
    # the bounded-wait check: workspace, expired flags, limit range (100 us .. 2 s)
    assert lib.moe_check_bounded_waits(1000000, fake, None, 512, None) == 3
    assert lib.moe_check_bounded_waits(1000000, fake, fake, 256, None) == 3
    assert lib.moe_check_bounded_waits(1000000, None, fake, 512, None) == 1
    assert lib.moe_check_bounded_waits(99999, fake, fake, 512, None) == 1
    assert lib.moe_check_bounded_waits(2000000001, fake, fake, 512, None) == 1


def test_status_strings(lib):
    for s in range(6):
        assert M.status_string(s)
    assert M.status_string(0) == "ok"
    assert M.status_string(99) == "unknown status"


def test_reroute_workspace_and_validation(lib):
    kw = dict(mode=M.ROUTE_BIAS_SELECT, capacity_factor=1.25)
    base = M.workspace_size(M.MoeConfig.make(4096, 1024, 64, 2, 512, **kw))
    rr = M.workspace_size(M.MoeConfig.make(4096, 1024, 64, 2, 512, overflow_reroute=1, **kw))
    # scores [T, E] fp32 + preference lists [T, E] bytes + per-token and per-expert state
    assert rr - base >= 4096 * 64 * 5
    # without a capacity limit there is nothing to re-route and no extra workspace
    nocap = dict(mode=M.ROUTE_BIAS_SELECT)
    assert M.workspace_size(M.MoeConfig.make(4096, 1024, 64, 2, 512, overflow_reroute=1,
                                             **nocap)) == \
        M.workspace_size(M.MoeConfig.make(4096, 1024, 64, 2, 512, **nocap))
    off = M.MoeConfig.make(64, 128, 8, 2, 128, capacity_factor=1.0)
    P = ctypes.c_void_p(0x1000)
    assert lib.moe_overflow_reroute(ctypes.byref(off), P, None, None, None, P, P, P, P, P, 1 << 30,
                                    None) == 1     # re-route not enabled in the config
    on = M.MoeConfig.make(64, 128, 8, 2, 128, capacity_factor=1.0, overflow_reroute=1)
    assert lib.moe_overflow_reroute(ctypes.byref(on), None, None, None, None, P, P, P, P, P, 1 << 30,
                                    None) == 1     # x missing
    assert lib.moe_overflow_reroute(ctypes.byref(on), P, None, None, None, P, P, P, P, None, 1 << 30,
                                    None) == 3     # no workspace


def test_quantize_weights_validation(lib):
    P = ctypes.c_void_p(0x1000)
    assert lib.moe_quantize_weights(3, 1, 128, 32, P, P, P, P, None) == 1     # bits
    assert lib.moe_quantize_weights(8, 0, 128, 32, P, P, P, P, None) == 1     # n_mat
    assert lib.moe_quantize_weights(8, 1, 192, 32, P, P, P, P, None) == 2     # K % 128
    assert lib.moe_quantize_weights(4, 1, 128, 48, P, P, P, P, None) == 2     # N % 32
    assert lib.moe_quantize_weights(4, 1, 128, 32, None, P, P, P, None) == 1  # W missing
    cfg = M.MoeConfig.make(64, 128, 8, 2, 128, weight_bits=8)
    q = M.MoeQWeights()
    assert lib.moe_grouped_ffn_quantized(ctypes.byref(cfg), P, P, P, None, ctypes.byref(q), P,
                                         P, 1 << 30, None) == 1            # codes missing
    cfg0 = M.MoeConfig.make(64, 128, 8, 2, 128)
    assert lib.moe_grouped_ffn_quantized(ctypes.byref(cfg0), P, P, P, None, ctypes.byref(q), P,
                                         P, 1 << 30, None) == 1            # weight_bits 0


def test_empty_batch_is_a_no_op_on_the_host(lib):
    """T = 0: the configuration is still validated, tensor pointers and the workspace are not
    examined, and the entry points that have nothing to clear return MOE_OK without a CUDA call
    (this machine may have no GPU at all)."""
    cfg = M.MoeConfig.make(0, 128, 8, 2, 128, n_shared=1, mode=M.ROUTE_GUMBEL, tau=0.5,
                           capacity_factor=1.0, overflow_reroute=1)
    n = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == 0 and n.value == 512
    z = None
    assert lib.moe_route(ctypes.byref(cfg), z, z, z, z, z, z, z, z, 0, z) == 0
    assert lib.moe_overflow_reroute(ctypes.byref(cfg), z, z, z, z, z, z, z, z, z, 0, z) == 0
    assert lib.moe_grouped_ffn(ctypes.byref(cfg), z, z, z, z, z, z, z, z, z, z, z, z, z, z, 0,
                               z) == 0
    assert lib.moe_combine(ctypes.byref(cfg), z, 0, z, z, z, 0, z) == 0
    assert lib.moe_layer_forward(ctypes.byref(cfg), z, z, z, z, z, z, 0, z) == 0
    assert lib.moe_layer_forward_host(ctypes.byref(cfg), z, z, z, z, z, 0, z) == 0
    q = M.MoeConfig.make(0, 128, 8, 2, 128, weight_bits=8)
    assert lib.moe_grouped_ffn_quantized(ctypes.byref(q), z, z, z, z, z, z, z, 0, z) == 0
    # the dispatch entry points still need their per-expert outputs
    assert lib.moe_permute(ctypes.byref(cfg), z, z, z, z, z, z, 0, z) == 1
    assert lib.moe_permute_noalloc(ctypes.byref(cfg), z, z, z, z, z, z, z) == 1
    # config-level errors are still reported for an empty batch
    bad = M.MoeConfig.make(0, 128, 8, 2, 128, weight_bits=8)
    assert lib.moe_grouped_ffn(ctypes.byref(bad), z, z, z, z, z, z, z, z, z, z, z, z, z, z, 0,
                               z) == 1
    plain = M.MoeConfig.make(0, 128, 8, 2, 128)
    assert lib.moe_overflow_reroute(ctypes.byref(plain), z, z, z, z, z, z, z, z, z, 0, z) == 1
