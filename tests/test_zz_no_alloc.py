"""moe_permute_noalloc: dispatch for callers that cannot allocate device memory (for instance a
plugin that a host application hands only input and output buffers, or a latency-critical loop
that may not call cudaMalloc/cudaFree). Its scratch is the library's own static device array, so
it takes no workspace.

Checked through the C ABI against the oracle's dispatch (the counting-sort definition of
"参数规模与稀疏激活的真相拆解", §3.2's capacity rule) and against moe_permute (the workspace-based
entry point) on two calls in a row with different routing, so a call that leaned on the previous
call's leftovers in the shared static array would show up. Dispatch outputs are integers: the
comparisons are exact."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import sparse_moe_layer_route_gb300 as M

pytestmark = pytest.mark.gpu


def _outputs(T, E, k, dev):
    i32 = dict(dtype=torch.int32, device=dev)
    return (torch.full((E,), -7, **i32), torch.full((E + 1,), -7, **i32),
            torch.full((T * k,), -7, **i32), torch.full((T * k,), -7, **i32))


def _routing(seed, T, E, k, skew):
    rng = np.random.default_rng(seed)
    keys = rng.random((T, E)) * (np.arange(1, E + 1) ** -skew)[None, :]
    return np.argsort(-keys, axis=1)[:, :k].astype(np.int32)


def test_noalloc_permute_matches_workspace_permute_twice():
    dev = "cuda"
    lib = M.lib()
    # two consecutive calls, different sizes and routing; the second has fewer dispatch blocks
    # and a capacity limit, so stale histogram rows from the first call would corrupt it
    for seed, (T, E, k, cap) in enumerate([(20000, 128, 8, 0), (3001, 64, 6, 150)]):
        idx_np = _routing(seed, T, E, k, 1.2)
        idx = torch.as_tensor(idx_np, device=dev)
        cfg = M.MoeConfig.make(T, 64, E, k, 64, capacity_override=cap)
        ref = _outputs(T, E, k, dev)
        ws = M.alloc_workspace(cfg)
        M.permute(cfg, idx, *ref, ws)
        got = _outputs(T, E, k, dev)
        fault = torch.full((1,), 99, dtype=torch.int32, device=dev)
        st = lib.moe_permute_noalloc(ctypes.byref(cfg), idx.data_ptr(), got[0].data_ptr(),
                                     got[1].data_ptr(), got[2].data_ptr(), got[3].data_ptr(),
                                     fault.data_ptr(),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == M.MOE_OK
        torch.cuda.synchronize()
        assert M.device_status(ws) == 0
        assert int(fault.item()) == 0          # cleared by the call, no fault recorded
        want = O.permute(idx_np, E, cap if cap else None)
        for name, a, b in zip(("counts", "offsets", "perm_slot", "slot_pos"), ref, got):
            assert np.array_equal(b.cpu().numpy(), want[name]), name + " differs from the oracle"
            assert torch.equal(a, b), name


def test_noalloc_permute_reports_bad_index_and_rejects_oversize():
    dev = "cuda"
    T, E, k = 500, 16, 2
    idx_np = _routing(7, T, E, k, 0.5)
    idx_np[3, 1] = E                            # out of range: reported, slot dropped
    idx = torch.as_tensor(idx_np, device=dev)
    cfg = M.MoeConfig.make(T, 64, E, k, 64)
    got = _outputs(T, E, k, dev)
    fault = torch.zeros(1, dtype=torch.int32, device=dev)
    M.permute_noalloc(cfg, idx, *got, fault)
    torch.cuda.synchronize()
    assert int(fault.item()) & M.DEVFAULT_BAD_EXPERT_INDEX
    assert int(got[3][3 * k + 1].item()) == -1
    # sizes past the static scratch are refused on the host, before anything is enqueued
    big = M.MoeConfig.make(M.NOALLOC_MAX_SLOTS // 2 + 1, 64, E, 2, 64)
    with pytest.raises(M.MoeError) as ei:
        M.permute_noalloc(big, idx, *got)
    assert ei.value.status == 2                 # MOE_ERR_UNSUPPORTED
