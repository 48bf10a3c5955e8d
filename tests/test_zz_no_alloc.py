"""The allocation-free entry point agrees with the workspace entry point.

verify_splitkv_fwd_noalloc exists for callers that may not allocate device
memory (engines that own all free HBM through their own pool allocator, plugin
hosts that pass only input and output pointers).  Its scratch is an array built
into the library's device image.  These tests call it through the C ABI twice
in a row, so the second call runs on whatever the first call left in that
array, and compare each result with verify_splitkv_fwd given a caller
workspace, within the parity tolerance used by the other GPU tests.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 1e-2


@pytest.fixture(scope="module")
def lib():
    import speculative_decode_verify_prefix_gb300 as vsk
    from speculative_decode_verify_prefix_gb300 import _native

    vsk.build()
    vsk.set_tuning(0, 0)
    L = _native.lib()
    P = ctypes.POINTER(_native.VskTensor)
    L.verify_splitkv_fwd_noalloc.restype = ctypes.c_int
    L.verify_splitkv_fwd_noalloc.argtypes = [P] * 9 + [ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                                       ctypes.c_float, ctypes.c_float, ctypes.c_void_p]
    return L


def _noalloc(lib, p, o):
    import speculative_decode_verify_prefix_gb300 as vsk

    r = vsk.api._ref
    stream = torch.cuda.current_stream()
    return lib.verify_splitkv_fwd_noalloc(
        r(p["q"]), r(p["k_ext"]), r(p["v_ext"]), r(o), r(p["k_buffer"]), r(p["v_buffer"]), r(p["qo_indptr"]),
        r(p["kv_indptr"]), r(p["kv_indices"]), 1, p["max_len_extend"], p["k_scale"], p["v_scale"],
        p["sm_scale"], ctypes.c_void_p(stream.cuda_stream))


def _with_workspace(p):
    import speculative_decode_verify_prefix_gb300 as vsk

    q = p["q"]
    o = torch.empty(q.shape[0], q.shape[1], p["v_ext"].shape[2], dtype=torch.bfloat16, device=q.device)
    ws = torch.zeros(vsk.workspace_size(len(p["prefix_lens"]), q.shape[1], p["k_ext"].shape[1], q.shape[2],
                                        p["v_ext"].shape[2], p["max_len_extend"]), dtype=torch.uint8,
                     device=q.device)
    assert vsk.verify_splitkv_fwd(q, p["k_ext"], p["v_ext"], o, p["k_buffer"], p["v_buffer"], p["qo_indptr"],
                                  p["kv_indptr"], p["kv_indices"], None, True, None, p["max_len_extend"],
                                  p["k_scale"], p["v_scale"], sm_scale=p["sm_scale"], workspace=ws)
    torch.cuda.synchronize()
    return o


SPECS = [
    # long prefixes split across several CTAs: the tickets and partials in the
    # built-in array are used, and must be clean for the second call
    workloads.Spec("noalloc_bf16", (3000, 4000, 10, 0, 777), 4, 32, 8, 128, 128, perm=True, seed=201),
    workloads.Spec("noalloc_fp8_d256", (4096, 1500), 4, 16, 2, 256, 256, pool="e4m3", perm=True, k_scale=0.5,
                   v_scale=0.25, seed=202),
]


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_noalloc_matches_workspace_entry_point(lib, spec):
    p = workloads.make_problem(spec, "cuda")
    ref = _with_workspace(p).float().cpu().numpy()
    for _ in range(2):
        o = torch.full_like(p["q"][:, :, : p["v_ext"].shape[2]], float("nan"))
        assert _noalloc(lib, p, o) == 1, lib.vsk_last_error().decode()
        torch.cuda.synchronize()
        got = o.float().cpu().numpy()
        assert np.isfinite(got).all()
        np.testing.assert_allclose(got, ref, atol=ATOL, rtol=RTOL)


def test_noalloc_rejects_problems_beyond_the_builtin_scratch(lib):
    spec = workloads.Spec("noalloc_big", tuple([4] * 2048), 4, 32, 8, 128, 128, seed=203)
    p = workloads.make_problem(spec, "cuda")
    o = torch.empty(p["q"].shape[0], 32, 128, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, p, o) == 0
    msg = lib.vsk_last_error().decode()
    assert "bytes of scratch" in msg and "built into the library" in msg
