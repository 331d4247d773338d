"""q4k_moe_gemv_noalloc: the routed-MoE call for callers that cannot allocate
device memory per call (engines that own all device memory in their own
arena, host code that does not own the allocator).  Its workspace is a fixed
device array inside the library, shared by every call on a device.

The GPU test calls it through the C ABI twice in a row, on two different
problems (so the second call runs over the first one's leftovers in the shared
array), and checks each result against the workspace-taking q4k_moe_gemv and
against the oracle, within the MoE tolerance the other tests use.  This file
sorts last so that a run stopping at the first failure has run everything else.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from _gpu import DEV


@pytest.fixture(scope="module")
def q4k():
    from bit_block_quantized_q4_gb300 import build
    build.build()
    import bit_block_quantized_q4_gb300 as m
    return m


def _noalloc_c_abi(q4k, c, ids, wts):
    """Call q4k_moe_gemv_noalloc through the raw C entry point."""
    L = q4k.lib()
    wg, wu, wd = (c[k].to(DEV) for k in ("wg", "wu", "wd"))
    x = c["x"].to(DEV)
    ids_d, wts_d = ids.to(DEV).contiguous(), wts.to(DEV).contiguous()
    T, top_k = ids.shape
    y = torch.full((T, c["H"]), float("nan"), dtype=torch.float32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = L.q4k_moe_gemv_noalloc(wg.data_ptr(), wu.data_ptr(), wd.data_ptr(), c["stride"], c["E"],
                                c["H"], c["F"], x.data_ptr(), T, x.stride(0), ids_d.data_ptr(),
                                wts_d.data_ptr(), top_k, y.data_ptr(), y.stride(0), stream)
    assert st == 0, q4k.status_str(st)
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_twice_in_a_row(q4k):
    from test_moe import _bound, _check, _gpu, _make
    cases = [_make(16, 1024, 512, 16, 8, seed=301), _make(8, 512, 768, 5, 3, seed=302)]
    for c in cases:  # two calls in a row on different problems
        y_na = _noalloc_c_abi(q4k, c, c["ids"], c["wts"])
        y_ws, err = _gpu(q4k, c)
        assert err == 0
        T = c["ids"].shape[0]
        yref, bound = _bound(c, c["ids"], c["wts"], list(range(T)))
        _check(y_na, y_ws, bound, "noalloc vs workspace call")
        _check(y_na, yref, bound, "noalloc vs oracle")
    assert q4k.q4k_get_device_error() == 0


@pytest.mark.gpu
def test_noalloc_allocates_no_device_memory(q4k):
    # after one warm-up call (which looks up the array's address), further
    # calls leave the device's free memory, as the driver reports it, unchanged
    from test_moe import _make
    c = _make(16, 1024, 512, 16, 8, seed=303)
    _noalloc_c_abi(q4k, c, c["ids"], c["wts"])
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc_c_abi(q4k, c, c["ids"], c["wts"])
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


@pytest.mark.gpu
def test_noalloc_rejects_problems_larger_than_its_array(q4k):
    L = q4k.lib()
    E, H, F, T, K = 64, 8192, 4096, 64, 8      # workspace far above the fixed array
    assert q4k.q4k_moe_workspace_size(E, T, K, H, F) > 8 << 20
    P = 0x10000
    st = L.q4k_moe_gemv_noalloc(P, P, P, F * H // 256 * 144, E, H, F, P, T, H, P, P, K, P, H, None)
    assert st == 4  # Q4K_ERR_WORKSPACE, returned before anything is launched
