"""The allocation-free router entry point against the ordinary one.

router_gate_topk_noalloc serves callers that cannot allocate device memory
(a plugin whose host hands it only its input and output buffers, or a path
that must not touch an allocator), so it keeps its scratch in a fixed array
inside the library.  This test calls it through the C ABI twice in a row and
checks both results against router_gate_topk with a caller workspace, and
that oversized shapes are refused.  It lives in its own file, collected last.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import workloads as WL  # noqa: E402
from gpu_util import to_device  # noqa: E402


def _noalloc(lib, x, W_fp4, W_sf, w_gsa, N, bias, k, scale, ids, w):
    from nvfp4_router_gate_gb300 import _native
    T, D = x.shape
    return lib.router_gate_topk_noalloc(
        x.data_ptr(), _native.NVR_BF16, T, D, W_fp4.data_ptr(), W_sf.data_ptr(), w_gsa.data_ptr(),
        N, None if bias is None else bias.data_ptr(), k, scale, 0, ids.data_ptr(), w.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice():
    import nvfp4_router_gate_gb300 as R
    from nvfp4_router_gate_gb300 import _native
    lib = _native.lib()
    wl = WL.WORKLOADS["decode"]
    W_fp4, W_sf, w_gsa = R.nvfp4_pack_weight(to_device(WL.make_w(wl), "bf16"))
    bias = torch.from_numpy(WL.make_bias(wl)).cuda()
    for T in (1, 8):
        w = wl.with_T(T)
        x = to_device(WL.make_x(w), "bf16")
        ref_ids, ref_w = R.router_gate_topk(x, W_fp4, W_sf, w_gsa, bias, w.k, w.routed_scaling)
        for _ in range(2):                           # two calls in a row share the scratch
            ids = torch.full((T, w.k), -1, dtype=torch.int32, device="cuda")
            wts = torch.zeros((T, w.k), dtype=torch.float32, device="cuda")
            st = _noalloc(lib, x, W_fp4, W_sf, w_gsa, w.N, bias, w.k, w.routed_scaling, ids, wts)
            assert st == _native.NVR_OK, _native.status_string(st)
            torch.cuda.synchronize()
            assert torch.equal(ids, ref_ids)
            assert np.max(np.abs(wts.cpu().numpy() - ref_w.cpu().numpy())) <= 1e-5


def test_noalloc_rejects_oversized_scratch():
    from nvfp4_router_gate_gb300 import _native
    lib = _native.lib()
    T, D, N = 16, 256, 16384                         # 16 * 16384 * 8 bytes > 1 MiB
    x = torch.zeros((T, D), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((N, D // 2), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(N * D // 16, dtype=torch.uint8, device="cuda")
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    ids = torch.empty((T, 8), dtype=torch.int32, device="cuda")
    wts = torch.empty((T, 8), dtype=torch.float32, device="cuda")
    st = _noalloc(lib, x, W, sf, g, N, None, 8, 1.0, ids, wts)
    assert st == _native.NVR_ERR_WORKSPACE
