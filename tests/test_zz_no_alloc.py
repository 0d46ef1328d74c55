"""The allocation-free router entry point against the ordinary one.

router_gate_topk_noalloc serves callers that cannot allocate device memory
(a plugin whose host hands it only its input and output buffers, or a path
that must not touch an allocator), so it keeps its scratch in a fixed array
inside the library.  These tests call it through the C ABI twice in a row and
check both results against router_gate_topk with a caller workspace (bf16
and fp32 activations, RAW mode, a shape near the array's size, inside a CUDA
graph), and that shapes beyond the decode plan are refused.  They live in
their own file, collected last.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

import workloads as WL  # noqa: E402
from gpu_util import to_device  # noqa: E402


def _noalloc(lib, x, W_fp4, W_sf, w_gsa, N, bias, k, scale, ids, w, flags=0, stream=None):
    from nvfp4_router_gate_gb300 import _native
    T, D = x.shape
    dt = _native.NVR_BF16 if x.dtype == torch.bfloat16 else _native.NVR_F32
    s = stream if stream is not None else torch.cuda.current_stream()
    return lib.router_gate_topk_noalloc(
        x.data_ptr(), dt, T, D, W_fp4.data_ptr(), W_sf.data_ptr(), w_gsa.data_ptr(),
        N, None if bias is None else bias.data_ptr(), k, scale, flags, ids.data_ptr(), w.data_ptr(),
        ctypes.c_void_p(s.cuda_stream))


def _check(ids, wts, ref_ids, ref_w):
    assert torch.equal(ids, ref_ids)
    assert np.max(np.abs(wts.cpu().numpy() - ref_w.cpu().numpy())) <= 1e-5


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
            _check(ids, wts, ref_ids, ref_w)


def test_noalloc_near_the_scratch_limit_raw_and_fp32():
    """T = 16 tokens on N = 1664 outputs: 213 KB of keys and scores, close to
    the 224 KiB array (and to the decode kernel's shared-memory plan); RAW
    mode; fp32 activations."""
    import nvfp4_router_gate_gb300 as R
    from nvfp4_router_gate_gb300 import _native
    lib = _native.lib()
    rng = np.random.default_rng(61)
    T, D, N, k = 16, 256, 1664, 8
    W = torch.from_numpy((rng.standard_normal((N, D)) * 0.05).astype(np.float32)).cuda()
    x32 = torch.from_numpy(rng.standard_normal((T, D)).astype(np.float32)).cuda()
    bias = torch.from_numpy(rng.uniform(-0.05, 0.05, N).astype(np.float32)).cuda()
    W_fp4, W_sf, w_gsa = R.nvfp4_pack_weight(W)
    for x, raw in ((x32, False), (x32.to(torch.bfloat16), True)):
        flags = _native.NVR_FLAG_RAW_LOGITS if raw else 0
        ref_ids, ref_w = R.router_gate_topk(x, W_fp4, W_sf, w_gsa, bias, k, 1.5, raw)
        assert R.last_router_plan()["sequence"] == "decode"
        for _ in range(2):
            ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
            wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
            st = _noalloc(lib, x, W_fp4, W_sf, w_gsa, N, bias, k, 1.5, ids, wts, flags=flags)
            assert st == _native.NVR_OK, _native.status_string(st)
            torch.cuda.synchronize()
            assert torch.equal(ids, ref_ids)
            tol = 1e-5 if not raw else 1e-3 * float(ref_w.abs().max())
            assert np.max(np.abs(wts.cpu().numpy() - ref_w.cpu().numpy())) <= tol


def test_noalloc_in_a_cuda_graph():
    """A first call outside capture (it looks up the array's device address),
    then the entry point captured in a CUDA graph and replayed twice."""
    import nvfp4_router_gate_gb300 as R
    from nvfp4_router_gate_gb300 import _native
    lib = _native.lib()
    wl = WL.WORKLOADS["decode"]
    W_fp4, W_sf, w_gsa = R.nvfp4_pack_weight(to_device(WL.make_w(wl), "bf16"))
    bias = torch.from_numpy(WL.make_bias(wl)).cuda()
    x = to_device(WL.make_x(wl.with_T(1)), "bf16")
    ref_ids, ref_w = R.router_gate_topk(x, W_fp4, W_sf, w_gsa, bias, wl.k, wl.routed_scaling)
    ids = torch.full((1, wl.k), -1, dtype=torch.int32, device="cuda")
    wts = torch.zeros((1, wl.k), dtype=torch.float32, device="cuda")
    assert _noalloc(lib, x, W_fp4, W_sf, w_gsa, wl.N, bias, wl.k, wl.routed_scaling, ids, wts) == 0
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert _noalloc(lib, x, W_fp4, W_sf, w_gsa, wl.N, bias, wl.k, wl.routed_scaling, ids, wts, stream=s) == 0
    for _ in range(2):
        ids.fill_(-1)
        wts.zero_()
        g.replay()
        torch.cuda.synchronize()
        _check(ids, wts, ref_ids, ref_w)


def test_noalloc_refuses_shapes_beyond_the_plan():
    """16 tokens on 16384 outputs need 2 MB of keys and scores, beyond the
    decode kernel's shared-memory plan and the array: refused before any
    launch."""
    from nvfp4_router_gate_gb300 import _native
    lib = _native.lib()
    T, D, N = 16, 256, 16384
    x = torch.zeros((T, D), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((N, D // 2), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(N * D // 16, dtype=torch.uint8, device="cuda")
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    ids = torch.empty((T, 8), dtype=torch.int32, device="cuda")
    wts = torch.empty((T, 8), dtype=torch.float32, device="cuda")
    st = _noalloc(lib, x, W, sf, g, N, None, 8, 1.0, ids, wts)
    assert st == _native.NVR_ERR_UNSUPPORTED
