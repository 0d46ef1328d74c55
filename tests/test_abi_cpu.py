"""The C-ABI library on a machine without a GPU: it builds, loads, exports every
symbol include/*.h declares, and rejects bad arguments on the host before any
CUDA call."""

import ctypes
import glob
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib():
    from nvfp4_router_gate_gb300 import _native, build
    if not os.path.exists(_native.LIB_PATH):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("library not built and no nvcc")
        build.build()
    return _native


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\**\s+\**([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                             text, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    nat = _lib()
    names = _declared_functions()
    assert len(names) >= 9
    L = nat.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(nat.SIGNATURES)


def test_status_strings_and_sizes():
    nat = _lib()
    L = nat.lib()
    for code in range(7):
        assert L.nvr_status_string(code)
    assert L.nvr_sf_bytes(4, 256, nat.NVR_SF_LINEAR) == 64
    assert L.nvr_sf_bytes(4, 256, nat.NVR_SF_TILED) == 128 * 16
    assert L.nvr_sf_bytes(130, 7168, nat.NVR_SF_TILED) == 256 * 448
    assert L.nvr_sf_bytes(4, 100, nat.NVR_SF_LINEAR) == 0          # D % 64 != 0
    # the workspace bound is monotone in T_max
    prev = 0
    for T in [1, 2, 16, 17, 128, 129, 4096, 16384]:
        v = L.router_gate_workspace_size(T, 7168, 256, 8)
        assert v >= prev
        prev = v


def test_host_argument_checks_without_gpu():
    nat = _lib()
    L = nat.lib()
    fake = ctypes.c_void_p(0x10000)          # aligned, never dereferenced
    odd = ctypes.c_void_p(0x10008)           # 8-byte aligned only
    ws_n = L.router_gate_workspace_size(4, 256, 16, 2)
    # the conversion sweep's null arguments are refused before any launch
    assert L.nvr_test_conversion_sweep(None, fake, fake, fake, None) == nat.NVR_ERR_INVALID_ARG
    assert L.nvr_test_conversion_sweep(fake, fake, None, fake, None) == nat.NVR_ERR_INVALID_ARG
    # null activations
    st = L.router_gate_topk(None, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, None, 2, 1.0, 0,
                            fake, fake, fake, ws_n, None)
    assert st == nat.NVR_ERR_INVALID_ARG
    # D not a multiple of 64
    st = L.router_gate_topk(fake, nat.NVR_BF16, 4, 200, fake, fake, fake, 16, None, 2, 1.0, 0,
                            fake, fake, fake, ws_n, None)
    assert st == nat.NVR_ERR_INVALID_ARG
    # k out of range
    for k in (0, 17, 32):
        st = L.router_gate_topk(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, None, k, 1.0, 0,
                                fake, fake, fake, ws_n, None)
        assert st == nat.NVR_ERR_INVALID_ARG
    # k > N
    st = L.router_gate_topk(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 4, None, 8, 1.0, 0,
                            fake, fake, fake, ws_n, None)
    assert st == nat.NVR_ERR_INVALID_ARG
    # bad dtype, bad flags, conflicting flags
    st = L.router_gate_topk(fake, 7, 4, 256, fake, fake, fake, 16, None, 2, 1.0, 0,
                            fake, fake, fake, ws_n, None)
    assert st == nat.NVR_ERR_INVALID_ARG
    st = L.router_gate_topk(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, None, 2, 1.0, 512,
                            fake, fake, fake, ws_n, None)
    assert st == nat.NVR_ERR_INVALID_ARG
    st = L.router_gate_topk(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, None, 2, 1.0,
                            nat.NVR_FLAG_STREAM | nat.NVR_FLAG_SPLIT_N, fake, fake, fake, ws_n, None)
    assert st == nat.NVR_ERR_INVALID_ARG
    # two kernel-choice flags at once
    st = L.router_gate_topk(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, None, 2, 1.0,
                            nat.NVR_FLAG_SPLIT_K_2 | nat.NVR_FLAG_SPLIT_N,
                            fake, fake, fake, ws_n, None)
    assert st == nat.NVR_ERR_INVALID_ARG
    st = L.router_gate_topk(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, None, 2, 1.0,
                            nat.NVR_FLAG_SPLIT_K_4 | nat.NVR_FLAG_FORCE_DECODE,
                            fake, fake, fake, ws_n, None)
    assert st == nat.NVR_ERR_INVALID_ARG
    st = L.router_gate_topk(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, None, 2, 1.0,
                            nat.NVR_FLAG_FORCE_DECODE | nat.NVR_FLAG_FORCE_TENSOR_CORE,
                            fake, fake, fake, ws_n, None)
    assert st == nat.NVR_ERR_INVALID_ARG
    # misaligned activations / workspace
    st = L.router_gate_topk(odd, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, None, 2, 1.0, 0,
                            fake, fake, fake, ws_n, None)
    assert st == nat.NVR_ERR_ALIGNMENT
    st = L.router_gate_topk(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, None, 2, 1.0, 0,
                            fake, fake, odd, ws_n, None)
    assert st == nat.NVR_ERR_ALIGNMENT
    # workspace too small
    st = L.router_gate_topk(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, None, 2, 1.0, 0,
                            fake, fake, fake, 16, None)
    assert st == nat.NVR_ERR_WORKSPACE
    # empty batch: valid, launches nothing
    st = L.router_gate_topk(fake, nat.NVR_BF16, 0, 256, fake, fake, fake, 16, None, 2, 1.0, 0,
                            fake, fake, fake, ws_n, None)
    assert st == nat.NVR_OK
    # quantize: bad layout, small workspace, empty
    qn = L.nvfp4_quantize_workspace_size(4, 256)
    assert L.nvfp4_quantize_act(fake, nat.NVR_F32, 4, 256, fake, fake, 5, fake, fake, qn, None) == \
        nat.NVR_ERR_INVALID_ARG
    assert L.nvfp4_quantize_act(fake, nat.NVR_F32, 4, 256, fake, fake, 0, fake, fake, 8, None) == \
        nat.NVR_ERR_WORKSPACE
    assert L.nvfp4_quantize_act(fake, nat.NVR_F32, 0, 256, fake, fake, 0, fake, fake, qn, None) == \
        nat.NVR_OK
    assert L.nvfp4_pack_weight(None, nat.NVR_F32, 4, 256, fake, fake, fake, fake, qn, None) == \
        nat.NVR_ERR_INVALID_ARG
    # logits hook rejects the raw flag
    assert L.router_gate_logits(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, nat.NVR_FLAG_RAW_LOGITS,
                                fake, fake, ws_n, None) == nat.NVR_ERR_INVALID_ARG
    assert L.nvr_read_device_status(None, None, None) == nat.NVR_ERR_INVALID_ARG
    # NVFP4 linear: NULL or misaligned output, bad output dtype, small workspace
    lw = L.nvfp4_linear_workspace_size(4, 256, 16)
    assert lw >= ws_n
    assert L.nvfp4_linear(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, None, nat.NVR_F32, fake, lw,
                          None) == nat.NVR_ERR_INVALID_ARG
    assert L.nvfp4_linear(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, odd, nat.NVR_F32, fake, lw,
                          None) == nat.NVR_ERR_ALIGNMENT
    assert L.nvfp4_linear(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, fake, 9, fake, lw,
                          None) == nat.NVR_ERR_INVALID_ARG
    assert L.nvfp4_linear(fake, nat.NVR_BF16, 4, 256, fake, fake, fake, 16, fake, nat.NVR_BF16, fake, 16,
                          None) == nat.NVR_ERR_WORKSPACE
    assert L.nvfp4_linear(fake, nat.NVR_BF16, 0, 256, fake, fake, fake, 16, fake, nat.NVR_BF16, fake, lw,
                          None) == nat.NVR_OK
    # hash router: NULL table, k > experts, misaligned ids, empty batch
    assert L.router_hash_topk(fake, 4, None, 10, 8, 2, 1.0, fake, fake, None) == nat.NVR_ERR_INVALID_ARG
    assert L.router_hash_topk(fake, 4, fake, 10, 1, 2, 1.0, fake, fake, None) == nat.NVR_ERR_INVALID_ARG
    assert L.router_hash_topk(fake, 4, fake, 10, 8, 17, 1.0, fake, fake, None) == nat.NVR_ERR_INVALID_ARG
    assert L.router_hash_topk(ctypes.c_void_p(0x10002), 4, fake, 10, 8, 2, 1.0, fake, fake, None) == \
        nat.NVR_ERR_ALIGNMENT
    assert L.router_hash_topk(fake, 0, fake, 10, 8, 2, 1.0, fake, fake, None) == nat.NVR_OK
    assert L.router_hash_topk(None, 0, fake, 10, 8, 2, 1.0, None, None, None) == nat.NVR_OK
    # plan query: NULL rejected; otherwise a kernel sequence code 0-6 (0 on a
    # thread that has not launched a router call)
    assert L.nvr_last_router_plan(None) == nat.NVR_ERR_INVALID_ARG
    plan = (ctypes.c_int * 4)()
    assert L.nvr_last_router_plan(plan) == nat.NVR_OK
    assert 0 <= plan[0] <= 6 and plan[3] in (0, 1)


def test_workspace_counters_do_not_move_with_T():
    """Calls of any size share a workspace sized for the largest: the bound
    grows with T_max by the data regions only, never shrinking below what a
    smaller call needs, and covers the fixed counter regions (65 536 N-split
    tickets and two sets of 1024 tile-barrier counters) even for one token."""
    nat = _lib()
    L = nat.lib()
    small = L.router_gate_workspace_size(1, 256, 16, 1)
    assert small >= 65536 * 4 + 2 * 1024 * 4
    for N in (16, 256, 384):
        prev = 0
        for T in (1, 15, 16, 17, 112, 113, 4096, 4097):
            v = L.router_gate_workspace_size(T, 7168, N, 8)
            assert v >= prev, (N, T)
            prev = v


def test_workspace_size_covers_every_call_size():
    """A workspace of router_gate_workspace_size(T_max, ...) bytes passes the
    router's own size check for every T <= T_max (the check runs before any
    device call; without a GPU the call then stops at the device query)."""
    nat = _lib()
    L = nat.lib()
    fake = ctypes.c_void_p(0x10000)          # aligned, never dereferenced
    for N in (16, 256, 300, 384, 129280):
        for T_max in (1, 16, 17, 600, 4096):
            ws = L.router_gate_workspace_size(T_max, 7168, N, 8)
            for T in sorted({1, 2, 15, 16, 17, 128, 129, 300, T_max}):
                if T > T_max:
                    continue
                st = L.router_gate_topk(fake, nat.NVR_BF16, T, 7168, fake, fake, fake, N, None, 8, 1.0, 0,
                                        fake, fake, fake, ws, None)
                assert st != nat.NVR_ERR_WORKSPACE, (N, T_max, T)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from nvfp4_router_gate_gb300 import _native
    monkeypatch.setattr(_native, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_native, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _native.lib()
