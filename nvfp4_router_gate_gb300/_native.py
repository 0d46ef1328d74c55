"""ctypes declarations of the C ABI in include/nvfp4_router.h.

Loading the library needs no GPU; it fails loudly (RuntimeError) when the
shared library has not been built.  There is no fallback of any kind.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4_router.so")

NVR_OK = 0
NVR_ERR_INVALID_ARG = 1
NVR_ERR_UNSUPPORTED = 2
NVR_ERR_ALIGNMENT = 3
NVR_ERR_WORKSPACE = 4
NVR_ERR_CUDA = 5
NVR_ERR_TIMEOUT = 6

NVR_BF16 = 0
NVR_F32 = 1
NVR_SF_LINEAR = 0
NVR_SF_TILED = 1

NVR_FLAG_RAW_LOGITS = 1
NVR_FLAG_FORCE_TENSOR_CORE = 2
NVR_FLAG_FORCE_DECODE = 4
NVR_FLAG_SPLIT_K_2 = 8
NVR_FLAG_SPLIT_K_4 = 16
NVR_FLAG_SPLIT_K_8 = 32
NVR_FLAG_SPLIT_N = 64
NVR_FLAG_STREAM = 128
NVR_FLAG_NO_COOPERATIVE = 256
NVR_FLAG_TEST_STALL = 1 << 30

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_i32 = ctypes.c_int
_u32 = ctypes.c_uint32
_f32 = ctypes.c_float

# name -> (restype, argtypes); the same list the header declares
SIGNATURES = {
    "nvr_status_string": (ctypes.c_char_p, [_i32]),
    "nvr_last_cuda_error": (ctypes.c_char_p, []),
    "nvr_last_router_plan": (_i32, [ctypes.POINTER(_i32)]),
    "nvr_router_cooperative_state": (_i32, []),
    "nvr_test_occupy": (_i32, [_i32, _i32, ctypes.c_uint64, _p]),
    "nvr_test_conversion_sweep": (_i32, [_p, _p, _p, _p, _p]),
    "nvr_plan_router": (_i32, [_i64, _i64, _i64, _i32, _u32, _i32, ctypes.POINTER(_i32), _i32,
                               ctypes.POINTER(_i32)]),
    "nvr_sf_bytes": (_sz, [_i64, _i64, _i32]),
    "nvfp4_quantize_workspace_size": (_sz, [_i64, _i64]),
    "nvfp4_quantize_act": (_i32, [_p, _i32, _i64, _i64, _p, _p, _i32, _p, _p, _sz, _p]),
    "nvfp4_pack_weight": (_i32, [_p, _i32, _i64, _i64, _p, _p, _p, _p, _sz, _p]),
    "router_gate_workspace_size": (_sz, [_i64, _i64, _i64, _i32]),
    "router_gate_x_gsa_offset": (_sz, []),
    "router_gate_topk": (_i32, [_p, _i32, _i64, _i64, _p, _p, _p, _i64, _p, _i32, _f32, _u32,
                                _p, _p, _p, _sz, _p]),
    "router_gate_topk_noalloc": (_i32, [_p, _i32, _i64, _i64, _p, _p, _p, _i64, _p, _i32, _f32,
                                        _u32, _p, _p, _p]),
    "router_hash_topk": (_i32, [_p, _i64, _p, _i64, _i64, _i32, _f32, _p, _p, _p]),
    "nvfp4_linear_workspace_size": (_sz, [_i64, _i64, _i64]),
    "nvfp4_linear": (_i32, [_p, _i32, _i64, _i64, _p, _p, _p, _i64, _p, _i32, _p, _sz, _p]),
    "nvfp4_moe_gemm_workspace_size": (_sz, [_i64, _i64, _i64, _i32]),
    "nvfp4_moe_gemm": (_i32, [_p, _i32, _i64, _i64, _p, _i32, _i64, _p, _p, _p, _i64, _p, _i32, _p, _sz, _p]),
    "nvfp4_moe_combine": (_i32, [_p, _i32, _i64, _i32, _i64, _p, _p, _p]),
    "router_gate_logits": (_i32, [_p, _i32, _i64, _i64, _p, _p, _p, _i64, _u32, _p, _p, _sz, _p]),
    "nvr_read_device_status": (_i32, [_p, _p, ctypes.POINTER(_i32)]),
    "nvr_set_profile_events": (_i32, [_p, _i32]),
}

_lib = None


def lib():
    """The loaded library (built by ``nvfp4_router_gate_gb300.build.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libnvfp4_router.so is not built; run nvfp4_router_gate_gb300.build.build() "
                "(needs nvcc with sm_103a support)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(code):
    return lib().nvr_status_string(int(code)).decode()


class RouterError(RuntimeError):
    def __init__(self, fn, code):
        self.code = int(code)
        msg = "%s failed: %s (status %d)" % (fn, status_string(code), int(code))
        if self.code == NVR_ERR_CUDA:
            msg += ": " + lib().nvr_last_cuda_error().decode()
        super().__init__(msg)


def check(fn, code):
    if code != NVR_OK:
        raise RouterError(fn, code)
