"""GB300 (sm_103a) NVFP4 MoE router gate: Python binding of the C ABI.

Every step of the router runs in the library's CUDA kernels; this module only
checks tensor arguments, allocates outputs with PyTorch when the caller does not
pass them, and forwards raw device pointers and the current CUDA stream.

Functions (same names as include/nvfp4_router.h):

* ``nvfp4_quantize_act(x, sf_layout="linear")`` -> (x_fp4, x_sf, x_gsa)
* ``nvfp4_pack_weight(W)`` -> (W_fp4, W_sf, w_gsa)  (tile-layout scales)
* ``router_gate_topk(x, W_fp4, W_sf, w_gsa, bias, k, routed_scaling, raw=False)``
  -> (ids int32 [T, k], weights fp32 [T, k])
* ``router_gate_logits(x, W_fp4, W_sf, w_gsa)`` -> logits fp32 [T, N]
* ``router_hash_topk(token_ids, tid2eid, n_experts, routed_scaling)`` -> (ids, weights)
* ``nvfp4_linear(x, W_fp4, W_sf, w_gsa, out_dtype=torch.float32)`` -> out [T, N]
  (``Nvfp4Linear`` keeps the packed weight and a workspace resident)
* ``nvfp4_pack_experts(W [E, N, D])``, ``nvfp4_moe_gemm(x, ids, W_fp4, W_sf, w_gsa)`` -> y [T, k, N],
  ``nvfp4_moe_combine(y, w)`` -> out [T, N]
* ``router_gate_workspace_size``, ``router_gate_x_gsa``, ``nvfp4_quantize_workspace_size``,
  ``nvr_sf_bytes``, ``nvr_read_device_status``

``RouterGate`` keeps the packed weight, the workspace and the output buffers
resident so that a call allocates nothing (CUDA-graph capturable).
"""

import ctypes

import torch

from . import _native
from ._native import (NVR_FLAG_FORCE_DECODE, NVR_FLAG_FORCE_TENSOR_CORE, NVR_FLAG_RAW_LOGITS,
                      NVR_FLAG_SPLIT_K_2, NVR_FLAG_SPLIT_K_4, NVR_FLAG_SPLIT_K_8, NVR_FLAG_SPLIT_N,
                      NVR_FLAG_STREAM, NVR_FLAG_NO_COOPERATIVE, RouterError)

__all__ = ["nvfp4_quantize_act", "nvfp4_pack_weight", "router_gate_topk", "router_gate_logits", "router_hash_topk",
           "router_gate_workspace_size", "router_gate_x_gsa", "nvfp4_quantize_workspace_size", "nvr_sf_bytes",
           "nvr_read_device_status", "last_router_plan", "plan_router", "RouterGate", "RouterError", "NVR_FLAG_RAW_LOGITS",
           "NVR_FLAG_FORCE_TENSOR_CORE", "NVR_FLAG_FORCE_DECODE", "NVR_FLAG_SPLIT_K_2",
           "NVR_FLAG_SPLIT_K_4", "NVR_FLAG_SPLIT_K_8", "NVR_FLAG_SPLIT_N", "NVR_FLAG_STREAM", "NVR_FLAG_NO_COOPERATIVE", "new_workspace",
           "nvfp4_linear", "nvfp4_linear_workspace_size", "Nvfp4Linear", "nvfp4_pack_experts",
           "nvfp4_moe_gemm", "nvfp4_moe_gemm_workspace_size", "nvfp4_moe_combine"]

_LAYOUTS = {"linear": _native.NVR_SF_LINEAR, "tiled": _native.NVR_SF_TILED}


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return _native.NVR_BF16
    if t.dtype == torch.float32:
        return _native.NVR_F32
    raise TypeError("activations must be bfloat16 or float32, got %s" % t.dtype)


def _dev(t, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def nvr_sf_bytes(rows, D, layout="linear"):
    return int(_native.lib().nvr_sf_bytes(rows, D, _LAYOUTS[layout]))


def nvfp4_quantize_workspace_size(rows, D):
    return int(_native.lib().nvfp4_quantize_workspace_size(rows, D))


def router_gate_workspace_size(T_max, D, N, k=8):
    return int(_native.lib().router_gate_workspace_size(T_max, D, N, k))


def router_gate_x_gsa(workspace):
    """A one-element fp32 view of the workspace word holding the global scale of
    x from the latest tensor-core router call on it (stays on the GPU)."""
    off = int(_native.lib().router_gate_x_gsa_offset())
    return workspace[off:off + 4].view(torch.float32)


def new_workspace(nbytes, device=None):
    """A zeroed, 256-byte aligned workspace (torch allocations are aligned)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def nvfp4_quantize_act(x, sf_layout="linear", x_fp4=None, x_sf=None, x_gsa=None, workspace=None,
                       stream=None):
    """Runtime NVFP4 quantization of x [T, D] (bf16/fp32) with one global scale."""
    T, D = x.shape
    dev = x.device
    if x_fp4 is None:
        x_fp4 = torch.empty((T, D // 2), dtype=torch.uint8, device=dev)
    if x_sf is None:
        x_sf = torch.empty(nvr_sf_bytes(T, D, sf_layout), dtype=torch.uint8, device=dev)
    if x_gsa is None:
        x_gsa = torch.empty(1, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(nvfp4_quantize_workspace_size(T, D), dev)
    st = _native.lib().nvfp4_quantize_act(
        _dev(x, "x"), _dtype_code(x), T, D, _dev(x_fp4, "x_fp4"), _dev(x_sf, "x_sf"),
        _LAYOUTS[sf_layout], _dev(x_gsa, "x_gsa"), _dev(workspace, "workspace"),
        workspace.numel(), _stream(stream))
    _native.check("nvfp4_quantize_act", st)
    return x_fp4, x_sf, x_gsa


def nvfp4_pack_weight(W, W_fp4=None, W_sf=None, w_gsa=None, workspace=None, stream=None):
    """Load-time NVFP4 quantization of the gate weight W [N, D]; tile-layout scales."""
    N, D = W.shape
    dev = W.device
    if W_fp4 is None:
        W_fp4 = torch.empty((N, D // 2), dtype=torch.uint8, device=dev)
    if W_sf is None:
        W_sf = torch.empty(nvr_sf_bytes(N, D, "tiled"), dtype=torch.uint8, device=dev)
    if w_gsa is None:
        w_gsa = torch.empty(1, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(nvfp4_quantize_workspace_size(N, D), dev)
    st = _native.lib().nvfp4_pack_weight(
        _dev(W, "W"), _dtype_code(W), N, D, _dev(W_fp4, "W_fp4"), _dev(W_sf, "W_sf"),
        _dev(w_gsa, "w_gsa"), _dev(workspace, "workspace"), workspace.numel(), _stream(stream))
    _native.check("nvfp4_pack_weight", st)
    return W_fp4, W_sf, w_gsa


def router_gate_topk(x, W_fp4, W_sf, w_gsa, bias=None, k=8, routed_scaling=1.0, raw=False,
                     out_ids=None, out_w=None, workspace=None, flags=0, stream=None):
    """Route x [T, D]: returns (ids int32 [T, k], weights fp32 [T, k])."""
    T, D = x.shape
    N = W_fp4.shape[0]
    dev = x.device
    if out_ids is None:
        out_ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    if out_w is None:
        out_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(router_gate_workspace_size(T, D, N, k), dev)
    f = int(flags) | (NVR_FLAG_RAW_LOGITS if raw else 0)
    st = _native.lib().router_gate_topk(
        _dev(x, "x"), _dtype_code(x), T, D, _dev(W_fp4, "W_fp4"), _dev(W_sf, "W_sf"),
        _dev(w_gsa, "w_gsa"), N, None if bias is None else _dev(bias, "bias"), int(k),
        float(routed_scaling), f, _dev(out_ids, "out_ids"), _dev(out_w, "out_w"),
        _dev(workspace, "workspace"), workspace.numel(), _stream(stream))
    _native.check("router_gate_topk", st)
    return out_ids, out_w


def router_gate_logits(x, W_fp4, W_sf, w_gsa, logits=None, workspace=None, flags=0, stream=None):
    """Test hook: the gate logits [T, N] fp32 of the quantized operands."""
    T, D = x.shape
    N = W_fp4.shape[0]
    dev = x.device
    if logits is None:
        logits = torch.empty((T, N), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(router_gate_workspace_size(T, D, N, 1), dev)
    st = _native.lib().router_gate_logits(
        _dev(x, "x"), _dtype_code(x), T, D, _dev(W_fp4, "W_fp4"), _dev(W_sf, "W_sf"),
        _dev(w_gsa, "w_gsa"), N, int(flags), _dev(logits, "logits"), _dev(workspace, "workspace"),
        workspace.numel(), _stream(stream))
    _native.check("router_gate_logits", st)
    return logits


def nvfp4_linear_workspace_size(T_max, D, N):
    return int(_native.lib().nvfp4_linear_workspace_size(T_max, D, N))


def nvfp4_linear(x, W_fp4, W_sf, w_gsa, out_dtype=torch.float32, out=None, workspace=None, stream=None):
    """NVFP4 linear with a runtime activation scale: quantize(x) [T, D] . W^T -> [T, N] fp32 or bf16."""
    T, D = x.shape
    N = W_fp4.shape[0]
    dev = x.device
    if out is None:
        out = torch.empty((T, N), dtype=out_dtype, device=dev)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be float32 or bfloat16")
    if workspace is None:
        workspace = new_workspace(nvfp4_linear_workspace_size(T, D, N), dev)
    code = _native.NVR_BF16 if out.dtype == torch.bfloat16 else _native.NVR_F32
    st = _native.lib().nvfp4_linear(
        _dev(x, "x"), _dtype_code(x), T, D, _dev(W_fp4, "W_fp4"), _dev(W_sf, "W_sf"), _dev(w_gsa, "w_gsa"), N,
        _dev(out, "out"), code, _dev(workspace, "workspace"), workspace.numel(), _stream(stream))
    _native.check("nvfp4_linear", st)
    return out


class Nvfp4Linear:
    """Resident NVFP4 linear layer: the weight [N, D] is quantized once at
    construction (nvfp4_pack_weight), the workspace and the output buffer
    stay allocated, and each call quantizes its activations with their own
    runtime global scale.  Calls allocate nothing (CUDA-graph capturable)."""

    def __init__(self, W, max_tokens=128, out_dtype=torch.float32):
        self.N, self.D = W.shape
        dev = W.device
        self.W_fp4, self.W_sf, self.w_gsa = nvfp4_pack_weight(W)
        self.max_tokens = int(max_tokens)
        self.workspace = new_workspace(nvfp4_linear_workspace_size(self.max_tokens, self.D, self.N), dev)
        self.out = torch.empty((self.max_tokens, self.N), dtype=out_dtype, device=dev)

    def __call__(self, x, stream=None):
        T = x.shape[0]
        if T > self.max_tokens:
            raise ValueError("batch of %d tokens exceeds max_tokens=%d" % (T, self.max_tokens))
        return nvfp4_linear(x, self.W_fp4, self.W_sf, self.w_gsa, out=self.out[:T], workspace=self.workspace,
                            stream=stream)


def nvfp4_pack_experts(W):
    """Load-time NVFP4 quantization of E expert weights W [E, N, D] (N a
    multiple of 128) into the stacked layout nvfp4_moe_gemm reads: codes
    [E * N, D/2], tile-layout scales over the E * N rows, w_gsa [E] (each
    expert with its own global scale)."""
    E, N, D = W.shape
    dev = W.device
    codes = torch.empty((E * N, D // 2), dtype=torch.uint8, device=dev)
    per = nvr_sf_bytes(N, D, "tiled")
    sf = torch.empty(E * per, dtype=torch.uint8, device=dev)
    gsa = torch.empty(E, dtype=torch.float32, device=dev)
    ws = new_workspace(nvfp4_quantize_workspace_size(N, D), dev)
    for e in range(E):
        nvfp4_pack_weight(W[e], W_fp4=codes[e * N:(e + 1) * N], W_sf=sf[e * per:(e + 1) * per],
                          w_gsa=gsa[e:e + 1], workspace=ws)
    return codes, sf, gsa


def nvfp4_moe_gemm_workspace_size(T_max, D, n_experts, k):
    return int(_native.lib().nvfp4_moe_gemm_workspace_size(T_max, D, n_experts, k))


def nvfp4_moe_gemm(x, ids, W_fp4, W_sf, w_gsa, out_dtype=torch.float32, y=None, workspace=None, stream=None):
    """Grouped expert GEMM of the routed pairs: y [T, k, N] (fp32 or bf16) with
    y[t, j] = quantize(x)[t] . W_{ids[t, j]}^T."""
    T, D = x.shape
    k = ids.shape[1]
    E = w_gsa.shape[0]
    N = W_fp4.shape[0] // E
    dev = x.device
    if ids.dtype != torch.int32:
        raise TypeError("ids must be int32")
    if y is None:
        y = torch.empty((T, k, N), dtype=out_dtype, device=dev)
    if workspace is None:
        workspace = new_workspace(nvfp4_moe_gemm_workspace_size(T, D, E, k), dev)
    code = _native.NVR_BF16 if y.dtype == torch.bfloat16 else _native.NVR_F32
    st = _native.lib().nvfp4_moe_gemm(
        _dev(x, "x"), _dtype_code(x), T, D, _dev(ids, "ids"), k, E, _dev(W_fp4, "W_fp4"), _dev(W_sf, "W_sf"),
        _dev(w_gsa, "w_gsa"), N, _dev(y, "y"), code, _dev(workspace, "workspace"), workspace.numel(),
        _stream(stream))
    _native.check("nvfp4_moe_gemm", st)
    return y


def nvfp4_moe_combine(y, w, out=None, stream=None):
    """out [T, N] fp32 = sum_j w[t, j] * y[t, j, :] (j in order)."""
    T, k, N = y.shape
    if out is None:
        out = torch.empty((T, N), dtype=torch.float32, device=y.device)
    code = _native.NVR_BF16 if y.dtype == torch.bfloat16 else _native.NVR_F32
    st = _native.lib().nvfp4_moe_combine(_dev(y, "y"), code, T, k, N, _dev(w, "w"), _dev(out, "out"),
                                         _stream(stream))
    _native.check("nvfp4_moe_combine", st)
    return out


def router_hash_topk(token_ids, tid2eid, n_experts, routed_scaling=1.0, out_ids=None, out_w=None, stream=None):
    """Hash router: ids int32 [T, k] = tid2eid[token_ids], weights routed_scaling / k."""
    if token_ids.dtype != torch.int32 or tid2eid.dtype != torch.int32:
        raise TypeError("token_ids and tid2eid must be int32")
    T = token_ids.shape[0]
    vocab, k = tid2eid.shape
    dev = token_ids.device
    if out_ids is None:
        out_ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    if out_w is None:
        out_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    st = _native.lib().router_hash_topk(
        _dev(token_ids, "token_ids"), T, _dev(tid2eid, "tid2eid"), vocab, int(n_experts), int(k),
        float(routed_scaling), _dev(out_ids, "out_ids"), _dev(out_w, "out_w"), _stream(stream))
    _native.check("router_hash_topk", st)
    return out_ids, out_w


_PLAN_SEQUENCES = {0: "none", 1: "decode", 2: "fused", 3: "amax+fused", 4: "amax+quantize+splitk+epilogue",
                   5: "amax+quantize+splitn", 6: "amax+quantize+stream"}


def last_router_plan():
    """The launch plan of this thread's latest router call: a dict with the
    kernel sequence, token-tile rows, CTAs per tile and whether they form a
    cluster."""
    out = (ctypes.c_int * 4)()
    _native.check("nvr_last_router_plan", _native.lib().nvr_last_router_plan(out))
    return {"sequence": _PLAN_SEQUENCES.get(out[0], str(out[0])), "tile_rows": out[1],
            "ctas_per_tile": out[2], "clustered": bool(out[3])}


def plan_router(T, D, N, *, num_sms, cluster_capacity, block_capacity, dtype="bf16", flags=0):
    """The launch plan a router call of this shape would get on a device with
    num_sms SMs holding cluster_capacity[i] clusters of 2**i CTAs of the fused
    kernel (five ints) and block_capacity of its CTAs without clusters (host
    arithmetic only), in the form of last_router_plan."""
    caps = (ctypes.c_int * 5)(*[int(c) for c in cluster_capacity])
    out = (ctypes.c_int * 4)()
    code = _native.NVR_BF16 if dtype == "bf16" else _native.NVR_F32
    _native.check("nvr_plan_router", _native.lib().nvr_plan_router(
        int(T), int(D), int(N), code, int(flags), int(num_sms), caps, int(block_capacity), out))
    return {"sequence": _PLAN_SEQUENCES.get(out[0], str(out[0])), "tile_rows": out[1],
            "ctas_per_tile": out[2], "clustered": bool(out[3])}


def nvr_read_device_status(workspace, stream=None):
    """The workspace status word (0 = ok, 6 = a device-side wait timed out)."""
    out = ctypes.c_int(0)
    st = _native.lib().nvr_read_device_status(_dev(workspace, "workspace"), _stream(stream),
                                              ctypes.byref(out))
    _native.check("nvr_read_device_status", st)
    return out.value


class RouterGate:
    """Resident router: packed NVFP4 gate weight, bias, workspace and outputs.

    ``gate(x)`` routes up to ``max_tokens`` tokens and returns views of the
    resident output buffers; nothing is allocated per call, so a call can be
    captured in a CUDA graph.
    """

    def __init__(self, W, bias=None, k=8, routed_scaling=1.0, raw=False, max_tokens=4096):
        self.N, self.D = W.shape
        self.k, self.routed_scaling, self.raw = int(k), float(routed_scaling), bool(raw)
        dev = W.device
        self.W_fp4, self.W_sf, self.w_gsa = nvfp4_pack_weight(W)
        self.bias = None if bias is None else bias.to(device=dev, dtype=torch.float32).contiguous()
        self.max_tokens = int(max_tokens)
        self.workspace = new_workspace(
            router_gate_workspace_size(self.max_tokens, self.D, self.N, self.k), dev)
        self.ids = torch.empty((self.max_tokens, self.k), dtype=torch.int32, device=dev)
        self.weights = torch.empty((self.max_tokens, self.k), dtype=torch.float32, device=dev)

    def status(self, stream=None):
        """The workspace status word (0 ok, 6 = a device-side bounded wait of
        some call timed out and its outputs are unspecified).  Reads device
        memory and waits for the stream: call it outside graph capture, e.g.
        every few steps; re-zero the workspace after a timeout."""
        return nvr_read_device_status(self.workspace, stream)

    def __call__(self, x, flags=0, stream=None):
        T = x.shape[0]
        if T > self.max_tokens:
            raise ValueError("batch of %d tokens exceeds max_tokens=%d" % (T, self.max_tokens))
        ids, w = self.ids[:T], self.weights[:T]
        router_gate_topk(x, self.W_fp4, self.W_sf, self.w_gsa, self.bias, self.k, self.routed_scaling,
                         self.raw, out_ids=ids, out_w=w, workspace=self.workspace, flags=flags,
                         stream=stream)
        return ids, w
