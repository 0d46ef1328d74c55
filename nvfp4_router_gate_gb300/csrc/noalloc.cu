// noalloc.cu -- router_gate_topk_noalloc: the single-launch decode router for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code
// that runs inside a host framework which owns every device allocation (a
// plugin or extension whose host gives it only its input and output
// buffers), or a latency-critical path that is not allowed to touch an
// allocator at all.  For them this entry point keeps its scratch -- the
// per-token keys and scores and the last-CTA ticket of the decode kernel --
// in a fixed array in the library's own device memory instead of a
// caller-provided workspace.
//
// The array is a file-scope __device__ variable.  Host code cannot use its
// name as a device address (on the host it names a stand-in object), so the
// first call on each device looks up the real address with
// cudaGetSymbolAddress while that device is current, and every launch
// receives that pointer.
#include <mutex>

#include "nvr_internal.h"

namespace {

// Scratch of the allocation-free entry point: 256 bytes of control words
// (the ticket at byte 8), then keys and scores [T, N] fp32.  The decode plan
// only accepts shapes whose T * N * 8 bytes of keys and scores fit one CTA's
// shared-memory plan (kDecodeMaxSmem), so that much after the control words
// holds every call the plan accepts.  Every GPU that loads the library holds
// this memory (224 KiB + 256 bytes) until the process exits.
constexpr size_t kNoAllocControl = 256;
constexpr size_t kNoAllocScratchBytes = kNoAllocControl + nvr::kDecodeMaxSmem;
static_assert(kNoAllocScratchBytes % 256 == 0, "the keys start 256-byte aligned");
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
uint8_t* g_scratch_ptr[nvr::kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device); nullptr on failure.
uint8_t* scratch_for_current_device(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= nvr::kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = static_cast<uint8_t*>(p);
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" nvr_status router_gate_topk_noalloc(const void* x, nvr_dtype dt, int64_t T, int64_t D,
                                               const uint8_t* W_fp4, const uint8_t* W_scales,
                                               const float* w_gsa, int64_t N, const float* bias,
                                               int k, float routed_scaling, uint32_t flags,
                                               int32_t* out_ids, float* out_w,
                                               nvr_stream_t stream) {
  using namespace nvr;
  if (!x || !W_fp4 || !W_scales || !w_gsa || !out_ids || !out_w) return NVR_ERR_INVALID_ARG;
  if (T < 0 || D <= 0 || D % 64 != 0 || D > (1 << 24) || N <= 0 || N > (1 << 28)) return NVR_ERR_INVALID_ARG;
  if (dt != NVR_BF16 && dt != NVR_F32) return NVR_ERR_INVALID_ARG;
  if (k < 1 || k > kMaxKmax || k > N) return NVR_ERR_INVALID_ARG;
  if (flags & ~static_cast<uint32_t>(NVR_FLAG_RAW_LOGITS)) return NVR_ERR_INVALID_ARG;
  const uintptr_t a16 = 15u, a4 = 3u;
  if ((reinterpret_cast<uintptr_t>(x) & a16) || (reinterpret_cast<uintptr_t>(W_fp4) & a16) ||
      (reinterpret_cast<uintptr_t>(W_scales) & a16) || (reinterpret_cast<uintptr_t>(w_gsa) & a4) ||
      (bias && (reinterpret_cast<uintptr_t>(bias) & a4)) || (reinterpret_cast<uintptr_t>(out_ids) & a4) ||
      (reinterpret_cast<uintptr_t>(out_w) & a4))
    return NVR_ERR_ALIGNMENT;
  if (T == 0) return NVR_OK;
  const int sms = device_sm_count();
  if (sms <= 0) return NVR_ERR_CUDA;
  const DecodePlan dp = plan_decode(T, D, N, sms, dt == NVR_BF16);
  if (!dp.ok) return NVR_ERR_UNSUPPORTED;
  // the keys and scores of every (token, expert) pair fit the fixed array for
  // every shape the decode plan accepts; checked all the same
  if (static_cast<size_t>(T) * static_cast<size_t>(N) * 8 > kNoAllocScratchBytes - kNoAllocControl)
    return NVR_ERR_WORKSPACE;
  cudaError_t e = cudaSuccess;
  uint8_t* scratch = scratch_for_current_device(&e);
  if (!scratch) return NVR_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The ticket starts at zero (a __device__ array is zero-initialised) and
  // the decode kernel puts it back to zero on every path it takes, so each
  // call is the one launch (which programmatic launch can overlap with its
  // predecessor's tail inside a graph).
  float* keys = reinterpret_cast<float*>(scratch + kNoAllocControl);
  float* scores = keys + T * N;
  // the last CTA's ticket, never a wait: a call here has no status word
  e = launch_decode(x, dt == NVR_BF16, T, D, W_fp4, W_scales, w_gsa, N, bias, k, routed_scaling,
                    (flags & NVR_FLAG_RAW_LOGITS) != 0, out_ids, out_w, nullptr, keys, scores,
                    reinterpret_cast<uint32_t*>(scratch + kWsDecodeTicket), nullptr, nullptr, false, dp, s);
  return cuda_status(e);
}
